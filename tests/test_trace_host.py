"""Host side of the trace tool (trellis_quantized_weight_gb300/trace.py): the
summary of a hand-built stamp buffer, worked out by hand below."""
import numpy as np

from trellis_quantized_weight_gb300 import trace


def _record():
    rec = np.zeros((4, trace.CTA_WORDS), dtype=np.int64)

    def cta(c, entry, loop_end, units):
        rec[c, 0:4] = (7 + c, entry, loop_end, units)

    def warp(c, w, left, tickets, sums, done, flags):
        rec[c, 8 + 8 * w: 8 + 8 * w + 5] = (left, tickets, sums, done, flags)

    # CTA 0: 16 units in 160,000 cycles; warp 0 reduces both split tiles,
    # warp 1 only takes its tickets
    cta(0, 1000, 161000, 16)
    warp(0, 0, 160500, 162500, 165000, 166000, 1 | 2 | 8 | 16)
    warp(0, 1, 160900, 162800, 0, 163100, 1 | 2)
    # CTA 1: 15 units in 135,000 cycles; one warp with no split segment
    cta(1, 500, 135500, 15)
    warp(1, 0, 135000, 0, 0, 135400, 0)
    # CTAs 2, 3 never stamped (the buffer is larger than the grid)
    return rec


def test_summary_of_a_hand_built_buffer():
    s = trace.summarise(_record())
    assert s["ctas"] == 2
    assert s["units"] == [15, 16]
    cpu = s["cycles_per_unit"]
    assert cpu["min"] == 9000.0 and cpu["max"] == 10000.0 and cpu["median"] == 9500.0
    g = s["warp_end"]
    both = g["first split, last split, reduces first+last"]
    assert both["tickets"] == {"n": 1, "median": 2000, "max": 2000}
    assert both["sums_loaded"] == {"n": 1, "median": 4500, "max": 4500}
    assert both["done"] == {"n": 1, "median": 5500, "max": 5500}
    none = g["first split, last split, reduces nothing"]
    assert none["tickets"]["max"] == 1900 and none["sums_loaded"] is None and none["done"]["max"] == 2200
    assert g["no split segment"]["done"] == {"n": 1, "median": 400, "max": 400}
    # per CTA: last warp done minus last warp out of the loop
    # CTA 0: 166000 - 160900 = 5100; CTA 1: 135400 - 135000 = 400
    assert s["cta_tail"] == {"median": 2750, "max": 5100}


def test_markdown_names_every_group():
    res = {"shape": {"M": 15, "K": 5120, "N": 17408, "k": 4}}
    res["back_to_back"] = res["isolated"] = trace.summarise(_record())
    md = trace.to_markdown(res)
    assert "M=15, K=5120, N=17408, k=4" in md
    for grp in res["isolated"]["warp_end"]:
        assert md.count(f"| {grp} |") == 2
    assert "9500 (9000, 10000)" in md


def test_flag_groups():
    assert trace._groups(0) == "no split segment"
    assert trace._groups(1) == "first split, reduces nothing"
    assert trace._groups(1 | 2 | 4 | 16) == "first split, last split, in-loop ticket, reduces last"
