"""The byte sums a 12-bit window can produce, against the quotient table's range.

The kernels' shared-memory quotient table only holds the byte sums S in
[kSumLo, kSumHi] (trellis_device.cuh).  This enumerates every 12-bit window,
hashes it as the pages define (z = win * 34038481 + 76625530 mod 2^32, S = the
sum of z's four bytes, i.e. code + 510) and checks that the reachable sums are
exactly that range, so no window can index outside the table.
"""
import pathlib
import re

HEADER = pathlib.Path(__file__).resolve().parents[1] / "trellis_quantized_weight_gb300" / "csrc" / "trellis_device.cuh"


def _const(name: str) -> int:
    m = re.search(rf"constexpr\s+(?:int|uint32_t)\s+{name}\s*=\s*(\d+)u?;", HEADER.read_text())
    assert m, f"{name} not found in {HEADER.name}"
    return int(m.group(1))


def test_reachable_byte_sums_match_table_range():
    lo, hi = _const("kSumLo"), _const("kSumHi")
    mul, add = _const("kHashMul"), _const("kHashAdd")
    assert (mul, add) == (34038481, 76625530)
    sums = set()
    for win in range(1 << 12):
        z = (win * 34038481 + 76625530) & 0xFFFFFFFF
        p = (z & 0x00FF00FF) + ((z >> 8) & 0x00FF00FF)
        sums.add((p & 0xFFFF) + (p >> 16))
    assert min(sums) == lo and max(sums) == hi
    assert hi - lo + 1 == 903
