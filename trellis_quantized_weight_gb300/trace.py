"""Phase timing of the small-M product kernel from a trace build of the library.

Builds a second copy of the library with ``-DTRELLIS_TRACE`` under
``_build/trace`` (the shipped library is untouched), runs one product shape
back to back and once on an idle GPU, and summarises the clock64 stamps the
kernel wrote (layout beside ``kTraceCtaWords`` in ``csrc/gemm_smallm_kernel.cuh``):

* the loop: cycles per unit (one 256-weight block of one tile-group) of every
  CTA, from its entry to thread 0 leaving the loop;
* the end: for every warp, the cycles from leaving the loop to its tickets'
  answers, to the partial sums of the tiles it reduces being loaded and added,
  and to its last instruction, grouped by what the warp had to do;
* per CTA, its last warp's end against its last warp's leaving the loop.

Stamps are SM cycle counts, compared only within one CTA.  The calls go
through the same C ABI as the shipped library.

    python -m trellis_quantized_weight_gb300.trace --rows 15 --bits 4
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os

import numpy as np

from . import binding, synth
from . import build as _build

CTA_WORDS = 8 + 8 * 16           # kTraceCtaWords
MAX_CTAS = 4096


def build_traced() -> str:
    return _build.build(defines=("TRELLIS_TRACE",), build_dir=os.path.join(_build.BUILD, "trace"))


def load_traced(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name, (res, args) in binding.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    lib.trellis_trace_attach.restype = ctypes.c_int
    lib.trellis_trace_attach.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    return lib


def _groups(flags: int) -> str:
    parts = []
    if flags & 1:
        parts.append("first split")
    if flags & 2:
        parts.append("last split")
    if flags & 4:
        parts.append("in-loop ticket")
    red = [t for t, bit in (("first", 8), ("last", 16)) if flags & bit]
    parts.append("reduces " + "+".join(red) if red else "reduces nothing")
    return ", ".join(parts) if flags & 3 else "no split segment"


def summarise(rec: np.ndarray) -> dict:
    """rec: [CTAs, CTA_WORDS] int64 of one launch."""
    live = rec[:, 1] != 0
    rec = rec[live]
    units = rec[:, 3]
    loop = rec[:, 2] - rec[:, 1]
    per_unit = loop / np.maximum(units, 1)
    out = {"ctas": int(rec.shape[0]), "units": sorted(set(int(u) for u in units)),
           "cycles_per_unit": {"median": float(np.median(per_unit)), "min": float(per_unit.min()),
                               "max": float(per_unit.max())}}
    warps = rec[:, 8:].reshape(rec.shape[0], 16, 8)
    groups: dict[str, list] = {}
    cta_tail = []
    for ci in range(rec.shape[0]):
        w = warps[ci]
        wl = w[:, 0] != 0
        if not wl.any():
            continue
        cta_tail.append(int(w[wl, 3].max() - w[wl, 0].max()))
        for wi in np.nonzero(wl)[0]:
            r = w[wi]
            g = groups.setdefault(_groups(int(r[4])), [[], [], []])
            if r[1]:
                g[0].append(int(r[1] - r[0]))
            if r[2]:
                g[1].append(int(r[2] - r[0]))
            g[2].append(int(r[3] - r[0]))
    stat = lambda v: {"n": len(v), "median": int(np.median(v)), "max": int(max(v))} if v else None
    out["warp_end"] = {k: {"tickets": stat(v[0]), "sums_loaded": stat(v[1]), "done": stat(v[2])}
                       for k, v in sorted(groups.items())}
    out["cta_tail"] = {"median": int(np.median(cta_tail)), "max": int(max(cta_tail))}
    return out


def to_markdown(res: dict) -> str:
    sh = res["shape"]
    lines = [f"M={sh['M']}, K={sh['K']}, N={sh['N']}, k={sh['k']}; SM cycles.", ""]
    lines.append("| run | CTAs | units a CTA | cycles a unit: median (min, max) | CTA end after its loop: median, max |")
    lines.append("|---|---|---|---|---|")
    for mode in ("back_to_back", "isolated"):
        r = res[mode]
        u = r["cycles_per_unit"]
        lines.append(f"| {mode.replace('_', ' ')} | {r['ctas']} | {', '.join(map(str, r['units']))} | "
                     f"{u['median']:.0f} ({u['min']:.0f}, {u['max']:.0f}) | {r['cta_tail']['median']}, {r['cta_tail']['max']} |")
    for mode in ("back_to_back", "isolated"):
        lines += ["", f"Warps, {mode.replace('_', ' ')}: cycles after leaving the loop, median / max.", "",
                  "| warp's segments | warps | tickets answered | sums loaded | done |", "|---|---|---|---|---|"]
        for g, v in res[mode]["warp_end"].items():
            cell = lambda x: f"{x['median']} / {x['max']}" if x else "-"
            lines.append(f"| {g} | {v['done']['n']} | {cell(v['tickets'])} | {cell(v['sums_loaded'])} | {cell(v['done'])} |")
    return "\n".join(lines)


def main(argv=None) -> dict:
    import torch

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--rows", type=int, default=15, help="M")
    ap.add_argument("--K", type=int, default=5120)
    ap.add_argument("--N", type=int, default=17408)
    ap.add_argument("--bits", type=int, default=4, help="k")
    ap.add_argument("--calls", type=int, default=60, help="back-to-back calls before the traced one")
    ap.add_argument("--copies", type=int, default=8, help="code copies rotated to defeat L2")
    ap.add_argument("--json", help="also write the summary here")
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("the trace needs a CUDA device")
    lib = load_traced(build_traced())
    M, K, N, k = a.rows, a.K, a.N, a.bits
    x, c, sc = synth.small(M, K, N, k, seed=5).generate()
    dx = torch.from_numpy(x.view(np.int16)).cuda()
    dcs = [torch.from_numpy(c.view(np.int32)).cuda() for _ in range(a.copies)]
    ds = torch.from_numpy(sc.view(np.int16)).cuda()
    out = torch.empty((M, N), dtype=torch.int16, device="cuda")
    buf = torch.zeros(MAX_CTAS * CTA_WORDS, dtype=torch.int64, device="cuda")
    if lib.trellis_trace_attach(buf.data_ptr(), buf.numel() * 8) != 0:
        raise RuntimeError("trellis_trace_attach failed")
    stream = torch.cuda.current_stream().cuda_stream

    def call(i):
        st = lib.trellis_gemm(dx.data_ptr(), dcs[i % a.copies].data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                              out.data_ptr(), stream)
        if st != 0:
            raise binding.TrellisError(st, "trellis_gemm")

    res = {"shape": {"M": M, "K": K, "N": N, "k": k}}
    try:
        for mode in ("back_to_back", "isolated"):
            buf.zero_()
            for i in range(a.calls):
                call(i)
            if mode == "isolated":
                torch.cuda.synchronize()
                buf.zero_()
                call(0)
            torch.cuda.synchronize()
            if lib.trellis_device_status(None) != 0:
                raise RuntimeError("device status reports a timeout")
            rec = buf.view(MAX_CTAS, CTA_WORDS).cpu().numpy()
            res[mode] = summarise(rec)
    finally:
        lib.trellis_trace_attach(None, 0)
    print(to_markdown(res))
    if a.json:
        with open(a.json, "w") as f:
            json.dump(res, f, indent=1)
    return res


if __name__ == "__main__":
    main()
