"""GB300 (sm_103a) packed-Trellis weight decode and decode-and-multiply.

The compute lives in ``_build/libtrellis_gb300.so`` (hand-written CUDA kernels
behind the C ABI declared in ``include/trellis.h``); this package only builds
it (``build.build()``), binds it (``binding``) and draws seeded synthetic inputs
(``synth``).  Calls fail loudly when the library is missing.
"""
from .binding import (TrellisError, decode, gemm, gemm_gateup, gemm_gateup_workspace_bytes, gemm_packed,
                      gemm_packed_workspace_bytes, gemm_workspace_bytes, load, status_string)

__all__ = ["TrellisError", "decode", "gemm", "gemm_gateup", "gemm_gateup_workspace_bytes", "gemm_packed",
           "gemm_packed_workspace_bytes", "gemm_workspace_bytes", "load", "status_string"]
