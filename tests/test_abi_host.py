"""The C-ABI library builds, loads, exports every declared symbol and rejects bad
arguments on the host (no GPU needed: validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from trellis_quantized_weight_gb300 import build, binding
    build.build()
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "trellis.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(trellis_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"trellis_decode", "trellis_gemm", "trellis_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_library_exports_only_the_declared_functions(lib):
    """Everything but the C ABI has hidden visibility: no internal symbol (in
    particular no template-local static, which the dynamic linker would merge
    across two copies of the library loaded into one process) is exported."""
    import shutil
    import subprocess
    from trellis_quantized_weight_gb300 import build
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm is not installed")
    out = subprocess.run([nm, "-D", "--defined-only", build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert exported == set(declared_functions())


def test_binding_signatures_cover_header(lib):
    from trellis_quantized_weight_gb300 import binding
    assert set(declared_functions()) == set(binding.SIGNATURES)


def test_abi_version_and_status_strings(lib):
    assert lib.trellis_abi_version() == 1
    for s in range(-7, 1):
        assert lib.trellis_status_string(s).decode().startswith("TRELLIS_")
    assert lib.trellis_status_string(123).decode() == "TRELLIS_ERR_UNKNOWN"


FAKE = 0x10000   # never dereferenced: every case below fails validation first (a call that could
                 # pass validation must use real device buffers)


@pytest.mark.parametrize("args,want", [
    ((0, FAKE, 5120, 8, 4, 12, 256, FAKE, None), -1),          # NULL codes
    ((FAKE, 0, 5120, 8, 4, 12, 256, FAKE, None), -1),          # NULL scales
    ((FAKE, FAKE, 5120, 8, 4, 12, 256, 0, None), -1),          # NULL out
    ((FAKE, FAKE, 5120, 8, 9, 12, 256, FAKE, None), -3),       # k = 9
    ((FAKE, FAKE, 5120, 8, 0, 12, 256, FAKE, None), -3),       # k = 0
    ((FAKE, FAKE, 5120, 8, 4, 4, 256, FAKE, None), -3),        # L = k
    ((FAKE, FAKE, 5120, 8, 8, 7, 256, FAKE, None), -3),        # L < k
    ((FAKE, FAKE, 5120, 8, 4, 25, 256, FAKE, None), -3),       # L = 25
    ((FAKE, FAKE, 5120, 8, 4, 12, 128, FAKE, None), -3),       # T = 128
    ((FAKE, FAKE, 5000, 8, 4, 12, 256, FAKE, None), -2),       # K % T != 0
    ((FAKE, FAKE, 0, 8, 4, 12, 256, FAKE, None), -2),          # K = 0
    ((FAKE, FAKE, 5120, 0, 4, 12, 256, FAKE, None), -2),       # N = 0
    ((FAKE, FAKE, 5120, -3, 4, 12, 256, FAKE, None), -2),      # N < 0
    ((FAKE + 4, FAKE, 5120, 8, 4, 12, 256, FAKE, None), -4),   # codes not 16-B aligned
    ((FAKE, FAKE + 1, 5120, 8, 4, 12, 256, FAKE, None), -4),   # scales odd address
    ((FAKE, FAKE, 5120, 8, 4, 12, 256, FAKE + 8, None), -4),   # out not 16-B aligned
    ((FAKE, FAKE, 2 ** 30, 2 ** 20, 4, 12, 256, FAKE, None), -2),   # too many (row, block) items
])
def test_decode_rejects(lib, args, want):
    assert lib.trellis_decode(*args) == want


@pytest.mark.parametrize("M,K,N,k,L,T,want", [
    (0, 5120, 64, 4, 12, 256, -3), (-1, 5120, 64, 4, 12, 256, -3), (65537, 5120, 64, 4, 12, 256, -3),
    (5, 5120, 64, 9, 12, 256, -3), (5, 5120, 64, 2, 2, 256, -3), (5, 5120, 64, 2, 25, 256, -3),
    (5, 5120, 64, 4, 12, 512, -3), (5, 5000, 64, 4, 12, 256, -2), (5, 5120, 0, 4, 12, 256, -2),
])
def test_gemm_rejects(lib, M, K, N, k, L, T, want):
    assert lib.trellis_gemm(FAKE, FAKE, FAKE, M, K, N, k, L, T, FAKE, None) == want
    assert lib.trellis_gemm_ws(FAKE, FAKE, FAKE, M, K, N, k, L, T, FAKE, FAKE, 1 << 20, None) == want
    n = ctypes.c_size_t(0)
    assert lib.trellis_gemm_workspace_size(M, K, N, k, L, T, ctypes.byref(n)) == want


@pytest.mark.parametrize("M", [17, 63, 64, 65, 128, 1000, 65536])
@pytest.mark.parametrize("k,L", [(4, 12), (1, 2), (8, 24), (5, 16)])
def test_tensor_core_m_needs_no_workspace(lib, M, k, L):
    n = ctypes.c_size_t(123)
    assert lib.trellis_gemm_workspace_size(M, 5120, 17408, k, L, 256, ctypes.byref(n)) == 0
    assert n.value == 0


def test_m64_checks_pointers(lib):
    # rejected before any launch: NULL / misaligned pointers, bad geometry
    assert lib.trellis_gemm(0, FAKE, FAKE, 64, 5120, 64, 4, 12, 256, FAKE, None) == -1
    assert lib.trellis_gemm(FAKE + 2, FAKE, FAKE, 64, 5120, 64, 4, 12, 256, FAKE, None) == -4
    assert lib.trellis_gemm(FAKE, FAKE, FAKE, 64, 5000, 64, 4, 12, 256, FAKE, None) == -2
    assert lib.trellis_gemm(FAKE, FAKE, FAKE, 64, 5120, 64, 9, 12, 256, FAKE, None) == -3
    assert lib.trellis_gemm(FAKE, FAKE, FAKE, 64, 5120, 64, 5, 5, 256, FAKE, None) == -3


def test_gemm_rejects_pointers(lib):
    assert lib.trellis_gemm(0, FAKE, FAKE, 5, 5120, 64, 4, 12, 256, FAKE, None) == -1
    assert lib.trellis_gemm(FAKE, FAKE, FAKE, 5, 5120, 64, 4, 12, 256, 0, None) == -1
    assert lib.trellis_gemm(FAKE + 2, FAKE, FAKE, 5, 5120, 64, 4, 12, 256, FAKE, None) == -4
    assert lib.trellis_gemm(FAKE, FAKE + 4, FAKE, 5, 5120, 64, 4, 12, 256, FAKE, None) == -4
    assert lib.trellis_gemm(FAKE, FAKE, FAKE, 5, 5120, 64, 4, 12, 256, FAKE + 1, None) == -4
    assert lib.trellis_gemm_workspace_size(5, 5120, 64, 4, 12, 256, None) == -1


def test_product_path_has_no_oracle_import():
    """The package never imports the oracle (the oracle is test infrastructure)."""
    pkg = os.path.join(ROOT, "trellis_quantized_weight_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), f
                assert "trellis_oracle" not in src and "liboracle" not in src, f


def _packed_args(rows, xs=None, outs=None):
    n = len(rows)
    r = (ctypes.c_int * max(n, 1))(*rows) if rows is not None else None
    xp = (ctypes.c_void_p * max(n, 1))(*(xs if xs is not None else [FAKE] * n))
    op = (ctypes.c_void_p * max(n, 1))(*(outs if outs is not None else [FAKE] * n))
    return xp, r, op


@pytest.mark.parametrize("rows,xs,outs,k,L,want", [
    ([], None, None, 4, 12, -2),                         # no groups
    ([3, 0, 2], None, None, 4, 12, -2),                  # an empty group
    ([3, -1], None, None, 4, 12, -2),                    # a negative row count
    ([40000, 30000], None, None, 4, 12, -3),             # M = 70000 > 65536
    ([3, 5], [FAKE, 0], None, 4, 12, -1),                # NULL x of group 1
    ([3, 5], None, [0, FAKE], 4, 12, -1),                # NULL out of group 0
    ([3, 5], [FAKE, FAKE + 8], None, 4, 12, -4),         # x of group 1 not 16-B aligned
    ([3, 5], None, [FAKE, FAKE + 1], 4, 12, -4),         # odd out address
    ([30, 40], None, None, 9, 12, -3),                   # k = 9
    ([30, 40], None, None, 4, 4, -3),                    # L = k
    ([30, 40], None, None, 4, 12, -7),                   # workspace of 256 bytes (needs MiBs)
])
def test_packed_rejects(lib, rows, xs, outs, k, L, want):
    xp, r, op = _packed_args(rows, xs, outs)
    assert lib.trellis_gemm_packed(xp, r, len(rows), FAKE, FAKE, 5120, 64, k, L, 256, op, FAKE, 256, None) == want


def test_packed_rejects_null_arrays(lib):
    xp, r, op = _packed_args([3, 5])
    assert lib.trellis_gemm_packed(None, r, 2, FAKE, FAKE, 5120, 64, 4, 12, 256, op, FAKE, 1 << 30, None) == -1
    assert lib.trellis_gemm_packed(xp, None, 2, FAKE, FAKE, 5120, 64, 4, 12, 256, op, FAKE, 1 << 30, None) == -1
    assert lib.trellis_gemm_packed(xp, r, 2, FAKE, FAKE, 5120, 64, 4, 12, 256, None, FAKE, 1 << 30, None) == -1
    assert lib.trellis_gemm_packed(xp, r, 2, 0, FAKE, 5120, 64, 4, 12, 256, op, FAKE, 1 << 30, None) == -1


def test_packed_workspace_size_on_the_tensor_core_path(lib):
    """M > 16 needs no product workspace, but the counter region (1 MiB) stays
    reserved ahead of the packed x and output."""
    rows, K, N = [30, 40], 5120, 17408
    r = (ctypes.c_int * 2)(*rows)
    n = ctypes.c_size_t(0)
    assert lib.trellis_gemm_packed_workspace_size(r, 2, K, N, 4, 12, 256, ctypes.byref(n)) == 0
    r256 = lambda b: (b + 255) // 256 * 256
    assert n.value == (1 << 20) + r256(70 * K * 2) + r256(70 * N * 2)
    one = (ctypes.c_int * 1)(70)
    assert lib.trellis_gemm_packed_workspace_size(one, 1, K, N, 4, 12, 256, ctypes.byref(n)) == 0
    assert n.value == 0    # one group runs in place on the tensor cores
    assert lib.trellis_gemm_packed_workspace_size(r, 2, K, N, 4, 12, 256, None) == -1


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++11")])
def test_header_compiles_without_cuda_headers(tmp_path, lang, std):
    """include/trellis.h is a plain C ABI: it compiles as C99 and as C++ with
    no CUDA header on the include path, and its prototypes match pointers of
    the documented types."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / "abi_check.c"
    src.write_text(
        '#include "trellis.h"\n'
        "int main(void) {\n"
        "    int (*gemm)(const uint16_t *, const uint32_t *, const uint16_t *, int, int, int, int, int, int,\n"
        "                uint16_t *, cudaStream_t) = trellis_gemm;\n"
        "    int (*dec)(const uint32_t *, const uint16_t *, int, int, int, int, int, uint16_t *,\n"
        "               cudaStream_t) = trellis_decode;\n"
        "    const char *(*name)(int) = trellis_status_string;\n"
        "    (void)gemm; (void)dec; (void)name;\n"
        "    return TRELLIS_OK;\n"
        "}\n")
    r = subprocess.run([cc, "-x", lang, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_abi_and_oracle_accept_the_same_geometries(lib):
    """The library and the oracle agree on which (k, L, T) are valid: the ABI's
    workspace query at M = 64 validates without touching a device, the oracle's
    geometry check is its own code."""
    import oracle
    o = oracle.get()
    n = ctypes.c_size_t(0)
    for k in range(0, 10):
        for L in range(0, 27):
            for T in (128, 256, 512):
                abi_ok = lib.trellis_gemm_workspace_size(64, 1024, 64, k, L, T, ctypes.byref(n)) == 0
                oracle_ok = o.lib.oracle_check_geometry(1024, 64, k, L, T) == 0
                if T == 256:
                    assert abi_ok == oracle_ok, (k, L, T)
                else:
                    assert not abi_ok, (k, L, T)   # the library takes the pages' block length only
