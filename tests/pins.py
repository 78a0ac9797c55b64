"""Independent checks that pin the CPU oracle to the definition on the pages.

Each check re-derives a fact from a formulation other than the oracle's own
code: explicit bit arrays instead of shifts and masks, the byte sum instead of
the masked add, exact rational rounding instead of fp32 division, torch's bf16
conversion, numpy's float64 matmul, closed forms and invariants.  Every
function takes an ``oracle.Oracle`` and raises ``AssertionError`` on a
mismatch, so the mutation tests can run the same checks against an oracle with
a planted mistake.

The definition: page "mlx-bun 0.2.0 -> 0.4.0",
package/src/model/trellis-wide-prefill.ts, body of the wide-prefill kernel.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

C_DIV = Fraction(147.800537109375)   # exactly representable in fp32
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# independent formulations
# ----------------------------------------------------------------------------
def block_bits(words: np.ndarray) -> np.ndarray:
    """The block's bit-string: bit j is bit (j mod 32) of word (j div 32), lsb first."""
    w = np.ascontiguousarray(words, dtype="<u4")
    return np.unpackbits(w.view(np.uint8), bitorder="little")


def window_brute(words: np.ndarray, t: int, k: int, L: int, T: int) -> int:
    """Window bit i of weight t is bit ((T-1-t)*k + i) mod (T*k) of the block (tail-biting)."""
    bits = block_bits(words)
    n = T * k
    assert bits.size == n
    start = (T - 1 - t) * k
    return sum(int(bits[(start + i) % n]) << i for i in range(L))


def code_bytesum(win: int) -> int:
    """code = (sum of the four bytes of win*34038481 + 76625530 mod 2^32) - 510."""
    z = (win * 34038481 + 76625530) % (1 << 32)
    return sum(z.to_bytes(4, "little")) - 510


def rn_f32(q: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to even); normal range only."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    assert -126 <= e <= 127
    scale = Fraction(2) ** (e - 23)
    m = a / scale                      # in [2^23, 2^24)
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return np.float32(sign * float(fl * scale))


def value_exact(code: int) -> np.float32:
    return rn_f32(Fraction(code) / C_DIV)


def value_pages_residual_form(code: int) -> np.float32:
    """The page's three-step quotient, each fp32 step rounded exactly once:
    approx = code*r, residual = fma(-approx, c, code), value = fma(residual, r, approx)."""
    r = rn_f32(1 / C_DIV)
    cf = Fraction(code)
    approx = rn_f32(cf * Fraction(float(r)))
    residual = rn_f32(cf - Fraction(float(approx)) * C_DIV)
    return rn_f32(Fraction(float(residual)) * Fraction(float(r)) + Fraction(float(approx)))


def bf16_bits_torch(f32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def decode_independent(codes: np.ndarray, scales: np.ndarray, K: int, N: int, k: int,
                       L: int = 12, T: int = 256) -> np.ndarray:
    """Dense bf16 bits built from the independent formulations above (slow; small inputs)."""
    wpb = T * k // 32
    vtab = {c: value_exact(c) for c in range(-510, 511)}
    out = np.empty((N, K), dtype=np.float32)
    for n in range(N):
        s = bf16_to_f32(np.array([scales[n]], dtype=np.uint16))[0]
        for b in range(K // T):
            blk = codes[n, b * wpb:(b + 1) * wpb]
            bits = block_bits(blk)
            nb = T * k
            for t in range(T):
                start = (T - 1 - t) * k
                win = 0
                for i in range(L):
                    win |= int(bits[(start + i) % nb]) << i
                out[n, b * T + t] = np.float32(vtab[code_bytesum(win)]) * np.float32(s)
    return bf16_bits_torch(out)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def read_golden(name: str):
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            s = line.strip()
            if s.startswith("# section:"):
                cur = s.split(":", 1)[1].strip()
                sections[cur] = []
            elif s and not s.startswith("#"):
                sections[cur].append(s.split())
    return sections


def pin_golden_worked_examples(o):
    g = read_golden("decode_worked_examples.txt")
    for win, zhex, b0, b1, b2, b3, bsum, code in g["hash"]:
        win, code = int(win), int(code)
        z = int(zhex, 16)
        assert list(z.to_bytes(4, "little")) == [int(b0), int(b1), int(b2), int(b3)]
        assert int(b0) + int(b1) + int(b2) + int(b3) == int(bsum)
        assert o.code(win) == code, (win, o.code(win), code)
    for k, word, scale, weight in g["block"]:
        k, T = int(k), 256
        blk = np.full(T * k // 32, int(word, 16), dtype=np.uint32)
        for t in range(T):
            assert o.weight(blk, t, k, 12, T, int(scale, 16)) == int(weight, 16), (k, word, t)


def pin_window_bruteforce(o, seed=1234):
    """Windows against the explicit bit-string, on random and crafted single blocks."""
    rng = np.random.default_rng(seed)
    # the pages' k in {2,3,4} with L = 12, then the general geometry 1 <= k <= 8,
    # k < L <= 24, including every k and the narrowest and widest windows
    for k, L in [(2, 12), (3, 12), (4, 12), (1, 12), (5, 12), (6, 16), (8, 16), (4, 24), (2, 9),
                 (7, 12), (7, 20), (1, 2), (1, 24), (8, 9), (8, 24), (3, 4)]:
        T = 256
        wpb = T * k // 32
        blocks = [rng.integers(0, 2 ** 32, wpb, dtype=np.uint64).astype(np.uint32) for _ in range(3)]
        last = np.zeros(wpb, np.uint32); last[-1] = 0xFFFFFFFF
        first = np.zeros(wpb, np.uint32); first[0] = 0x00000FFF
        blocks += [last, first]
        for bit in [0, 1, 11, 12, 31, 32, T * k - 12, T * k - 1]:     # single 1-bit blocks
            one = np.zeros(wpb, np.uint32)
            one[bit // 32] = np.uint32(1 << (bit % 32))
            blocks.append(one)
        for blk in blocks:
            for t in range(T):
                assert o.window(blk, t, k, L, T) == window_brute(blk, t, k, L, T), (k, L, t)


def pin_hash_exhaustive(o):
    codes = [o.code(w) for w in range(4096)]
    for w, c in enumerate(codes):
        assert c == code_bytesum(w), (w, c)
        assert -510 <= c <= 510
    # Beyond 12 bits the hash is the same formula on the wider window.
    for w in [4096, 65535, (1 << 24) - 1, 0xABCDE]:
        assert o.code(w) == code_bytesum(w)


def pin_value_exhaustive(o):
    vmax = 0.0
    for c in range(-510, 511):
        v = o.value(c)
        assert v == value_exact(c), (c, v, value_exact(c))
        vmax = max(vmax, abs(float(v)))
    assert vmax <= 3.4506, vmax


def pin_bf16_rounding(o, seed=7):
    rng = np.random.default_rng(seed)
    f = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    # exact ties: low 16 bits 0x8000 with even and odd kept lsb
    # (finite values near 1: random sign and 7-bit mantissa, exponent 2^-1 or 2^0)
    ties = (rng.integers(0, 2 ** 8, 200, dtype=np.uint32) << np.uint32(16)
            | (rng.integers(0, 2, 200, dtype=np.uint32) << np.uint32(31))
            | np.uint32(0x3F000000) | np.uint32(0x8000)).view(np.float32)
    allf = np.concatenate([f, ties, np.array([0.0, -0.0, 1.0, -2.5, 3.4506], np.float32)])
    want = bf16_bits_torch(allf)
    got = np.array([o.f32_to_bf16(v) for v in allf], dtype=np.uint16)
    assert np.array_equal(got, want)
    for h in [0x3F80, 0xBFA0, 0x3FA3, 0x0001, 0x7F7F]:
        assert o.bf16_to_f32(h) == bf16_to_f32(np.array([h], np.uint16))[0]


def pin_decode_composition(o, seed=99):
    """Whole decode of small matrices against the independent composition."""
    rng = np.random.default_rng(seed)
    # the pages' geometries, then the general-geometry reading (1 <= k <= 8, k < L <= 24)
    for k, L in [(2, 12), (3, 12), (4, 12), (1, 12), (5, 16), (7, 20), (8, 24)]:
        N, K = 3, 512
        codes = rng.integers(0, 2 ** 32, (N, K * k // 32), dtype=np.uint64).astype(np.uint32)
        scales = bf16_bits_torch(rng.uniform(0.005, 0.02, N).astype(np.float32))
        got = o.decode(codes, scales, K, N, k, L=L)
        want = decode_independent(codes, scales, K, N, k, L=L)
        assert np.array_equal(got, want), (k, L)


def pin_scale_linearity(o, seed=5):
    """W(s * 2^j) == 2^j * W(s) exactly; W(1) == bf16(value)."""
    rng = np.random.default_rng(seed)
    N, K, k = 4, 256, 3
    codes = rng.integers(0, 2 ** 32, (N, K * k // 32), dtype=np.uint64).astype(np.uint32)
    s = rng.uniform(0.005, 0.02, N).astype(np.float32)
    base = o.decode(codes, bf16_bits_torch(s), K, N, k)
    for j in (-3, -1, 1, 4):
        sj = bf16_bits_torch(s * np.float32(2.0 ** j))
        got = bf16_to_f32(o.decode(codes, sj, K, N, k))
        assert np.array_equal(got, bf16_to_f32(base) * np.float32(2.0 ** j)), j
    ones = np.full(N, 0x3F80, np.uint16)
    w1 = o.decode(codes, ones, K, N, k)
    for n in range(N):
        for t in (0, 1, 100, 255):
            win = window_brute(codes[n, :K * k // 32], t, k, 12, 256)
            assert w1[n, t] == bf16_bits_torch(np.array([value_exact(code_bytesum(win))]))[0]


def pin_gemm(o, seed=11):
    """Product against numpy's float64 matmul, one-hot columns, and linearity."""
    rng = np.random.default_rng(seed)
    M, K, N = 5, 768, 7
    W = bf16_bits_torch(rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02))
    x = bf16_bits_torch(rng.standard_normal((M, K)).astype(np.float32))
    ref, refabs = o.gemm_dense(x, W)
    Wd = bf16_to_f32(W).astype(np.float64)
    xd = bf16_to_f32(x).astype(np.float64)
    want = xd @ Wd.T
    wabs = np.abs(xd) @ np.abs(Wd).T
    assert ref.shape == (M, N)
    assert np.all(np.abs(ref.astype(np.float64) - want) <= np.abs(want) * 2.0 ** -23 + 1e-12 * wabs)
    assert np.allclose(refabs, wabs, rtol=1e-12)
    # one-hot x picks a weight column exactly
    for j in (0, 17, K - 1):
        e = np.zeros((1, K), np.float32); e[0, j] = 1.0
        r1, _ = o.gemm_dense(bf16_bits_torch(e), W)
        assert np.array_equal(r1[0].astype(np.float32), bf16_to_f32(W[:, j]))
    # linearity in x: x1 and x2 chosen so x1 + x2 is exact in bf16
    x1 = bf16_bits_torch(np.round(rng.standard_normal((2, K)) * 8).astype(np.float32) / 8)
    x2 = bf16_bits_torch(np.round(rng.standard_normal((2, K)) * 8).astype(np.float32) / 8)
    x12 = bf16_bits_torch(bf16_to_f32(x1) + bf16_to_f32(x2))
    a, _ = o.gemm_dense(x1, W)
    b, _ = o.gemm_dense(x2, W)
    c, cab = o.gemm_dense(x12, W)
    assert np.all(np.abs((a.astype(np.float64) + b) - c) <= 1e-6 * (cab + 1e-30) + 1e-30)


def pin_silu_mul(o, seed=21):
    """Gate/up activation act = bf16(silu(g) * u), silu(v) = v / (1 + e^-v).
    Values worked out by hand from that definition: silu(1) = 0.731058...
    -> bf16 0x3F3B (0.73046875); silu(2) = 1.761594... -> 0x3FE1 (1.7578125);
    silu(64) = 64 - 64 e^-64 -> 0x4280 (64.0); silu(0) = 0; with u = 2 the
    product doubles exactly (0x3FBB = 1.4609375).  Also: doubling u doubles
    every result exactly (power-of-two scaling commutes with each rounding)."""
    g = np.array([0x0000, 0x3F80, 0x4000, 0x4280, 0x3F80], np.uint16)
    u = np.array([0x3F80, 0x3F80, 0x3F80, 0x3F80, 0x4000], np.uint16)
    want = np.array([0x0000, 0x3F3B, 0x3FE1, 0x4280, 0x3FBB], np.uint16)
    got = o.silu_mul(g, u)
    assert np.array_equal(got, want), (got, want)
    rng = np.random.default_rng(seed)
    gf = rng.normal(0.0, 2.0, 4096).astype(np.float32)
    uf = rng.normal(0.0, 1.0, 4096).astype(np.float32)
    gb, ub = bf16_bits_torch(gf), bf16_bits_torch(uf)
    ub2 = bf16_bits_torch(2.0 * bf16_to_f32(ub))
    a1 = bf16_to_f32(o.silu_mul(gb, ub))
    a2 = bf16_to_f32(o.silu_mul(gb, ub2))
    assert np.array_equal(a2, 2.0 * a1)


ALL_PINS = [pin_silu_mul, pin_golden_worked_examples, pin_window_bruteforce, pin_hash_exhaustive,
            pin_value_exhaustive, pin_bf16_rounding, pin_decode_composition,
            pin_scale_linearity, pin_gemm]
