"""The CPU oracle pinned to the page's definition (no GPU needed).

Definition: page "mlx-bun 0.2.0 -> 0.4.0", package/src/model/trellis-wide-prefill.ts,
wide-prefill kernel body (window, hash, quotient, scale, bf16 rounding, product).
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_pages_residual_quotient_equals_ieee_quotient():
    """The page's residual-corrected quotient is the correctly rounded fp32 quotient
    for every code the hash can produce, which is the reading the oracle uses."""
    for c in range(-510, 511):
        assert pins.value_pages_residual_form(c) == pins.value_exact(c), c


def test_plain_reciprocal_product_is_not_enough():
    """code * fp32(1/c) alone misses the correctly rounded quotient for some codes,
    so the correction step of the page is needed (and the oracle's division is not
    interchangeable with a reciprocal multiply)."""
    r = pins.rn_f32(1 / pins.C_DIV)
    bad = [c for c in range(-510, 511)
           if np.float32(np.float32(c) * r) != pins.value_exact(c)]
    assert len(bad) > 0


def test_hash_realised_range(oracle_lib):
    """Over all 12-bit windows the code stays inside the closed-form bound [-510, 510]
    and the value inside |v| <= 510 / 147.800537109375."""
    codes = np.array([oracle_lib.code(w) for w in range(4096)])
    assert codes.min() >= -510 and codes.max() <= 510
    assert codes.min() == min(pins.code_bytesum(w) for w in range(4096))
    assert 510 / 147.800537109375 < 3.4506


# --- planted mistakes: each mutation of the oracle must fail at least one pin ---
MUTATIONS = {
    "wrap_to_word1": ("? 0u : wi + 1u", "? 1u : wi + 1u"),
    "forward_bit_order": ("(uint32_t)(T - 1 - t) * (uint32_t)k", "(uint32_t)t * (uint32_t)k"),
    "bias_off_by_one": ("(p >> 16)) - 510;", "(p >> 16)) - 511;"),
    "hash_addend": ("76625530u", "76625531u"),
    "hash_multiplier": ("34038481u", "34038483u"),
    "reciprocal_multiply": ("return (float)code / c;", "return (float)code * (1.0f / c);"),
    "bf16_truncate": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;"),
    "bf16_ties_away": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "short_mask": ("win &= (1u << L) - 1u;", "win &= (1u << (L - 1)) - 1u;"),
    "no_straddle": ("if (off + (uint32_t)L > 32u) {", "if (off + (uint32_t)L > 64u) {"),
    "scale_row0": ("oracle_weight(blk, t, k, L, T, scales[n])", "oracle_weight(blk, t, k, L, T, scales[0])"),
    "gemm_x_row0": ("(double)oracle_bf16_to_f32(x[m * K + kk])", "(double)oracle_bf16_to_f32(x[kk])"),
    "gemm_transposed_w": ("oracle_bf16_to_f32(W[i * K + kk])", "oracle_bf16_to_f32(W[kk * nrows + i])"),
    "silu_is_sigmoid": ("const double s = v / (1.0 + exp(-v));", "const double s = 1.0 / (1.0 + exp(-v));"),
    "silu_sign": ("const double s = v / (1.0 + exp(-v));", "const double s = v / (1.0 + exp(v));"),
    "silu_gate_up_swapped": ("const double v = (double)oracle_bf16_to_f32(g[i]);",
                             "const double v = (double)oracle_bf16_to_f32(u[i]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    import oracle
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "trellis_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    try:
        path = os.path.join(d, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.Oracle(oracle.compile_source(path, os.path.join(d, "libmut.so")))
        caught = []
        for pin in pins.ALL_PINS:
            try:
                pin(lib)
            except (AssertionError, ValueError, IndexError):
                caught.append(pin.__name__)
                break
        assert caught, f"no pin caught the planted mistake {name}"
    finally:
        shutil.rmtree(d, ignore_errors=True)
