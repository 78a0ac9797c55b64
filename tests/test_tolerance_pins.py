"""Pins of the product tolerance that every GPU product parity check uses.

The tolerance is the one stated for the decode-and-multiply: an output may
differ from the oracle's exactly summed fp32 result by at most
max(2 bf16 ulp of that result, 1e-4 * sum_k |w_k x_k|).  ``oracle.ulp_bf16``
and ``oracle.gemm_tolerance`` implement it; these checks pin both to facts
that do not come from their code:

* the bf16 format itself: for every positive finite bf16 bit pattern below
  the largest (subnormals included) the spacing is the value of the next
  pattern minus its own, and an fp32 value inside a binade has the spacing of
  that binade;
* values worked by hand: ulp(1) = ulp(1.5) = 2^-7, ulp(3) = 2^-6,
  ulp(0.75) = 2^-8, ulp(v) = 2^-133 below 2^-126, and both branches of the
  maximum on small cases;
* planted mistakes in a copy of the two functions, each caught by a pin.
"""
import inspect

import numpy as np
import pytest

import oracle


def bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# pins: each takes a namespace holding ulp_bf16 and gemm_tolerance
# ----------------------------------------------------------------------------
def pin_ulp_hand_worked(t):
    # bf16 keeps 8 significant bits, so the spacing in [2^e, 2^(e+1)) is 2^(e-7)
    cases = [(1.0, 2.0 ** -7), (1.5, 2.0 ** -7), (3.0, 2.0 ** -6), (0.75, 2.0 ** -8),
             (-2.0, 2.0 ** -6), (2.0 - 2.0 ** -23, 2.0 ** -7), (1000.0, 2.0 ** 2),
             (0.0, 2.0 ** -133), (2.0 ** -130, 2.0 ** -133), (-(2.0 ** -127), 2.0 ** -133),
             (2.0 ** -126, 2.0 ** -133), (3.4506, 2.0 ** -6)]
    v = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases])
    got = np.asarray(t.ulp_bf16(v), dtype=np.float64)
    assert np.array_equal(got, want), list(zip(v, got, want))


def pin_ulp_is_the_bf16_spacing(t):
    """Exhaustive over the positive finite bf16 patterns: ulp(v) = next(v) - v."""
    bits = np.arange(0x0001, 0x7F7F, dtype=np.uint32)       # 0x7F7F is the largest finite
    v = bf16_value(bits)
    spacing = bf16_value(bits + 1) - v
    got = np.asarray(t.ulp_bf16(v), dtype=np.float64)
    assert np.array_equal(got, spacing)
    assert np.array_equal(np.asarray(t.ulp_bf16(-v), dtype=np.float64), spacing)   # sign-blind
    # an fp32 value strictly inside a binade has the binade's spacing
    mid = (v[:-1] + 0.25 * spacing[:-1]).astype(np.float32).astype(np.float64)
    inside = (mid > v[:-1]) & (mid < v[1:])
    assert np.array_equal(np.asarray(t.ulp_bf16(mid[inside]), dtype=np.float64), spacing[:-1][inside])


def pin_tolerance_hand_worked(t):
    # (ref, sum |w x|, allowed): the larger of 2 ulp and 1e-4 of the absolute sum
    cases = [(1.0, 10.0, 2 * 2.0 ** -7),        # 2 ulp = 0.015625 > 0.001
             (1.0, 1000.0, 0.1),                 # 1e-4 * 1000 = 0.1 > 0.015625
             (-3.0, 0.0, 2 * 2.0 ** -6),
             (0.0, 0.0, 2 * 2.0 ** -133),
             (0.5, 39.0625, 2 * 2.0 ** -8),      # 1e-4 * 39.0625 = 0.00390625 < 2 ulp
             (0.5, 78.125, 2 * 2.0 ** -8),       # both branches equal: 0.0078125
             (0.5, 100.0, 0.01),
             (96.0, 12.0, 2 * 2.0 ** -1)]
    ref = np.array([c[0] for c in cases], dtype=np.float32)
    refabs = np.array([c[1] for c in cases], dtype=np.float64)
    want = np.array([c[2] for c in cases])
    got = np.asarray(t.gemm_tolerance(ref, refabs), dtype=np.float64)
    assert np.allclose(got, want, rtol=1e-15, atol=0.0), list(zip(ref, refabs, got, want))
    assert got.shape == ref.shape


ALL_TOL_PINS = [pin_ulp_hand_worked, pin_ulp_is_the_bf16_spacing, pin_tolerance_hand_worked]


@pytest.mark.parametrize("pin", ALL_TOL_PINS, ids=lambda p: p.__name__)
def test_tolerance_pin(pin):
    pin(oracle)


def test_checker_accepts_the_bound_and_rejects_beyond_it():
    """assert_gemm_close passes an error equal to the tolerance and fails the next bf16 value."""
    from helpers import assert_gemm_close
    ref = np.array([[1.0]], dtype=np.float32)
    refabs = np.array([[10.0]])                        # tolerance max(2 * 2^-7, 1e-3) = 2^-6
    on_bound = np.array([[0x3F82]], dtype=np.uint16)   # 1 + 2 * 2^-7: error exactly 2 ulp
    beyond = np.array([[0x3F83]], dtype=np.uint16)     # 1 + 3 * 2^-7
    assert bf16_value(0x3F82) - 1.0 == 2 * 2.0 ** -7
    assert bf16_value(0x3F83) - 1.0 == 3 * 2.0 ** -7
    assert_gemm_close(on_bound, ref, refabs, "on the bound")
    with pytest.raises(AssertionError):
        assert_gemm_close(beyond, ref, refabs, "beyond the bound")


def test_helpers_use_the_oracle_tolerance():
    """The tests have one bf16 spacing function: the oracle's."""
    import helpers
    assert helpers.ulp_bf16_of is oracle.ulp_bf16


# --- planted mistakes in a copy of the tolerance functions ---------------------
TOL_MUTATIONS = {
    "ulp_exponent_off_by_one": ("e - 7", "e - 6"),
    "ulp_exponent_off_by_one_low": ("e - 7", "e - 8"),
    "dropped_factor_two": ("2.0 * ulp_bf16(ref)", "ulp_bf16(ref)"),
    "relative_term_1e3": ("1e-4 * np.asarray", "1e-3 * np.asarray"),
    "min_instead_of_max": ("return np.maximum(2.0", "return np.minimum(2.0"),
    "no_min_normal_floor": ("np.maximum(a, 2.0 ** -126)", "np.maximum(a, 2.0 ** -149)"),
    "round_not_floor": ("np.floor(np.log2", "np.round(np.log2"),
    "ceil_not_floor": ("np.floor(np.log2", "np.ceil(np.log2"),
}


def _tolerance_copy(src: str):
    ns = {"np": np}
    exec(compile(src, "<tolerance copy>", "exec"), ns)
    return type("TolCopy", (), {"ulp_bf16": staticmethod(ns["ulp_bf16"]),
                                "gemm_tolerance": staticmethod(ns["gemm_tolerance"])})


def _tolerance_source() -> str:
    return inspect.getsource(oracle.ulp_bf16) + "\n" + inspect.getsource(oracle.gemm_tolerance)


def test_unmutated_copy_passes_every_pin():
    copy = _tolerance_copy(_tolerance_source())
    for pin in ALL_TOL_PINS:
        pin(copy)


@pytest.mark.parametrize("name", sorted(TOL_MUTATIONS))
def test_planted_tolerance_mistake_is_caught(name):
    old, new = TOL_MUTATIONS[name]
    src = _tolerance_source()
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    copy = _tolerance_copy(src.replace(old, new))
    caught = []
    for pin in ALL_TOL_PINS:
        try:
            pin(copy)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
