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


def _float_const(name: str) -> float:
    m = re.search(rf"constexpr\s+float\s+{name}\s*=\s*(0x[0-9a-fA-F.]+p[-+]?\d+)f;", HEADER.read_text())
    assert m, f"{name} not found in {HEADER.name}"
    return float.fromhex(m.group(1))


def test_two_part_reciprocal_rounds_every_code_correctly():
    """The kernels compute value = fma(code, kRecipLo, code * kRecipHi) in fp32.
    Checked here for every code in [-510, 510] with exact rationals: the product
    code * kRecipHi is exact, and the FMA's single rounding of
    code * kRecipLo + code * kRecipHi gives the fp32 nearest to code / c."""
    import sys
    sys.path.insert(0, str(pathlib.Path(__file__).resolve().parent))
    from fractions import Fraction
    import pins
    hi, lo = Fraction(_float_const("kRecipHi")), Fraction(_float_const("kRecipLo"))
    assert hi.numerator < (1 << 14) and (hi.denominator & (hi.denominator - 1)) == 0, "kRecipHi: 14 bits"
    assert Fraction(float(pins.rn_f32(1 / pins.C_DIV - hi))) == lo, "kRecipLo is fp32(1/c - kRecipHi)"
    for code in range(-510, 511):
        prod = code * hi
        assert Fraction(float(pins.rn_f32(prod))) == prod, code
        got = pins.rn_f32(code * lo + prod)
        assert got == pins.value_exact(code), code
