"""The KV codec's scale s = fp16_RN(fp32_RN(amax / qmax)) takes its fp32
quotient from a multiply by y = fp32_RN(1 / qmax) corrected by one fused
multiply-add with the remainder (division by a constant, Cornea, Harrison and
Tang). This checks, for qmax in {7, 31, 127} and every positive finite fp16
amax, that the corrected quotient is the correctly rounded one, in exact
rational arithmetic (host logic; no GPU)."""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest


def _rn32(v: Fraction) -> Fraction:
    """v rounded to the nearest binary32 value, ties to even (v > 0, normal range)."""
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    k, rem = divmod(v, ulp)
    if rem * 2 > ulp or (rem * 2 == ulp and k % 2 == 1):
        k += 1
    return k * ulp


def _fma_div(x: Fraction, c: int) -> Fraction:
    y = _rn32(Fraction(1, c))
    q = _rn32(x * y)
    r = x - q * c          # exact: the fma's product and sum before its one rounding
    r = _rn32(r) if r > 0 else (-_rn32(-r) if r < 0 else Fraction(0))
    t = r * y + q
    return _rn32(t)


@pytest.mark.parametrize("qmax", [7, 31, 127])
def test_fma_corrected_division_is_correctly_rounded(qmax):
    h = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    bad = [x for x in h if _fma_div(Fraction(float(x)), qmax) != _rn32(Fraction(float(x)) / qmax)]
    assert not bad, f"qmax {qmax}: {len(bad)} fp16 magnitudes round differently, e.g. {bad[:3]}"


def test_rn32_matches_numpy_float32():
    # the rounding helper agrees with numpy's float64 -> float32 conversion on
    # values a double holds exactly
    rng = np.random.default_rng(0)
    for v in rng.uniform(1e-6, 1e6, 200):
        assert _rn32(Fraction(float(v))) == Fraction(float(np.float32(v)))


def test_kernel_reciprocals_are_the_rounded_ones():
    # the constants the kernel multiplies by are RN(1 / qmax)
    import pathlib
    import re
    src = (pathlib.Path(__file__).resolve().parents[1] / "quantized_weight_exq_gb300" / "csrc" / "exq_kv.cu").read_text()
    m = re.search(r"C == 7 \? (\S+)f : C == 31 \? (\S+)f : (\S+)f;", src)
    assert m, "div_by_const's constants not found"
    for c, hx in zip((7, 31, 127), m.groups()):
        assert Fraction(float.fromhex(hx)) == _rn32(Fraction(1, c)), (c, hx)


@pytest.mark.parametrize("qmax", [7, 31, 127])
def test_normal_scale_keeps_codes_in_range(qmax):
    # The write kernel clamps q only for subnormal scales. For every positive
    # finite fp16 amax whose scale s = fp16_RN(fp32_RN(amax / qmax)) is a
    # normal fp16, amax / s stays below qmax + 1/2 by more than the 2^-15 by
    # which the kernel's quotient may differ from fp32_RN(x / s), so
    # rint(x / s) is within [-qmax, qmax] for every |x| <= amax. Exhaustive
    # over the fp16 magnitudes, exact rational arithmetic for the ratio.
    h = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16)
    s = (h.astype(np.float32) / np.float32(qmax)).astype(np.float16)
    normal = s.astype(np.float64) >= 2.0 ** -14
    assert normal.any()
    worst = max(Fraction(float(a)) / Fraction(float(b)) for a, b in zip(h[normal], s[normal]))
    assert worst + Fraction(1, 2 ** 15) < Fraction(2 * qmax + 1, 2), (qmax, float(worst))
