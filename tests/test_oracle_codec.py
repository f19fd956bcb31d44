"""Pins of the oracle's FP8 codec (E4M3 "FN" and E5M2, OCP 8-bit floating point spec).

The formats are the ones the LLMQ summary names for FP8 training (§5, Figure 2: E4M3 forward,
E5M2 activation gradients); their encodings are the OCP spec's.  The pins:
  * decode anchors listed by hand (max values, smallest subnormals, 1.0, NaN/Inf codes);
  * the decode table is strictly increasing over the positive finite codes, and the positive
    finite set equals an independently characterised set (multiples of the smallest subnormal
    with at most 1+frac significant bits, up to the maximum);
  * encode against a brute-force nearest-value search over that independent set (ties to the
    even code, saturation at +-max) on every fp32 bit pattern whose low 16 bits are one of the
    rounding-boundary neighbourhoods, on all 65536 high halves, plus a random sample.
"""

import numpy as np
import pytest

import oracle

FORMATS = {
    # fmt: (frac bits, log2 smallest subnormal, max, number of positive finite codes incl. zero)
    oracle.E4M3: (3, -9, 448.0, 127),
    oracle.E5M2: (2, -16, 57344.0, 124),
}


def test_decode_anchors():
    d4 = oracle.fp8_decode(np.arange(256, dtype=np.uint8), oracle.E4M3)
    assert d4[0x7E] == 448.0 and d4[0xFE] == -448.0
    assert d4[0x01] == 2.0 ** -9 and d4[0x08] == 2.0 ** -6 and d4[0x07] == 7 * 2.0 ** -9
    assert d4[0x38] == 1.0 and d4[0x40] == 2.0 and d4[0x3C] == 1.5
    assert d4[0x00] == 0.0 and d4[0x80] == 0.0 and np.signbit(d4[0x80])
    assert np.isnan(d4[0x7F]) and np.isnan(d4[0xFF])
    assert np.isfinite(np.delete(d4, [0x7F, 0xFF])).all()     # E4M3 FN has no infinities

    d5 = oracle.fp8_decode(np.arange(256, dtype=np.uint8), oracle.E5M2)
    assert d5[0x7B] == 57344.0 and d5[0xFB] == -57344.0
    assert d5[0x01] == 2.0 ** -16 and d5[0x04] == 2.0 ** -14 and d5[0x03] == 3 * 2.0 ** -16
    assert d5[0x3C] == 1.0 and d5[0x3E] == 1.5
    assert d5[0x7C] == np.inf and d5[0xFC] == -np.inf
    assert all(np.isnan(d5[c]) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))


def independent_positive_set(fmt):
    """Positive finite values characterised without exponent/mantissa fields: multiples k*2^emin_sub
    (k >= 0) whose k has at most frac+1 significant bits, not above max."""
    frac, lsub, vmax, count = FORMATS[fmt]
    kmax = int(vmax / 2.0 ** lsub)
    ks = {m << j for m in range(1 << (frac + 1)) for j in range(64) if (m << j) <= kmax}
    vals = np.array(sorted(k * 2.0 ** lsub for k in ks))
    assert vals.size == count
    return vals


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_positive_codes_are_the_independent_set_in_order(fmt):
    vals = independent_positive_set(fmt)
    dec = oracle.fp8_decode(np.arange(vals.size, dtype=np.uint8), fmt)
    np.testing.assert_array_equal(dec, vals)
    neg = oracle.fp8_decode(np.arange(vals.size, dtype=np.uint8) | 0x80, fmt)
    np.testing.assert_array_equal(neg, -vals)


def brute_force_encode(v32: np.ndarray, fmt) -> np.ndarray:
    """Nearest element of the independent set, ties to the even code, saturation, sign kept."""
    vals = independent_positive_set(fmt)
    a = np.abs(v32.astype(np.float64))
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, vals.size - 1)
    lo = hi - 1
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= vals[-1], vals.size - 1, pick)          # saturate (incl. +-inf)
    code = pick.astype(np.uint8) | np.where(np.signbit(v32), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(v32), np.uint8(0x7F), code)


def boundary_patterns(seed=1234):
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    rnd = np.random.default_rng(seed).integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([pats, rnd]).view(np.float32)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_brute_force(fmt):
    v = boundary_patterns()
    got = oracle.fp8_encode(v, fmt)
    want = brute_force_encode(v, fmt)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {v[bad[:5]]}: got {got[bad[:5]]} want {want[bad[:5]]}"


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_decode_roundtrip(fmt):
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.fp8_decode(codes, fmt)
    finite = np.isfinite(dec)
    back = oracle.fp8_encode(dec[finite].astype(np.float32), fmt)
    np.testing.assert_array_equal(back, codes[finite])


def test_bf16_round_single_rounding():
    # 1 + 2^-8 is the midpoint of bf16 1 and 1+2^-7: ties to even -> 1.
    # 1 + 2^-8 + 2^-30 is above the midpoint (a detour through fp32 would lose the 2^-30 and tie).
    v = np.array([1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -30, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.5e38, -0.0])
    got = oracle.bf16_round(v)
    assert list(got) == [0x3F80, 0x3F81, 0x3F82, 0xBF80, 0x7F80, 0x8000]
