"""Pins of the oracle's per-tensor absmax quantizer and scaled FP8 GEMM.

Quantizer (FastML report, "FP8 training without delayed scaling": just-in-time tensor-level absmax
scaling, no clipping; LLMQ §1): hand-worked fixtures; the absmax element lands on +-max; power-of-two
scale invariance; sign symmetry; dequantization error within half an FP8 ulp; amax = 0 and
non-finite inputs.
GEMM (LLMQ §4: the pipeline is dominated by FP8 matmuls): a hand-worked 2x2; exact rational
arithmetic (Python integers) on random small shapes in every layout and format mix; layout
consistency; identity operand; bf16 output with residual.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests._golden import load


def bf16(v):
    return oracle.bf16_round(np.asarray(v, dtype=np.float64))


@pytest.mark.parametrize("name", ["quantize_e4m3_hand.txt", "quantize_e4m3_rounding.txt"])
def test_quantize_hand_worked(name):
    G = load(name)
    x = bf16(G["x"])
    assert (oracle.bf16_to_f64(x) == G["x"]).all()
    q, scal, st = oracle.quantize_absmax(x, oracle.E4M3)
    assert st == 0
    assert scal[0] == np.float32(G["amax"])
    assert scal[1] == np.float32(G["scale"])
    assert scal[2] == np.float32(G["scale_inv"])
    np.testing.assert_array_equal(q, G["codes"])
    # fp32 input path gives the same answer
    q32, scal32, _ = oracle.quantize_absmax(G["x"].astype(np.float32), oracle.E4M3)
    np.testing.assert_array_equal(q32, q)
    np.testing.assert_array_equal(scal32, scal)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_quantize_invariants(fmt):
    rng = np.random.default_rng(11 + fmt)
    v = rng.standard_normal(4096) * np.exp(rng.uniform(-6, 6, 4096))
    x = bf16(v)
    q, scal, st = oracle.quantize_absmax(x, fmt)
    fmax = oracle.FMT_MAX[fmt]
    xv = oracle.bf16_to_f64(x)
    # the absmax element maps to +-max, nothing is clipped
    i = int(np.argmax(np.abs(xv)))
    assert oracle.fp8_decode(q[i:i + 1], fmt)[0] == np.sign(xv[i]) * fmax
    assert scal[0] == np.abs(xv).max()
    # sign symmetry
    qn, scaln, _ = oracle.quantize_absmax(bf16(-oracle.bf16_to_f64(x)), fmt)
    np.testing.assert_array_equal(qn, q ^ 0x80)
    np.testing.assert_array_equal(scaln, scal)
    # power-of-two invariance of the codes
    for k in (-3, 5):
        qk, scalk, _ = oracle.quantize_absmax(bf16(xv * 2.0 ** k), fmt)
        np.testing.assert_array_equal(qk, q)
        assert scalk[1] == scal[1] * np.float32(2.0 ** -k)
    # dequantization error: half an FP8 ulp (relative 2^-(frac+1)) in the normal range, half the
    # subnormal spacing below it (values are fp32 products x*s, rounded once to FP8)
    frac, sub = (3, 2.0 ** -9) if fmt == oracle.E4M3 else (2, 2.0 ** -16)
    p = (xv.astype(np.float32) * scal[1]).astype(np.float64)
    dq = oracle.fp8_decode(q, fmt)
    bound = np.maximum(np.abs(p) * 2.0 ** -(frac + 1), sub / 2)
    assert (np.abs(dq - p) <= bound * (1 + 1e-12)).all()


def test_quantize_zero_and_nonfinite():
    q, scal, st = oracle.quantize_absmax(np.zeros(16, np.uint16), oracle.E4M3)
    assert st == 0 and (q == 0).all() and list(scal) == [0.0, 1.0, 1.0]
    x = np.zeros(8, np.float32)
    x[3] = np.inf
    _, scal, st = oracle.quantize_absmax(x, oracle.E4M3)
    assert st == 1 and scal[0] == np.inf
    x[3] = np.nan
    _, scal, st = oracle.quantize_absmax(x, oracle.E5M2)
    assert st == 1 and np.isnan(scal[0])


# ---------------------------------------------------------------------------- GEMM
def test_gemm_hand_worked():
    G = load("gemm_2x2_hand.txt")
    for A, fa in ((G["A_e4m3"], oracle.E4M3), (G["A_e5m2"], oracle.E5M2)):
        C = oracle.gemm_scaled(oracle.NN, A.reshape(2, 2), fa, G["B_e4m3"].reshape(2, 2), oracle.E4M3,
                               G["sinvA"], G["sinvB"], out="f64")
        np.testing.assert_array_equal(C.ravel(), G["C"])


def exact_value(code, fmt):
    """Exact rational value of an FP8 code, from the decoded double (FP8 values are dyadic)."""
    return Fraction(float(oracle.fp8_decode(np.array([code], np.uint8), fmt)[0]))


def random_codes(rng, shape, fmt):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    nan = (c & 0x7F) == 0x7F if fmt == oracle.E4M3 else (c & 0x7C) == 0x7C
    c[nan] = 0x00
    return c


@pytest.mark.parametrize("layout", [oracle.NN, oracle.NT, oracle.TN])
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_gemm_exact_rational(layout, fa, fb):
    rng = np.random.default_rng(100 + 10 * layout + 2 * fa + fb)
    M, N, K = 3, 5, 7
    A = random_codes(rng, (K, M) if layout == oracle.TN else (M, K), fa)
    B = random_codes(rng, (N, K) if layout == oracle.NT else (K, N), fb)
    sA, sB = np.float32(0.37), np.float32(1.9)
    C = oracle.gemm_scaled(layout, A, fa, B, fb, float(sA), float(sB), out="f64")
    C32 = oracle.gemm_scaled(layout, A, fa, B, fb, float(sA), float(sB), out="f32")
    alpha = Fraction(float(np.float32(sA * sB)))
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = A[k, i] if layout == oracle.TN else A[i, k]
                b = B[j, k] if layout == oracle.NT else B[k, j]
                acc += exact_value(a, fa) * exact_value(b, fb)
            want = alpha * acc
            assert C[i, j] == float(want)                       # one rounding of the exact value
            ulp = float(np.spacing(np.float32(abs(float(want))))) if want != 0 else 0.0
            assert abs(float(C32[i, j]) - float(want)) <= ulp   # fp32 output within 1 ulp


def test_gemm_layout_consistency_and_identity():
    rng = np.random.default_rng(5)
    M, N, K = 17, 9, 33
    A = random_codes(rng, (M, K), oracle.E4M3)
    B = random_codes(rng, (K, N), oracle.E5M2)
    c_nn = oracle.gemm_scaled(oracle.NN, A, 0, B, 1, 0.5, 2.0, out="f64")
    c_nt = oracle.gemm_scaled(oracle.NT, A, 0, np.ascontiguousarray(B.T), 1, 0.5, 2.0, out="f64")
    c_tn = oracle.gemm_scaled(oracle.TN, np.ascontiguousarray(A.T), 0, B, 1, 0.5, 2.0, out="f64")
    np.testing.assert_array_equal(c_nn, c_nt)
    np.testing.assert_array_equal(c_nn, c_tn)
    eye = np.where(np.eye(K, dtype=bool), np.uint8(0x38), np.uint8(0))       # E4M3 1.0 on the diagonal
    c_id = oracle.gemm_scaled(oracle.NN, A, 0, eye, 0, 0.25, 1.0, out="f64")
    np.testing.assert_array_equal(c_id, 0.25 * oracle.fp8_decode(A, 0))


def test_gemm_bf16_residual():
    rng = np.random.default_rng(6)
    M, N, K = 8, 16, 32
    A = random_codes(rng, (M, K), 0)
    B = random_codes(rng, (K, N), 0)
    R = bf16(rng.standard_normal((M, N)))
    C = oracle.gemm_scaled(oracle.NN, A, 0, B, 0, 0.01, 0.02, out="bf16", residual=R)
    acc = oracle.gemm_scaled(oracle.NN, A, 0, B, 0, 0.01, 0.02, out="f64")
    want = oracle.bf16_round(acc + oracle.bf16_to_f64(R))
    np.testing.assert_array_equal(C, want)
