"""Pins of the oracle's exp_ref, SwiGLU and RMSNorm (the fused non-matmul ops of LLMQ §3/§3.1).

exp_ref: within 2 ulp of the correctly rounded e^x (fp64 reference) on a dense grid of [-104, 89]
(every fp32 whose low 8 bits are zero) plus random points; exact special cases.
SwiGLU: closed-form values (tests/golden/swiglu_closed_form.txt) within 2 ulp; silu(0) = 0;
silu(h) = h once e^-h is below half an ulp.
RMSNorm: hand-worked rows (golden), the pairwise order of the sum of squares (golden), the
fp64 closed form on a 4x4 block within 2 ulp, scale invariance under powers of two (eps = 0).
RMSNorm backward (with the residual gradient): in exact mode equal to central finite differences of
L = sum dN (x rstd(x) g) + sum dY x for every element of x and g; the rounded mode is the exact
result rounded once (dX to bf16, dg to fp32); dN = 0 passes dY through unchanged; with eps = 0
the input gradient of the normalization is orthogonal to x (scale invariance).
"""

import numpy as np
import pytest

import oracle
from tests._golden import load


def ulp_err(got32, ref64):
    ref32 = ref64.astype(np.float32)
    sp = np.spacing(np.abs(ref32)).astype(np.float64)
    return np.abs(got32.astype(np.float64) - ref64) / sp


def test_exp_ref_dense_grid():
    lo = np.float32(-104.0).view(np.uint32)
    hi = np.float32(89.0).view(np.uint32)
    # negatives: bit patterns 0x80000000..lo, positives 0..hi; keep those with low 8 bits zero
    neg = np.arange(0x80000000, lo + 1, 256, dtype=np.uint64).astype(np.uint32).view(np.float32)
    pos = np.arange(0, hi + 1, 256, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rnd = np.random.default_rng(7).uniform(-104, 89, 1 << 20).astype(np.float32)
    x = np.concatenate([neg, pos, rnd])
    y = oracle.exp_ref(x)
    ref = np.exp(x.astype(np.float64))
    ok = ref < np.finfo(np.float32).max
    err = ulp_err(y[ok], ref[ok])
    assert err.max() <= 2.0, f"max ulp error {err.max()} at x={x[ok][np.argmax(err)]}"
    assert np.isinf(y[~ok]).all()


def test_exp_ref_special_values():
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 89.0, -105.0, 1.0], dtype=np.float32)
    y = oracle.exp_ref(x)
    assert y[0] == 1.0 and y[1] == 1.0
    assert y[2] == np.inf and y[3] == 0.0 and np.isnan(y[4])
    assert y[5] == np.inf and y[6] == 0.0
    assert abs(float(y[7]) - np.e) <= float(np.spacing(np.float32(np.e)))




def test_swiglu_closed_form():
    G = load("swiglu_closed_form.txt")
    gate, up, a_ref = G["gate"], G["up"], G["a"]
    # all inputs are exactly representable in bf16
    H = np.concatenate([oracle.bf16_round(gate), oracle.bf16_round(up)])[None, :]
    assert (oracle.bf16_to_f64(H[0, : gate.size]) == gate).all()
    # Evaluate one (gate, up) pair at a time: the quantizer's amax is then exactly |a| in fp32.
    for j in range(gate.size):
        Hj = np.array([[H[0, j], H[0, gate.size + j]]], dtype=np.uint16)
        _, scal, _ = oracle.swiglu_quant(Hj)
        amax = float(scal[0])
        ref = abs(a_ref[j])
        if ref == 0.0 or ref < 1e-30:
            assert amax <= 1e-30
            continue
        err = abs(amax - ref) / float(np.spacing(np.float32(ref)))
        assert err <= 2.0, (gate[j], up[j], amax, ref, err)


def test_swiglu_limits_and_sign():
    # silu(0) = 0; silu(h) = h for h >= 17 (e^-h below half an ulp of 1); the product keeps the sign
    gate = np.array([0.0, 17.0, 30.0, -2.0], dtype=np.float64)
    up = np.array([5.0, 1.0, -2.0, -1.0], dtype=np.float64)
    for gv, uv, want in [(0.0, 5.0, 0.0), (17.0, 1.0, 17.0), (30.0, -2.0, 60.0)]:
        Hj = np.array([[oracle.bf16_round(np.array([gv]))[0], oracle.bf16_round(np.array([uv]))[0]]])
        q, scal, _ = oracle.swiglu_quant(Hj)
        assert float(scal[0]) == want
    # sign: silu(-2) * (-1) > 0 -> positive max code 0x7E
    Hj = np.array([[oracle.bf16_round(np.array([-2.0]))[0], oracle.bf16_round(np.array([-1.0]))[0]]])
    q, scal, _ = oracle.swiglu_quant(Hj)
    assert q[0, 0] == 0x7E


def bf16(v):
    return oracle.bf16_round(np.asarray(v, dtype=np.float64))


@pytest.mark.parametrize("name", ["rmsnorm_constant_row.txt"])
def test_rmsnorm_hand_worked(name):
    G = load(name)
    T, d = int(G["T"]), int(G["d"])
    x = bf16(G["x"]).reshape(T, d)
    g = bf16(G["g"])
    q, scal, rstd, st = oracle.rmsnorm_quant(x, g, G["eps"])
    assert st == 0
    assert rstd[0] == np.float32(G["rstd"])
    assert scal[0] == G["amax"] and scal[1] == G["scale"]
    np.testing.assert_array_equal(q.ravel(), G["codes"])


def test_rmsnorm_pairwise_order():
    G = load("rmsnorm_pairwise_order.txt")
    x = bf16(G["x"])
    assert (oracle.bf16_to_f64(x) == G["x"]).all()
    sq = (G["x"] ** 2).astype(np.float32)
    assert oracle.pairwise_sum_f32(sq) == np.float32(G["pairwise_sum_sq"])
    _, _, rstd, _ = oracle.rmsnorm_quant(x[None, :], bf16(G["g"]), G["eps"])
    assert rstd[0] == np.float32(G["rstd"])
    assert rstd[0] != np.float32(G["rstd_sequential"])


def test_pairwise_sum_exact_on_integers_and_split_rule():
    # small integers: every partial sum exact -> equals the exact total
    v = np.arange(1, 1001, dtype=np.float32)
    assert oracle.pairwise_sum_f32(v) == np.float32(500500)
    # the split point: [2^24, 1, 1] splits as [2^24, 1] + [1] -> (2^24 + 1 -> 2^24) + 1 -> 2^24
    # while a split [2^24] + [1, 1] would give 2^24 + 2.
    v = np.array([2.0 ** 24, 1.0, 1.0], dtype=np.float32)
    assert oracle.pairwise_sum_f32(v) == np.float32(2.0 ** 24)


def test_rmsnorm_closed_form_4x4():
    rng = np.random.default_rng(3)
    x = bf16(rng.standard_normal((4, 4)))
    g = bf16(1 + 0.1 * rng.standard_normal(4))
    eps = 1e-6
    _, _, rstd, _ = oracle.rmsnorm_quant(x, g, eps)
    xf = oracle.bf16_to_f64(x)
    ref = 1.0 / np.sqrt((xf ** 2).mean(axis=1) + np.float64(np.float32(eps)))
    assert (ulp_err(rstd, ref) <= 2.0).all()


def test_rmsnorm_power_of_two_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64))
    g = bf16(1 + 0.1 * rng.standard_normal(64))
    q1, s1, r1, _ = oracle.rmsnorm_quant(bf16(x), g, 0.0)
    q2, s2, r2, _ = oracle.rmsnorm_quant(bf16(x * 8.0), g, 0.0)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_array_equal(r1, r2 * 8)


def _rms_loss(x, g, dN, dY, eps):
    rs = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    return float((dN * (x * rs[:, None] * g)).sum() + (dY * x).sum())


def test_rmsnorm_bwd_exact_matches_finite_differences():
    T, d, eps, h = 3, 8, 1e-3, 1e-6
    rng = np.random.default_rng(11)
    x, dN, dY = rng.standard_normal((T, d)), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    g = 1 + 0.2 * rng.standard_normal(d)
    rstd = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    dX, dg = oracle.rmsnorm_bwd(dN, x, g, rstd, dY, exact=True)
    fx = np.zeros_like(x)
    for t in range(T):
        for j in range(d):
            xp, xm = x.copy(), x.copy()
            xp[t, j] += h
            xm[t, j] -= h
            fx[t, j] = (_rms_loss(xp, g, dN, dY, eps) - _rms_loss(xm, g, dN, dY, eps)) / (2 * h)
    fg = np.zeros_like(g)
    for j in range(d):
        gp, gm = g.copy(), g.copy()
        gp[j] += h
        gm[j] -= h
        fg[j] = (_rms_loss(x, gp, dN, dY, eps) - _rms_loss(x, gm, dN, dY, eps)) / (2 * h)
    np.testing.assert_allclose(dX, fx, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dg, fg, rtol=1e-6, atol=1e-7)


def test_rmsnorm_bwd_rounds_once_and_passes_the_residual():
    T, d = 5, 48
    rng = np.random.default_rng(12)
    x, dN = rng.standard_normal((T, d)), rng.standard_normal((T, d)).astype(np.float32).astype(np.float64)
    dY = oracle.bf16_to_f64(oracle.bf16_round(rng.standard_normal((T, d))))
    g = oracle.bf16_to_f64(oracle.bf16_round(1 + 0.1 * rng.standard_normal(d)))
    rstd = (1.0 / np.sqrt((x * x).mean(axis=1) + 1e-6)).astype(np.float32).astype(np.float64)
    ex, exg = oracle.rmsnorm_bwd(dN, x, g, rstd, dY, exact=True)
    dX, dg = oracle.rmsnorm_bwd(dN, x, g, rstd, dY)
    assert np.array_equal(dX, oracle.bf16_to_f64(oracle.bf16_round(ex)))
    assert np.array_equal(dg, exg.astype(np.float32).astype(np.float64))
    z, zg = oracle.rmsnorm_bwd(np.zeros((T, d)), x, g, rstd, dY)
    assert np.array_equal(z, dY) and not zg.any()


def test_rmsnorm_bwd_orthogonal_to_x_without_eps():
    T, d = 4, 64
    rng = np.random.default_rng(13)
    x, dN = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    g = 1 + 0.1 * rng.standard_normal(d)
    rstd = 1.0 / np.sqrt((x * x).mean(axis=1))
    dX, _ = oracle.rmsnorm_bwd(dN, x, g, rstd, np.zeros((T, d)), exact=True)
    dot = (dX * x).sum(axis=1)
    assert np.all(np.abs(dot) <= 1e-12 * np.abs(dX).sum(axis=1) * np.abs(x).max(axis=1))
