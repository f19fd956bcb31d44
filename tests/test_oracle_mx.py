"""Pins of the oracle's block-scaled (MXFP8) quantizer, GEMM and MLP-block mode.

LLMQ §2 ("LLMQ: Efficient Lower-Precision Pretraining for Consumer GPUs") names inner-dimension
block scaling as the scaling Blackwell supports natively; the block format is the OCP Microscaling
one (32 elements along the contraction dimension share an E8M0 power-of-two scale).  The scale
rule is this library's reading (the smallest power of two that clips nothing, the FastML report's
rule per block).

Quantizer: hand-worked blocks (tests/golden/mx_block_hand.txt); the scale is the smallest
unclipped power of two, checked with exact float64 arithmetic; blocks whose absmax is fmax * 2^k
give the per-tensor quantizer's codes (pinned on its own); power-of-two invariance; sign symmetry;
the column direction is the row direction of the transpose; half-step error; NaN blocks.
GEMM: exact rational arithmetic (Python integers) in every layout; unit scales reduce to the
per-tensor scaled GEMM with unit scales; layout consistency.
Block: the MX block is the composition of these pinned primitives (every GEMM reads the slot
quantized along its own contraction dimension) and lands as close to the exact block as the
per-tensor FP8 block does.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests._golden import load

FMAX = {0: 448.0, 1: 57344.0}


def bf16(v):
    return oracle.bf16_round(np.asarray(v, dtype=np.float64))


@pytest.mark.parametrize("case", [1, 2, 3, 4, 5])
def test_mx_hand_worked(case):
    G = load("mx_block_hand.txt")
    fmt = 0 if G[f"case{case}_fmt"] == "e4m3" else 1
    x = np.zeros(32, dtype=np.float32)
    x[: G[f"case{case}_x"].size] = G[f"case{case}_x"]
    codes = np.zeros(32, dtype=np.uint8)
    codes[: G[f"case{case}_codes"].size] = G[f"case{case}_codes"]
    for along_rows, shape in ((False, (1, 32)), (True, (32, 1))):
        q, sf, st = oracle.mx_quantize(x.reshape(shape), fmt, along_rows)
        assert st == 0
        assert sf.size == 1 and sf.ravel()[0] == G[f"case{case}_sf"][0]
        np.testing.assert_array_equal(q.ravel(), codes)
    xb = bf16(x.astype(np.float64))
    if (oracle.bf16_to_f64(xb) == x).all():  # bf16-exact cases: the bf16 input path agrees
        q, sf, _ = oracle.mx_quantize(xb.reshape(1, 32), fmt, False)
        np.testing.assert_array_equal(q.ravel(), codes)


def random_tensor(rng, R, C, kind):
    if kind == "normal":
        v = rng.standard_normal((R, C))
    elif kind == "outliers":
        v = rng.standard_normal((R, C))
        v[:, rng.choice(C, 3, replace=False)] *= 40.0
    else:  # magnitudes over most of the fp32 range
        v = rng.standard_normal((R, C)) * np.exp2(rng.integers(-100, 100, (R, C)))
    return v.astype(np.float32)


def blocks(v, along_rows):
    """The 32-element blocks as rows of a [n_blocks, 32] array (R, C multiples of 32)."""
    R, C = v.shape
    if along_rows:
        return v.reshape(R // 32, 32, C).transpose(0, 2, 1).reshape(-1, 32)
    return v.reshape(R, C // 32, 32).reshape(-1, 32)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("kind", ["normal", "outliers", "wide"])
@pytest.mark.parametrize("along_rows", [False, True])
def test_mx_scale_is_smallest_unclipped_power_of_two(fmt, kind, along_rows):
    rng = np.random.default_rng(7 + fmt + 2 * along_rows)
    v = random_tensor(rng, 64, 96, kind)
    q, sf, st = oracle.mx_quantize(v, fmt, along_rows)
    assert st == 0
    amax = np.abs(blocks(v.astype(np.float64), along_rows)).max(axis=1)
    X = blocks_sf(sf, along_rows).astype(np.int64) - 127
    assert (amax <= np.ldexp(FMAX[fmt], X)).all()                          # nothing clipped
    assert ((X == -127) | (amax > np.ldexp(FMAX[fmt], X - 1))).all()       # the smallest such X
    # the decoded value is within half a step of v * 2^-X (RNE), i.e. within half a step scaled
    dq = oracle.fp8_decode(blocks(q, along_rows), fmt)
    p = blocks(v.astype(np.float64), along_rows) * np.exp2(-X)[:, None]
    frac, sub = (3, 2.0 ** -9) if fmt == 0 else (2, 2.0 ** -16)
    bound = np.maximum(np.abs(p) * 2.0 ** -(frac + 1), sub / 2) * (1 + 1e-12)
    assert (np.abs(dq - p) <= bound).all()


def blocks_sf(sf, along_rows):
    """Scale codes in the block order of blocks(): [R/32, C] and [R, C/32] both ravel that way."""
    return sf.ravel()


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_matches_per_tensor_quantizer_on_power_of_two_blocks(fmt):
    """A block whose absmax is exactly fmax * 2^k has X = k, and the per-tensor quantizer of that
    block alone has scale 2^-k: both give the same codes."""
    rng = np.random.default_rng(3 + fmt)
    for k in (-20, -3, 0, 5, 17):
        v = rng.standard_normal(32).astype(np.float32) * np.float32(2.0 ** k)
        v[int(rng.integers(32))] = np.float32(-FMAX[fmt] * 2.0 ** k)
        q, sf, _ = oracle.mx_quantize(v.reshape(1, 32), fmt, False)
        assert sf[0, 0] == 127 + k
        qt, scal, _ = oracle.quantize_absmax(v, fmt)
        assert scal[1] == np.float32(2.0 ** -k)
        np.testing.assert_array_equal(q.ravel(), qt)


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_power_of_two_invariance_sign_and_transpose(fmt):
    rng = np.random.default_rng(11 + fmt)
    v = random_tensor(rng, 64, 64, "outliers")
    q, sf, _ = oracle.mx_quantize(v, fmt, False)
    for j in (-9, 4):
        q2, sf2, _ = oracle.mx_quantize(v * np.float32(2.0 ** j), fmt, False)
        np.testing.assert_array_equal(q2, q)
        np.testing.assert_array_equal(sf2.astype(int), sf.astype(int) + j)
    qn, sfn, _ = oracle.mx_quantize(-v, fmt, False)
    np.testing.assert_array_equal(sfn, sf)
    np.testing.assert_array_equal(qn, q ^ 0x80)            # no exact zeros in v: every sign flips
    qc, sfc, _ = oracle.mx_quantize(v, fmt, True)
    qt, sft, _ = oracle.mx_quantize(np.ascontiguousarray(v.T), fmt, False)
    np.testing.assert_array_equal(qc, qt.T)
    np.testing.assert_array_equal(sfc, sft.T)


def test_mx_nonfinite_block():
    v = np.ones((1, 64), dtype=np.float32)
    v[0, 40] = np.nan
    q, sf, st = oracle.mx_quantize(v, 0, False)
    assert st == 1
    assert sf[0, 0] == 127 - 8 and sf[0, 1] == 0xFF       # 1 <= 448 * 2^-8, > 448 * 2^-9
    assert (q[0, 32:] == 0x7F).all()


def exact_value(code, sfc, fmt):
    return Fraction(oracle.fp8_decode(np.array([code], np.uint8), fmt)[0]) * Fraction(2) ** (int(sfc) - 127)


@pytest.mark.parametrize("layout", [oracle.NN, oracle.NT, oracle.TN])
def test_mx_gemm_exact_rational(layout):
    rng = np.random.default_rng(20 + layout)
    M, N, K = 5, 6, 96
    fa, fb = 0, 1
    A = oracle.fp8_encode(rng.standard_normal((K, M) if layout == oracle.TN else (M, K)).astype(np.float32) * 50, fa)
    B = oracle.fp8_encode(rng.standard_normal((N, K) if layout == oracle.NT else (K, N)).astype(np.float32) * 900, fb)
    sfA = rng.integers(124, 131, (M, K // 32)).astype(np.uint8)
    sfB = rng.integers(124, 131, (N, K // 32)).astype(np.uint8)
    C = oracle.gemm_mx(layout, A, fa, sfA, B, fb, sfB, out="f64")
    a = lambda i, k: A[k, i] if layout == oracle.TN else A[i, k]
    b = lambda k, j: B[j, k] if layout == oracle.NT else B[k, j]
    for i in range(M):
        for j in range(N):
            ref = sum(exact_value(a(i, k), sfA[i, k // 32], fa) * exact_value(b(k, j), sfB[j, k // 32], fb)
                      for k in range(K))
            assert C[i, j] == float(ref)   # few terms of close exponents: the fp64 sum is exact


def test_mx_gemm_unit_scales_is_the_scaled_gemm():
    rng = np.random.default_rng(5)
    M, N, K = 24, 40, 64
    A = oracle.fp8_encode(rng.standard_normal((M, K)).astype(np.float32) * 30, 0)
    B = oracle.fp8_encode(rng.standard_normal((K, N)).astype(np.float32) * 30, 0)
    one = lambda r: np.full((r, K // 32), 127, np.uint8)
    for out in ("f64", "f32", "bf16"):
        np.testing.assert_array_equal(oracle.gemm_mx(oracle.NN, A, 0, one(M), B, 0, one(N), out=out),
                                      oracle.gemm_scaled(oracle.NN, A, 0, B, 0, 1.0, 1.0, out=out))


def test_mx_gemm_layouts_agree():
    rng = np.random.default_rng(9)
    M, N, K = 16, 48, 128
    A = oracle.fp8_encode(rng.standard_normal((M, K)).astype(np.float32) * 30, 0)
    B = oracle.fp8_encode(rng.standard_normal((K, N)).astype(np.float32) * 30, 1)
    sfA = rng.integers(110, 140, (M, K // 32)).astype(np.uint8)
    sfB = rng.integers(110, 140, (N, K // 32)).astype(np.uint8)
    nn = oracle.gemm_mx(oracle.NN, A, 0, sfA, B, 1, sfB, out="f64")
    nt = oracle.gemm_mx(oracle.NT, A, 0, sfA, np.ascontiguousarray(B.T), 1, sfB, out="f64")
    tn = oracle.gemm_mx(oracle.TN, np.ascontiguousarray(A.T), 0, sfA, B, 1, sfB, out="f64")
    np.testing.assert_array_equal(nn, nt)
    np.testing.assert_array_equal(nn, tn)


def small_inputs(T, d, f):
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    return synth.mlp_inputs(w, seed=3, T=T, d=d, f=f)


def swiglu_f32(H, f):
    """a = fl32(fl32(h / fl32(1 + exp_ref(-h))) * u) of the stored bf16 H, one IEEE rounding per op."""
    h = oracle.bf16_to_f64(H[:, :f]).astype(np.float32)
    u = oracle.bf16_to_f64(H[:, f:]).astype(np.float32)
    return (h / (np.float32(1) + oracle.exp_ref(-h))) * u


def sfk(sf, along_rows):
    """Scale codes as [rows of the GEMM operand, K blocks] (what gemm_mx takes)."""
    return np.ascontiguousarray(sf.T if along_rows else sf)


def test_mx_block_is_composition_of_primitives():
    T, d, f = 64, 96, 64
    inp = small_inputs(T, d, f)
    eps = 1e-6
    out = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], eps=eps, mx=True)
    assert out["status"] == 0
    mx = {}
    for name, src, fmt in (("Wgu", inp["W_gu"], 0), ("Wd", inp["W_d"], 0), ("dY", inp["dY"], 1)):
        for ax in ("r", "c"):
            q, sf, _ = oracle.mx_quantize(src, fmt, ax == "c")
            np.testing.assert_array_equal(out[f"mx_{name}_{ax}"], q)
            np.testing.assert_array_equal(out[f"mx_{name}_{ax}_sf"], sf)
            mx[name + ax] = (q, sf)
    # n: the RMSNorm of the per-tensor path (its rstd pinned there), block-quantized
    _, _, rstd, _ = oracle.rmsnorm_quant(inp["x"], inp["g"], eps)
    np.testing.assert_array_equal(out["rstd"], rstd.astype(np.float64))
    x32 = oracle.bf16_to_f64(inp["x"]).astype(np.float32)
    n = (x32 * rstd[:, None]) * oracle.bf16_to_f64(inp["g"]).astype(np.float32)
    for ax in ("r", "c"):
        q, sf, _ = oracle.mx_quantize(n, 0, ax == "c")
        np.testing.assert_array_equal(out[f"mx_n_{ax}"], q)
        np.testing.assert_array_equal(out[f"mx_n_{ax}_sf"], sf)
        mx["n" + ax] = (q, sf)
    # the gate/up GEMM reads n along d and W_gu along d
    H = oracle.gemm_mx(oracle.NN, mx["nr"][0], 0, sfk(mx["nr"][1], False), mx["Wguc"][0], 0,
                       sfk(mx["Wguc"][1], True), out="bf16")
    np.testing.assert_array_equal(bf16(out["H"]), H)
    a = swiglu_f32(H, f)
    for ax in ("r", "c"):
        q, sf, _ = oracle.mx_quantize(a, 0, ax == "c")
        np.testing.assert_array_equal(out[f"mx_a_{ax}"], q)
        np.testing.assert_array_equal(out[f"mx_a_{ax}_sf"], sf)
        mx["a" + ax] = (q, sf)
    y = oracle.gemm_mx(oracle.NN, mx["ar"][0], 0, sfk(mx["ar"][1], False), mx["Wdc"][0], 0,
                       sfk(mx["Wdc"][1], True), out="bf16", residual=inp["x"])
    np.testing.assert_array_equal(bf16(out["y"]), y)
    # backward: dA along d (dY_r, W_d_r), the wgrads along T (the _c slots), dN along 2f
    dA = oracle.gemm_mx(oracle.NT, mx["dYr"][0], 1, sfk(mx["dYr"][1], False), mx["Wdr"][0], 0,
                        sfk(mx["Wdr"][1], False), out="f64")
    h, u = oracle.bf16_to_f64(H[:, :f]), oracle.bf16_to_f64(H[:, f:])
    sg = 1 / (1 + np.exp(-h))
    np.testing.assert_allclose(out["dH"][:, f:], dA * h * sg, rtol=2 ** -8, atol=1e-30)
    dHb = bf16(out["dH"])
    for ax in ("r", "c"):
        q, sf, _ = oracle.mx_quantize(dHb, 1, ax == "c")
        np.testing.assert_array_equal(out[f"mx_dH_{ax}"], q)
        np.testing.assert_array_equal(out[f"mx_dH_{ax}_sf"], sf)
        mx["dH" + ax] = (q, sf)
    dWd = oracle.gemm_mx(oracle.TN, mx["ac"][0], 0, sfk(mx["ac"][1], True), mx["dYc"][0], 1,
                         sfk(mx["dYc"][1], True), out="f32")
    np.testing.assert_array_equal(out["dWd"], dWd.astype(np.float64))
    dN = oracle.gemm_mx(oracle.NT, mx["dHr"][0], 1, sfk(mx["dHr"][1], False), mx["Wgur"][0], 0,
                        sfk(mx["Wgur"][1], False), out="f32")
    np.testing.assert_array_equal(out["dN"], dN.astype(np.float64))
    dWgu = oracle.gemm_mx(oracle.TN, mx["nc"][0], 0, sfk(mx["nc"][1], True), mx["dHc"][0], 1,
                          sfk(mx["dHc"][1], True), out="f32")
    np.testing.assert_array_equal(out["dWgu"], dWgu.astype(np.float64))
    # the RMSNorm backward is the per-tensor block's (pinned by finite differences): same dN -> same dX
    ref = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], eps=eps)
    x = oracle.bf16_to_f64(inp["x"]); g = oracle.bf16_to_f64(inp["g"]); r = out["rstd"][:, None]
    nh = x * r
    uu = out["dN"] * g
    dX = oracle.bf16_to_f64(inp["dY"]) + r * (uu - nh * (uu * nh).mean(axis=1, keepdims=True))
    np.testing.assert_allclose(out["dX"], dX, rtol=2 ** -8, atol=1e-12)
    assert ref["status"] == 0


def test_mx_block_accuracy_against_exact():
    """Block scaling is at least as close to the exact block as per-tensor scaling."""
    T, d, f = 256, 128, 128
    inp = small_inputs(T, d, f)
    mx = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], mx=True)
    pt = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"])
    f64 = oracle.bf16_to_f64
    ex = oracle.block(f64(inp["x"]), f64(inp["g"]), f64(inp["W_gu"]), f64(inp["W_d"]), dY=f64(inp["dY"]),
                      exact=True)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    for k in ("y", "H", "dX", "dN", "dWgu", "dWd"):
        assert rel(mx[k], ex[k]) < 1.1 * rel(pt[k], ex[k]), k
