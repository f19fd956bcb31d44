"""Pins of the oracle's MLP block (forward + backward).

Block: y = x + W_d-projection(SwiGLU(RMSNorm(x) W_gu)) with per-tensor FP8 quantizers in front of
every GEMM operand (LLMQ §1, §3, §3.1; FastML report "FP8 training without delayed scaling"),
E5M2 gradients (LLMQ §5, Figure 2).
  * exact mode (no quantizers, fp64): the backward equals central finite differences of the
    forward for every input and weight element (T=4, d=8, f=16) -- pins every backward formula;
  * quantized mode: the block equals the composition of the separately pinned primitives,
    bit for bit (quantize_absmax, rmsnorm_quant, gemm_scaled, swiglu_quant) -- pins the wiring
    (operands, transposes, alphas, bf16 storage points);
  * quantized mode stays close to exact mode; results do not depend on the thread count.
"""

import numpy as np
import pytest

import oracle
import synth


def small_inputs(T, d, f, seed=0):
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    return synth.mlp_inputs(w, seed=seed, T=T, d=d, f=f)


def test_exact_backward_matches_finite_differences():
    T, d, f = 4, 8, 16
    rng = np.random.default_rng(0)
    x = rng.standard_normal((T, d))
    g = 1 + 0.1 * rng.standard_normal(d)
    Wgu = 0.3 * rng.standard_normal((d, 2 * f))
    Wd = 0.3 * rng.standard_normal((f, d))
    dY = rng.standard_normal((T, d))
    eps = 1e-6
    out = oracle.block(x, g, Wgu, Wd, dY=dY, eps=eps, exact=True)

    def loss(x_, g_, Wgu_, Wd_):
        return float((oracle.block(x_, g_, Wgu_, Wd_, eps=eps, exact=True)["y"] * dY).sum())

    params = {"dX": x, "dg": g, "dWgu": Wgu, "dWd": Wd}
    for key, P in params.items():
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            h = 1e-6 * max(1.0, abs(P[idx]))
            args = [x.copy(), g.copy(), Wgu.copy(), Wd.copy()]
            which = list(params).index(key)
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - out[key]).max() / np.abs(fd).max()
        assert err < 1e-6, (key, err)


def test_quantized_block_is_composition_of_primitives():
    T, d, f = 32, 64, 48
    inp = small_inputs(T, d, f)
    eps = 1e-6
    out = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], eps=eps)
    assert out["status"] == 0
    sf, sb = out["scal_fwd"], out["scal_bwd"]

    wgu8, s, _ = oracle.quantize_absmax(inp["W_gu"], oracle.E4M3)
    np.testing.assert_array_equal(out["Wgu8"], wgu8); np.testing.assert_array_equal(sf[0], s)
    wd8, s, _ = oracle.quantize_absmax(inp["W_d"], oracle.E4M3)
    np.testing.assert_array_equal(out["Wd8"], wd8); np.testing.assert_array_equal(sf[1], s)
    n8, s, rstd, _ = oracle.rmsnorm_quant(inp["x"], inp["g"], eps)
    np.testing.assert_array_equal(out["n8"], n8); np.testing.assert_array_equal(sf[2], s)
    np.testing.assert_array_equal(out["rstd"], rstd.astype(np.float64))

    H = oracle.gemm_scaled(oracle.NN, n8, 0, wgu8, 0, sf[2, 2], sf[0, 2], out="bf16")
    np.testing.assert_array_equal(oracle.bf16_round(out["H"]), H)
    a8, s, _ = oracle.swiglu_quant(H)
    np.testing.assert_array_equal(out["a8"], a8); np.testing.assert_array_equal(sf[3], s)
    y = oracle.gemm_scaled(oracle.NN, a8, 0, wd8, 0, sf[3, 2], sf[1, 2], out="bf16", residual=inp["x"])
    np.testing.assert_array_equal(oracle.bf16_round(out["y"]), y)

    dY8, s, _ = oracle.quantize_absmax(inp["dY"], oracle.E5M2)
    np.testing.assert_array_equal(out["dY8"], dY8); np.testing.assert_array_equal(sb[0], s)
    dH8, s, _ = oracle.quantize_absmax(oracle.bf16_round(out["dH"]), oracle.E5M2)
    np.testing.assert_array_equal(out["dH8"], dH8); np.testing.assert_array_equal(sb[1], s)
    dWd = oracle.gemm_scaled(oracle.TN, a8, 0, dY8, 1, sf[3, 2], sb[0, 2], out="f32")
    np.testing.assert_array_equal(out["dWd"], dWd.astype(np.float64))
    dN = oracle.gemm_scaled(oracle.NT, dH8, 1, wgu8, 0, sb[1, 2], sf[0, 2], out="f32")
    np.testing.assert_array_equal(out["dN"], dN.astype(np.float64))
    dWgu = oracle.gemm_scaled(oracle.TN, n8, 0, dH8, 1, sf[2, 2], sb[1, 2], out="f32")
    np.testing.assert_array_equal(out["dWgu"], dWgu.astype(np.float64))
    # dA and the SwiGLU backward are checked by the exact-mode finite differences; here: dH is
    # the bf16 rounding of the fp64 SwiGLU gradient of dA = alpha3 * dY8 @ Wd8^T.
    dA = oracle.gemm_scaled(oracle.NT, dY8, 1, wd8, 0, sb[0, 2], sf[1, 2], out="f64")
    h, u = oracle.bf16_to_f64(H[:, :f]), oracle.bf16_to_f64(H[:, f:])
    sg = 1 / (1 + np.exp(-h))
    np.testing.assert_allclose(out["dH"][:, f:], dA * h * sg, rtol=2 ** -8, atol=1e-30)


def test_quantized_close_to_exact_and_thread_invariant():
    T, d, f = 64, 128, 96
    inp = small_inputs(T, d, f, seed=3)
    q1 = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], nthreads=1)
    q4 = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], nthreads=4)
    for k in ("y", "H", "dX", "dWgu", "dWd", "dg", "a8", "dH8"):
        np.testing.assert_array_equal(q1[k], q4[k])
    ex = oracle.block(*(oracle.bf16_to_f64(inp[k]) for k in ("x", "g", "W_gu", "W_d")),
                      dY=oracle.bf16_to_f64(inp["dY"]), exact=True)
    # y is dominated by the residual x; the FP8 branch is checked through H (pre-residual)
    rel = np.linalg.norm(q1["y"] - ex["y"]) / np.linalg.norm(ex["y"])
    assert rel < 0.01, rel
    rel = np.linalg.norm(q1["H"] - ex["H"]) / np.linalg.norm(ex["H"])
    assert rel < 0.1, rel
    for k in ("dWgu", "dWd", "dg"):
        rel = np.linalg.norm(q1[k] - ex[k]) / np.linalg.norm(ex[k])
        assert rel < 0.2, (k, rel)


def test_full_block_exact_backward_matches_finite_differences():
    """Attention-side matmuls of the full block (QKV and O projections around a given attention
    core): with L = sum(y dY) + sum(qkv dQKV), the exact-mode gradients of x, g1, W_qkv, W_o and
    the core output att equal central finite differences."""
    T, d, f, nq = 3, 8, 8, 12
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, d))
    g1 = 1 + 0.1 * rng.standard_normal(d)
    Wqkv = 0.3 * rng.standard_normal((d, nq))
    Wo = 0.3 * rng.standard_normal((d, d))
    att = rng.standard_normal((T, d))
    g2 = 1 + 0.1 * rng.standard_normal(d)
    Wgu = 0.3 * rng.standard_normal((d, 2 * f))
    Wd = 0.3 * rng.standard_normal((f, d))
    dY = rng.standard_normal((T, d))
    dQKV = rng.standard_normal((T, nq))
    args = [x, g1, Wqkv, Wo, att]
    out = oracle.full_block(*args, g2, Wgu, Wd, dY=dY, dQKV=dQKV, exact=True)

    def loss(a):
        o = oracle.full_block(*a, g2, Wgu, Wd, exact=True)
        return float((o["y"] * dY).sum() + (o["qkv"] * dQKV).sum())

    for which, key in enumerate(("dX", "dg1", "dWqkv", "dWo", "d_att")):
        P = args[which]
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            h = 1e-6 * max(1.0, abs(P[idx]))
            a = [v.copy() for v in args]
            a[which][idx] += h
            lp = loss(a)
            a[which][idx] -= 2 * h
            lm = loss(a)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - out[key]).max() / np.abs(fd).max()
        assert err < 1e-6, (key, err)


def test_full_block_quantized_wiring():
    """Quantized full block = composition of the pinned primitives and of the MLP block on h."""
    T, d, f, nq = 40, 64, 48, 96
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    inp = synth.mlp_inputs(w, T=T, d=d, f=f)
    g1 = synth.normal_bf16((d,), 0.1, 0, synth.TID_G1, mean=1.0)
    Wqkv = synth.normal_bf16((d, nq), 0.01, 0, synth.TID_WQKV)
    Wo = synth.normal_bf16((d, d), 0.01, 0, synth.TID_WO)
    att = synth.normal_bf16((T, d), 1.0, 0, synth.TID_ATT)
    dQKV = synth.normal_bf16((T, nq), 1e-3, 0, synth.TID_DQKV)
    o = oracle.full_block(inp["x"], g1, Wqkv, Wo, att, inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"],
                          dQKV=dQKV)
    assert o["status"] == 0
    sa = o["scal_attn"]
    n1, s, r1, _ = oracle.rmsnorm_quant(inp["x"], g1, 1e-6)
    np.testing.assert_array_equal(o["n1_8"], n1); np.testing.assert_array_equal(sa[2], s)
    wq, s, _ = oracle.quantize_absmax(Wqkv, 0)
    np.testing.assert_array_equal(o["Wqkv8"], wq); np.testing.assert_array_equal(sa[0], s)
    wo, s, _ = oracle.quantize_absmax(Wo, 0)
    np.testing.assert_array_equal(o["Wo8"], wo); np.testing.assert_array_equal(sa[1], s)
    a8, s, _ = oracle.quantize_absmax(att, 0)
    np.testing.assert_array_equal(o["att8"], a8); np.testing.assert_array_equal(sa[3], s)
    qkv = oracle.gemm_scaled(oracle.NN, n1, 0, wq, 0, sa[2, 2], sa[0, 2], out="bf16")
    np.testing.assert_array_equal(oracle.bf16_round(o["qkv"]), qkv)
    h = oracle.gemm_scaled(oracle.NN, a8, 0, wo, 0, sa[3, 2], sa[1, 2], out="bf16", residual=inp["x"])
    np.testing.assert_array_equal(oracle.bf16_round(o["h"]), h)
    mlp = oracle.block(h, inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"])
    for k in ("y", "H", "a8", "dWgu", "dWd", "dg"):
        np.testing.assert_array_equal(o[k], mlp[k])
    np.testing.assert_array_equal(o["dh"], mlp["dX"])
    dh8, s, _ = oracle.quantize_absmax(oracle.bf16_round(o["dh"]), 1)
    np.testing.assert_array_equal(o["dh8"], dh8); np.testing.assert_array_equal(sa[4], s)
    d_att = oracle.gemm_scaled(oracle.NT, dh8, 1, wo, 0, sa[4, 2], sa[1, 2], out="bf16")
    np.testing.assert_array_equal(oracle.bf16_round(o["d_att"]), d_att)
    dWo = oracle.gemm_scaled(oracle.TN, a8, 0, dh8, 1, sa[3, 2], sa[4, 2], out="f32")
    np.testing.assert_array_equal(o["dWo"], dWo.astype(np.float64))
    dq8, s, _ = oracle.quantize_absmax(dQKV, 1)
    np.testing.assert_array_equal(o["dqkv8"], dq8); np.testing.assert_array_equal(sa[5], s)
    dWqkv = oracle.gemm_scaled(oracle.TN, n1, 0, dq8, 1, sa[2, 2], sa[5, 2], out="f32")
    np.testing.assert_array_equal(o["dWqkv"], dWqkv.astype(np.float64))


def test_e4m3_gradient_recipe_wiring():
    """With grad_fmt = E4M3 the gradient quantizers and the dgrad/wgrad GEMM operands are E4M3
    (LLMQ §5 Figure 2's E4M3 forward and backward)."""
    T, d, f = 32, 64, 48
    inp = small_inputs(T, d, f)
    out = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], grad_fmt=oracle.E4M3)
    sf, sb = out["scal_fwd"], out["scal_bwd"]
    dY8, s, _ = oracle.quantize_absmax(inp["dY"], oracle.E4M3)
    np.testing.assert_array_equal(out["dY8"], dY8); np.testing.assert_array_equal(sb[0], s)
    assert s[1] == np.float32(448.0) / s[0]
    dH8, s, _ = oracle.quantize_absmax(oracle.bf16_round(out["dH"]), oracle.E4M3)
    np.testing.assert_array_equal(out["dH8"], dH8); np.testing.assert_array_equal(sb[1], s)
    dWd = oracle.gemm_scaled(oracle.TN, out["a8"], 0, dY8, 0, sf[3, 2], sb[0, 2], out="f32")
    np.testing.assert_array_equal(out["dWd"], dWd.astype(np.float64))
    dN = oracle.gemm_scaled(oracle.NT, dH8, 0, out["Wgu8"], 0, sb[1, 2], sf[0, 2], out="f32")
    np.testing.assert_array_equal(out["dN"], dN.astype(np.float64))
    e5 = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"])
    for k in ("dX", "dWgu", "dWd"):   # both recipes approximate the same gradients
        rel = np.linalg.norm(out[k] - e5[k]) / np.linalg.norm(e5[k])
        assert 0 < rel < 0.2, (k, rel)


def _half_bf16_ulp(v):
    """Half a bf16 ulp of |v| (normal range): 2^(floor(log2|v|) - 8)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (e - 8).astype(int))


def _is_bf16(v):
    f32 = np.asarray(v, dtype=np.float32)
    return np.array_equal(f32.astype(np.float64), np.asarray(v)) and not np.any(f32.view(np.uint32) & 0xFFFF)


def test_bf16_baseline_wiring_and_storage_points():
    """BF16 baseline (LLMQ §4/§5 compare FP8 with BF16 training): each stored tensor is bf16 and
    within half a bf16 ulp (plus fp32 arithmetic slack) of the fp64 closed form of its inputs;
    the fp32 GEMM outputs equal numpy's fp64 product of the stored bf16 operands rounded once to
    fp32 (bf16 x bf16 products are exact in fp64 and these sums stay exact)."""
    T, d, f = 32, 64, 48
    inp = small_inputs(T, d, f)
    out = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], bf16=True)
    x, g, Wgu, Wd, dY = (oracle.bf16_to_f64(inp[k]) for k in ("x", "g", "W_gu", "W_d", "dY"))
    n16, a16, H, dH = out["n16"], out["a16"], out["H"], out["dH"]
    for k in ("n16", "a16", "H", "y", "dH", "dX"):
        assert _is_bf16(out[k]), k
    # RMSNorm closed form
    n_ref = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6) * g
    assert np.all(np.abs(n16 - n_ref) <= _half_bf16_ulp(n_ref) * (1 + 2.0 ** -6)), "n16"
    # H = bf16(n16 @ W_gu); a = bf16(silu(gate) * up); y = bf16(x + a16 @ W_d)
    H_ref = n16 @ Wgu
    assert np.all(np.abs(H - H_ref) <= _half_bf16_ulp(H_ref) * (1 + 2.0 ** -20)), "H"
    hg, hu = H[:, :f], H[:, f:]
    a_ref = hg / (1 + np.exp(-hg)) * hu
    assert np.all(np.abs(a16 - a_ref) <= _half_bf16_ulp(a_ref) * (1 + 2.0 ** -6)), "a16"
    y_ref = x + a16 @ Wd
    assert np.all(np.abs(out["y"] - y_ref) <= _half_bf16_ulp(y_ref) * (1 + 2.0 ** -20)), "y"
    # backward: unscaled products of the stored bf16 operands, rounded once to fp32
    f32 = lambda v: v.astype(np.float32).astype(np.float64)  # noqa: E731
    np.testing.assert_array_equal(out["dWd"], f32(a16.T @ dY))
    np.testing.assert_array_equal(out["dN"], f32(dH @ Wgu.T))
    np.testing.assert_array_equal(out["dWgu"], f32(n16.T @ dH))
    dA = dY @ Wd.T
    s = 1 / (1 + np.exp(-hg))
    dg_ref, du_ref = dA * hu * s * (1 + hg * (1 - s)), dA * hg * s
    assert np.all(np.abs(dH[:, :f] - dg_ref) <= _half_bf16_ulp(dg_ref) * (1 + 2.0 ** -20) + 1e-300)
    assert np.all(np.abs(dH[:, f:] - du_ref) <= _half_bf16_ulp(du_ref) * (1 + 2.0 ** -20) + 1e-300)


def test_bf16_baseline_accuracy_against_exact():
    """The BF16 block tracks the exact block (itself pinned by finite differences) to the bf16
    storage error -- a few 2^-9 relative -- and far closer than the FP8 block does."""
    T, d, f = 32, 64, 48
    inp = small_inputs(T, d, f)
    args = [inp[k] for k in ("x", "g", "W_gu", "W_d")]
    b = oracle.block(*args, dY=inp["dY"], bf16=True)
    q = oracle.block(*args, dY=inp["dY"])
    e = oracle.block(*(oracle.bf16_to_f64(a) for a in args), dY=oracle.bf16_to_f64(inp["dY"]), exact=True)
    for k in ("H", "y", "dX", "dWgu", "dWd", "dg", "dN"):
        rb = np.linalg.norm(b[k] - e[k]) / np.linalg.norm(e[k])
        rq = np.linalg.norm(q[k] - e[k]) / np.linalg.norm(e[k])
        assert rb < 8 * 2.0 ** -9, (k, rb)
        assert rb <= rq, (k, rb, rq)
        if k not in ("y", "dX"):  # y, dX are dominated by the exact residual terms x, dY
            assert rb < rq / 5, (k, rb, rq)


def test_full_block_bf16_baseline_accuracy():
    """The full block's BF16 baseline (every operand stored as bf16): close to the exact block
    (pinned by finite differences), several times closer than the FP8 block, and its stored
    n1 is the bf16 closed form of the attention-side RMSNorm."""
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    T, d, f, nq = 64, 256, 192, 512
    inp = synth.block_inputs(w, seed=0, T=T, d=d, f=f, n_qkv=nq)
    args = [inp[k] for k in ("x", "g1", "W_qkv", "W_o", "att", "g", "W_gu", "W_d")]
    b = oracle.full_block(*args, dY=inp["dY"], dQKV=inp["dQKV"], bf16=True)
    q = oracle.full_block(*args, dY=inp["dY"], dQKV=inp["dQKV"])
    e = oracle.full_block(*(oracle.bf16_to_f64(a) for a in args), dY=oracle.bf16_to_f64(inp["dY"]),
                          dQKV=oracle.bf16_to_f64(inp["dQKV"]), exact=True)
    for k in ("qkv", "h", "y", "dX", "dWqkv", "dWo", "dWgu", "dWd"):
        rb = np.linalg.norm(b[k] - e[k]) / np.linalg.norm(e[k])
        rq = np.linalg.norm(q[k] - e[k]) / np.linalg.norm(e[k])
        assert rb < 8 * 2.0 ** -9, (k, rb)
        assert rb < rq / 2, (k, rb, rq)
    x, g1 = oracle.bf16_to_f64(inp["x"]), oracle.bf16_to_f64(inp["g1"])
    n1 = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6) * g1
    assert np.all(np.abs(b["n1_16"] - n1) <= _half_bf16_ulp(n1) * (1 + 2.0 ** -6))
