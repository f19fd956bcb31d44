"""Pins of the oracle's attention core (causal grouped-query softmax attention between the QKV and
O projections of the transformer block; LLMQ §2/§3 name the block, the pages fix no attention
arithmetic, so the core is the plain definition).
  * exact mode: the backward equals central finite differences of the forward for every qkv
    element (two sequences, grouped K/V heads) -- pins dq, dk, dv, the causal mask and the
    group sums;
  * multi-head case (one K/V head per query head) equals scipy's softmax with a causal mask;
  * grouped heads equal multi-head attention with each K/V head repeated for its group;
  * q = 0: every key equally likely, att_i = mean of v_0..v_i, lse_i = log(i + 1);
  * causality and independence of the sequences;
  * bf16 mode rounds att and dqkv once from the exact values; the full block with the core wires
    att and dQKV through it.
"""

import numpy as np
import pytest
import scipy.special

import oracle
import synth


def rand_qkv(T, Hq, Hkv, dh, seed=0, scale=1.0):
    return scale * np.random.default_rng(seed).standard_normal((T, (Hq + 2 * Hkv) * dh))


def test_exact_backward_matches_finite_differences():
    S, Hq, Hkv, dh, B = 5, 4, 2, 3, 2
    qkv = rand_qkv(B * S, Hq, Hkv, dh)
    dO = np.random.default_rng(1).standard_normal((B * S, Hq * dh))
    g = oracle.attention(qkv, S, Hq, Hkv, dh, d_att=dO, exact=True)["dqkv"]
    loss = lambda q: float((oracle.attention(q, S, Hq, Hkv, dh, exact=True)["att"] * dO).sum())  # noqa: E731
    h = 1e-6
    num = np.zeros_like(qkv)
    for idx in np.ndindex(*qkv.shape):
        e = np.zeros_like(qkv)
        e[idx] = h
        num[idx] = (loss(qkv + e) - loss(qkv - e)) / (2 * h)
    np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_multi_head_equals_scipy_softmax():
    S, H, dh = 7, 3, 5
    qkv = rand_qkv(S, H, H, dh, seed=2)
    out = oracle.attention(qkv, S, H, H, dh, exact=True)
    q, k, v = (qkv[:, i * H * dh:(i + 1) * H * dh].reshape(S, H, dh) for i in range(3))
    mask = np.triu(np.ones((S, S), bool), 1)
    for h in range(H):
        s = q[:, h] @ k[:, h].T / np.sqrt(dh)
        s[mask] = -np.inf
        ref = scipy.special.softmax(s, axis=1) @ v[:, h]
        np.testing.assert_allclose(out["att"][:, h * dh:(h + 1) * dh], ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["lse"][h], scipy.special.logsumexp(s, axis=1), rtol=1e-12)


def test_grouped_heads_equal_repeated_kv_heads():
    S, Hq, Hkv, dh = 6, 6, 2, 4
    qkv = rand_qkv(2 * S, Hq, Hkv, dh, seed=3)
    dO = np.random.default_rng(4).standard_normal((2 * S, Hq * dh))
    rep = Hq // Hkv
    q = qkv[:, :Hq * dh]
    k = qkv[:, Hq * dh:(Hq + Hkv) * dh].reshape(-1, Hkv, dh)
    v = qkv[:, (Hq + Hkv) * dh:].reshape(-1, Hkv, dh)
    mha = np.concatenate([q, np.repeat(k, rep, axis=1).reshape(2 * S, -1), np.repeat(v, rep, axis=1).reshape(2 * S, -1)], 1)
    a = oracle.attention(qkv, S, Hq, Hkv, dh, d_att=dO, exact=True)
    b = oracle.attention(mha, S, Hq, Hq, dh, d_att=dO, exact=True)
    np.testing.assert_allclose(a["att"], b["att"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a["dqkv"][:, :Hq * dh], b["dqkv"][:, :Hq * dh], rtol=1e-12, atol=1e-14)
    # the grouped dk, dv are the sums of the repeated heads' gradients
    for part in range(2):
        ga = a["dqkv"][:, (Hq + part * Hkv) * dh:(Hq + (part + 1) * Hkv) * dh].reshape(-1, Hkv, dh)
        gb = b["dqkv"][:, (Hq + part * Hq) * dh:(Hq + (part + 1) * Hq) * dh].reshape(-1, Hkv, rep, dh).sum(2)
        np.testing.assert_allclose(ga, gb, rtol=1e-12, atol=1e-14)


def test_zero_queries_average_the_prefix():
    S, Hq, Hkv, dh = 9, 2, 1, 4
    qkv = rand_qkv(S, Hq, Hkv, dh, seed=5)
    qkv[:, :Hq * dh] = 0.0
    out = oracle.attention(qkv, S, Hq, Hkv, dh, exact=True, with_abs=True)
    v = qkv[:, (Hq + Hkv) * dh:]
    prefix_mean = np.cumsum(v, 0) / np.arange(1, S + 1)[:, None]
    for h in range(Hq):
        np.testing.assert_allclose(out["att"][:, h * dh:(h + 1) * dh], prefix_mean, rtol=1e-13)
        np.testing.assert_allclose(out["att_abs"][:, h * dh:(h + 1) * dh],
                                   np.cumsum(np.abs(v), 0) / np.arange(1, S + 1)[:, None], rtol=1e-13)
        np.testing.assert_allclose(out["lse"][h], np.log(np.arange(1, S + 1)), rtol=1e-13)


def test_att_abs_bounds_att():
    S, Hq, Hkv, dh = 12, 4, 2, 6
    qkv = rand_qkv(3 * S, Hq, Hkv, dh, seed=7, scale=2.0)
    out = oracle.attention(qkv, S, Hq, Hkv, dh, exact=True, with_abs=True)
    assert np.all(out["att_abs"] >= np.abs(out["att"]) * (1 - 1e-14))
    dO = np.random.default_rng(8).standard_normal((3 * S, Hq * dh))
    g = oracle.attention(qkv, S, Hq, Hkv, dh, d_att=dO, exact=True, with_abs=True)
    assert np.all(g["dqkv_abs"] >= np.abs(g["dqkv"]) * (1 - 1e-12))
    np.testing.assert_array_equal(g["dqkv"], oracle.attention(qkv, S, Hq, Hkv, dh, d_att=dO, exact=True)["dqkv"])
    # a constant-sign V makes the two equal
    qkv[:, (Hq + Hkv) * dh:] = np.abs(qkv[:, (Hq + Hkv) * dh:])
    out = oracle.attention(qkv, S, Hq, Hkv, dh, exact=True, with_abs=True)
    np.testing.assert_allclose(out["att_abs"], out["att"], rtol=1e-13)


def test_causal_and_sequences_independent():
    S, Hq, Hkv, dh = 8, 2, 2, 4
    qkv = rand_qkv(2 * S, Hq, Hkv, dh, seed=6)
    base = oracle.attention(qkv, S, Hq, Hkv, dh, exact=True)["att"]
    pert = qkv.copy()
    pert[5] += 1.0                     # token 5 of sequence 0
    pert[S + 3:] *= 2.0                # tokens 3.. of sequence 1
    out = oracle.attention(pert, S, Hq, Hkv, dh, exact=True)["att"]
    np.testing.assert_array_equal(out[:5], base[:5])
    np.testing.assert_array_equal(out[S:S + 3], base[S:S + 3])
    assert not np.allclose(out[5], base[5])


def test_bf16_mode_rounds_storage_points_once():
    S, Hq, Hkv, dh = 16, 4, 2, 8
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    qkv = synth.normal_bf16((2 * S, (Hq + 2 * Hkv) * dh), 0.7, 0, 40)
    dO = synth.normal_bf16((2 * S, Hq * dh), 1e-3, 0, 41)
    r = oracle.attention(qkv, S, Hq, Hkv, dh, d_att=dO)
    e = oracle.attention(oracle.bf16_to_f64(qkv), S, Hq, Hkv, dh, d_att=oracle.bf16_to_f64(dO), exact=True)
    np.testing.assert_array_equal(r["att"], oracle.bf16_to_f64(oracle.bf16_round(e["att"])))
    np.testing.assert_array_equal(r["dqkv"], oracle.bf16_to_f64(oracle.bf16_round(e["dqkv"])))
    np.testing.assert_array_equal(r["lse"], e["lse"])
    assert w.qkv == 7168


def test_full_block_with_core_wires_att_and_dqkv():
    T, S, Hq, Hkv, dh, f = 64, 32, 4, 2, 16, 48
    d, nq = Hq * dh, (Hq + 2 * Hkv) * dh
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    inp = synth.block_inputs(w, seed=0, T=T, d=d, f=f, n_qkv=nq)
    args = [inp[k] for k in ("x", "g1", "W_qkv", "W_o")]
    mlp = [inp[k] for k in ("g", "W_gu", "W_d")]
    c = oracle.full_block(*args, None, *mlp, dY=inp["dY"], core=(Hq, Hkv, dh, S))
    a = oracle.attention(synth.bf16_bits(c["qkv"].astype(np.float32)), S, Hq, Hkv, dh,
                         d_att=synth.bf16_bits(c["d_att"].astype(np.float32)))
    np.testing.assert_array_equal(c["att"], a["att"])
    np.testing.assert_array_equal(c["dqkv"], a["dqkv"])
    g = oracle.full_block(*args, synth.bf16_bits(c["att"].astype(np.float32)), *mlp, dY=inp["dY"],
                          dQKV=synth.bf16_bits(c["dqkv"].astype(np.float32)))
    for k in ("y", "h", "dX", "dWqkv", "dWo", "dg1", "dWgu", "dWd"):
        np.testing.assert_array_equal(c[k], g[k], err_msg=k)
