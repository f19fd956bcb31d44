"""GPU parity: the BF16 baseline block through the C ABI against the oracle's BF16 mode.

LLMQ §4 and §5 measure FP8 training against BF16 training.  The baseline is the same MLP block
with every FP8 cast replaced by bf16 storage: n16 = bf16(RMSNorm(x) g), H = bf16(n16 @ W_gu),
a16 = bf16(SwiGLU(H)), y = bf16(x + a16 @ W_d), and the backward on the same bf16 operands
(tcgen05 kind::f16 GEMMs, alpha = 1).
  * rstd and n16 are bit-exact (the same fp32 formula on an exact input);
  * H, a16, y within 2e-3 max row-relative L2; dH, dN, dX, dW_gu, dW_d, dg within 5e-3;
  * at the 7B-class workload's full size: nothing in the BF16 block needs a tensor-wide scale,
    so every forward output and dH, dN, dX are row-local -- the oracle recomputes sampled token
    rows with the full weights; the weight gradients and dg are checked through their GEMM
    identities on sampled rows/columns, in numpy from the GPU's own operands.
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import dev_bf16, host_f64, row_rel

pytestmark = pytest.mark.gpu


def run_bf16(w, T, d, f, seed=0):
    inp = synth.mlp_inputs(w, seed=seed, T=T, d=d, f=f)
    if "dY" not in inp:
        inp["dY"] = synth.normal_bf16((T, d), 1e-3, seed, synth.TID_DY)
    b = fq.MlpBuffers.allocate(T, d, f, backward=True, keep_intermediates=True, bf16=True)
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    return b, inp


def check_rows(b, ref, rows=None):
    sel = (lambda t: t[rows]) if rows is not None else (lambda t: t)
    np.testing.assert_array_equal(sel(b.rstd.cpu().numpy()), ref["rstd"].astype(np.float32))
    np.testing.assert_array_equal(sel(host_f64(b.n16)), ref["n16"])
    for t, k, tol in ((b.H, "H", 2e-3), (b.a16, "a16", 2e-3), (b.y, "y", 2e-3),
                      (b.dH, "dH", 5e-3), (b.dN, "dN", 5e-3), (b.dX, "dX", 5e-3)):
        assert row_rel(sel(host_f64(t)), ref[k]) < tol, k


@pytest.mark.parametrize("T,d,f", [(192, 256, 384), (272, 528, 400), (1, 16, 16), (640, 1024, 1280), (96, 5136, 1024)])
def test_bf16_block_small_shapes(T, d, f):
    b, inp = run_bf16(synth.BY_NAME["7b-mlp-fwd-bwd"], T, d, f)
    ref = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], eps=b.eps, nthreads=16,
                       bf16=True)
    check_rows(b, ref)
    assert row_rel(host_f64(b.dW_gu), ref["dWgu"]) < 5e-3
    assert row_rel(host_f64(b.dW_d), ref["dWd"]) < 5e-3
    assert row_rel(host_f64(b.dg)[None, :], ref["dg"][None, :]) < 5e-3


def test_bf16_block_deterministic():
    outs = []
    for _ in range(2):
        b, _ = run_bf16(synth.BY_NAME["14b-mlp-fwd-bwd"], 320, 512, 768)
        outs.append([t.clone() for t in (b.y, b.dX, b.dW_gu, b.dW_d, b.dg)])
    for a, c in zip(*outs):
        assert torch.equal(a, c)


def test_bf16_rejects_fp8_only_switches():
    b = fq.MlpBuffers.allocate(64, 64, 64, backward=True, bf16=True)
    b.recompute = True
    with pytest.raises(fq.Fp8qError):
        fq.mlp_block_bwd(b)
    b.recompute, b.grad_e4m3 = False, True
    with pytest.raises(fq.Fp8qError):
        fq.mlp_block_fwd(b)


def test_bf16_full_size_7b():
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = w.T, w.d, w.f
    b, inp = run_bf16(w, T, d, f)
    rows = np.sort(np.random.default_rng(1).choice(T, size=6, replace=False))
    rows[-1] = T - 1
    ref = oracle.block(inp["x"][rows], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"][rows], eps=b.eps,
                       nthreads=16, bf16=True)
    check_rows(b, ref, rows)
    # weight gradients through their GEMM identities on sampled rows / columns
    rng = np.random.default_rng(2)
    dY = synth.f32_from_bf16_bits(inp["dY"]).astype(np.float64)
    i_wd = np.sort(rng.choice(f, size=8, replace=False))
    a16_cols = host_f64(b.a16[:, torch.from_numpy(i_wd).cuda()])
    assert row_rel(host_f64(b.dW_d[torch.from_numpy(i_wd).cuda()]), a16_cols.T @ dY) < 5e-3
    j_wgu = np.sort(rng.choice(2 * f, size=8, replace=False))
    dH_cols = host_f64(b.dH[:, torch.from_numpy(j_wgu).cuda()])
    n16 = host_f64(b.n16)
    assert row_rel(host_f64(b.dW_gu[:, torch.from_numpy(j_wgu).cuda()]).T, (n16.T @ dH_cols).T) < 5e-3
    x = synth.f32_from_bf16_bits(inp["x"]).astype(np.float64)
    nh = x * b.rstd.cpu().numpy().astype(np.float64)[:, None]
    dg_ref = (host_f64(b.dN) * nh).sum(axis=0)
    assert row_rel(host_f64(b.dg)[None, :], dg_ref[None, :]) < 5e-3


@pytest.mark.parametrize("T,d,f,nq,core", [(192, 256, 384, 512, None), (256, 512, 640, 1024, (4, 2, 128))])
def test_bf16_full_block(T, d, f, nq, core):
    """The full block's BF16 baseline (and with its attention core inside) against the oracle's
    BF16 full block: rstd1 and n1_16 bit-exact; qkv, h, y within 2e-3; gradients within 5e-3 (no
    FP8 requantization, so no cascade bars); with the core, att within the core's elementwise bound
    around the oracle's attention of the oracle's qkv."""
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    inp = synth.block_inputs(w, seed=0, T=T, d=d, f=f, n_qkv=nq)
    b = fq.BlockBuffers.allocate(T, d, f, nq, keep_intermediates=True, bf16=True, core=core)
    names = ["x", "g1", "W_qkv", "W_o", "g", "W_gu", "W_d", "dY"] + ([] if core else ["att", "dQKV"])
    for k in names:
        t = {"g": b.mlp.g, "W_gu": b.mlp.W_gu, "W_d": b.mlp.W_d, "dY": b.mlp.dY}.get(k, None)
        (t if t is not None else getattr(b, k)).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.block_fwd(b)
    fq.block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    oc = None if core is None else (core[0], core[1], 128, core[2])
    ref = oracle.full_block(inp["x"], inp["g1"], inp["W_qkv"], inp["W_o"], None if core else inp["att"], inp["g"],
                            inp["W_gu"], inp["W_d"], dY=inp["dY"], dQKV=None if core else inp["dQKV"],
                            nthreads=16, bf16=True, core=oc)
    np.testing.assert_array_equal(b.rstd1.cpu().numpy(), ref["rstd1"].astype(np.float32))
    np.testing.assert_array_equal(host_f64(b.n1_16), ref["n1_16"])
    for t, k in ((b.qkv, "qkv"), (b.h, "h"), (b.mlp.y, "y")):
        assert row_rel(host_f64(t), ref[k]) < 2e-3, k
    if core:
        ra = oracle.attention(synth.bf16_bits(ref["qkv"].astype(np.float32)), core[2], core[0], core[1], 128,
                              nthreads=16, with_abs=True)
        bound = 2.0 ** -8 * (ra["att_abs"] + 2 * np.abs(ra["att"])) * (1 + 2.0 ** -6)
        assert np.all(np.abs(host_f64(b.att) - ref["att"]) <= bound)
    for t, k in ((b.dX, "dX"), (b.d_att, "d_att"), (b.mlp.dX, "dh")):
        assert row_rel(host_f64(t), ref[k]) < 5e-3, k
    if core:
        assert row_rel(host_f64(b.dQKV), ref["dqkv"]) < 5e-3
    for t, k in ((b.dW_qkv, "dWqkv"), (b.dW_o, "dWo"), (b.mlp.dW_gu, "dWgu"), (b.mlp.dW_d, "dWd")):
        assert row_rel(host_f64(t), ref[k]) < 5e-3, k
    for t, k in ((b.dg1, "dg1"), (b.mlp.dg, "dg")):
        assert row_rel(host_f64(t)[None, :], ref[k][None, :]) < 5e-3, k
