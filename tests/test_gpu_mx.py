"""GPU parity of the block-scaled MXFP8 path against the oracle.

mx_quantize: E8M0 scales and element codes bit-exact, both block directions, bf16 and fp32 input,
E4M3 and E5M2, value ranges from tiny to huge, all-zero and non-finite blocks.  fp8_gemm_mx
(tcgen05.mma kind::mxf8f6f4.block_scale): every layout and format mix, ragged M and N tiles, bf16
output with residual, scales that vary by row, by column and by K block; bar: max row-relative
L2 error 2e-3 against the oracle's fp64 GEMM.  The MXFP8 MLP block: every quantized operand bit-exact
where its input is a given tensor (weights, n, dY), in-block requantizations (a, dH) within the
requantization rule, outputs 2e-3 and gradients 5e-3 row-relative, bit-identical reruns.
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import (code_step_diff, dev_bf16, dev_u8, host_f64, mx_sf_from_chunked, mx_sf_to_chunked, row_rel)

pytestmark = pytest.mark.gpu


def host_u8(t):
    return t.cpu().numpy()


def tensor(rng, R, C, kind):
    v = rng.standard_normal((R, C)).astype(np.float32)
    if kind == "outliers":
        v[:, rng.choice(C, 4, replace=False)] *= 50.0
    elif kind == "wide":
        v *= np.exp2(rng.integers(-60, 60, (R, C))).astype(np.float32)
    elif kind == "zeros":
        v[:64, :] = 0.0
        v[:, :32] = 0.0
    return v


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R,C,kind", [(128, 128, "normal"), (256, 384, "outliers"), (384, 256, "wide"),
                                      (256, 256, "zeros")])
def test_mx_quantize_bit_exact(fmt, dtype, R, C, kind):
    rng = np.random.default_rng(R + C + fmt)
    v = tensor(rng, R, C, kind)
    host = synth.bf16_bits(v) if dtype == "bf16" else v
    x = dev_bf16(host) if dtype == "bf16" else torch.from_numpy(v).cuda()
    fq.get_status(clear=True)
    (qr, sfr), (qc, sfc) = fq.mx_quantize(x, fmt)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    oq, osf, st = oracle.mx_quantize(host, fmt, False)
    assert st == 0
    np.testing.assert_array_equal(host_u8(qr), oq)
    np.testing.assert_array_equal(mx_sf_from_chunked(host_u8(sfr), R, C), osf)
    oq, osf, _ = oracle.mx_quantize(host, fmt, True)
    np.testing.assert_array_equal(host_u8(qc), oq)
    np.testing.assert_array_equal(mx_sf_from_chunked(host_u8(sfc), C, R), osf.T)


def test_mx_quantize_nonfinite_block():
    v = np.ones((128, 128), dtype=np.float32)
    v[5, 70] = np.inf
    v[40, 3] = np.nan
    fq.get_status(clear=True)
    (qr, sfr), (qc, sfc) = fq.mx_quantize(torch.from_numpy(v).cuda(), 0)
    torch.cuda.synchronize()
    assert fq.get_status() & fq.STATUS_NONFINITE
    for along, (q, sf) in ((False, (qr, sfr)), (True, (qc, sfc))):
        oq, osf, st = oracle.mx_quantize(v, 0, along)
        assert st == 1
        np.testing.assert_array_equal(host_u8(q), oq)
        rows, K = (128, 128)
        got = mx_sf_from_chunked(host_u8(sf), rows, K)
        np.testing.assert_array_equal(got, osf.T if along else osf)
    fq.get_status(clear=True)


def random_operand(rng, shape, fmt):
    v = rng.standard_normal(shape).astype(np.float32) * (100.0 if fmt == 0 else 3000.0)
    return oracle.fp8_encode(v, fmt)


def run_gemm(layout, M, N, K, fa, fb, sf_kind, out="f32", residual=False, seed=0):
    rng = np.random.default_rng(seed)
    A = random_operand(rng, (K, M) if layout == fq.TN else (M, K), fa)
    B = random_operand(rng, (N, K) if layout == fq.NT else (K, N), fb)
    kb = K // 32
    if sf_kind == "unit":
        sfA, sfB = np.full((M, kb), 127, np.uint8), np.full((N, kb), 127, np.uint8)
    elif sf_kind == "rows":      # varies with the operand row only
        sfA = np.repeat(rng.integers(115, 140, (M, 1)), kb, axis=1).astype(np.uint8)
        sfB = np.repeat(rng.integers(115, 140, (N, 1)), kb, axis=1).astype(np.uint8)
    elif sf_kind == "kblocks":   # varies with the K block only
        sfA = np.repeat(rng.integers(115, 140, (1, kb)), M, axis=0).astype(np.uint8)
        sfB = np.repeat(rng.integers(115, 140, (1, kb)), N, axis=0).astype(np.uint8)
    else:
        sfA = rng.integers(110, 145, (M, kb)).astype(np.uint8)
        sfB = rng.integers(110, 145, (N, kb)).astype(np.uint8)
    R = synth.bf16_bits(rng.standard_normal((M, N)).astype(np.float32) * 5.0) if residual else None
    C = fq.fp8_gemm_mx(layout, dev_u8(A), fa, dev_u8(mx_sf_to_chunked(sfA)), dev_u8(B), fb,
                       dev_u8(mx_sf_to_chunked(sfB)), out_dtype=torch.float32 if out == "f32" else torch.bfloat16,
                       residual=None if R is None else dev_bf16(R))
    torch.cuda.synchronize()
    ref = oracle.gemm_mx(layout, A, fa, sfA, B, fb, sfB, out="bf16" if residual else "f64", residual=R, nthreads=8)
    if residual:
        ref = oracle.bf16_to_f64(ref)
    return host_f64(C), ref


@pytest.mark.parametrize("sf_kind", ["unit", "rows", "kblocks", "random"])
def test_mx_gemm_one_tile_scale_patterns(sf_kind):
    got, ref = run_gemm(fq.NN, 128, 256, 128, 0, 0, sf_kind, seed=1)
    assert row_rel(got, ref) < 2e-3


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1)])
def test_mx_gemm_layouts_and_formats(layout, fa, fb):
    got, ref = run_gemm(layout, 272, 528, 384, fa, fb, "random", seed=10 * layout + 3 * fa + fb)
    assert row_rel(got, ref) < 2e-3


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (16, 16, 128), (400, 272, 1024), (1024, 768, 256)])
def test_mx_gemm_shapes(layout, M, N, K):
    got, ref = run_gemm(layout, M, N, K, 0, 0, "random", seed=M + N + K)
    assert row_rel(got, ref) < 2e-3


def test_mx_gemm_bf16_residual_and_deterministic():
    got, ref = run_gemm(fq.NN, 300, 512, 256, 0, 0, "random", out="bf16", residual=True, seed=6)
    assert row_rel(got, ref) < 2e-3
    got2, _ = run_gemm(fq.NN, 300, 512, 256, 0, 0, "random", out="bf16", residual=True, seed=6)
    assert np.array_equal(got, got2)


# --------------------------------------------------------------------------- the MXFP8 block
SLOT_SHAPES = {"W_gu": "Wgu", "W_d": "Wd", "n": "n", "a": "a", "dY": "dY", "dH": "dH"}


def gpu_slot(b, slot, R, C):
    q, sf = b.mx[slot]
    ax = slot.rsplit("_", 1)[1]
    sfp = mx_sf_from_chunked(host_u8(sf), R, C) if ax == "r" else mx_sf_from_chunked(host_u8(sf), C, R).T
    return host_u8(q), sfp


def requant_ok(got_q, ref_q, got_sf, ref_sf, along_rows):
    """In-block requantization (input from a GEMM the oracle accumulates in fp64): >= 99.9 % of the
    blocks have the oracle's scale (the others one power of two away); inside the blocks whose
    scales agree >= 99.9 % identical codes, every other one a step away."""
    sfd = np.abs(got_sf.astype(int) - ref_sf.astype(int))
    R, C = got_q.shape
    agree = (sfd == 0)
    agree_el = np.repeat(agree, 32, axis=0) if along_rows else np.repeat(agree, 32, axis=1)
    steps = code_step_diff(got_q, ref_q)[agree_el[:R, :C]]
    ok = agree.mean() >= 0.999 and sfd.max() <= 1 and (steps == 0).mean() >= 0.999 and steps.max() <= 1
    return ok, (agree.mean(), sfd.max(), (steps == 0).mean(), steps.max())


@pytest.mark.parametrize("T,d,f,grad_e4m3", [(256, 256, 384, False), (512, 384, 640, False), (256, 128, 256, True)])
def test_mx_block_against_oracle(T, d, f, grad_e4m3):
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    inp = synth.mlp_inputs(w, seed=2, T=T, d=d, f=f)
    b = fq.MlpBuffers.allocate(T, d, f, backward=True, keep_intermediates=True, mx=True)
    b.grad_e4m3 = grad_e4m3
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    ref = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], mx=True, nthreads=8,
                       grad_fmt=0 if grad_e4m3 else 1)
    shapes = {"W_gu": (d, 2 * f), "W_d": (f, d), "n": (T, d), "a": (T, f), "dY": (T, d), "dH": (T, 2 * f)}
    for slot in fq.MX_SLOTS:
        name, ax = slot.rsplit("_", 1)
        q, sf = gpu_slot(b, slot, *shapes[name])
        rq, rsf = ref[f"mx_{SLOT_SHAPES[name]}_{ax}"], ref[f"mx_{SLOT_SHAPES[name]}_{ax}_sf"]
        if name in ("W_gu", "W_d", "n", "dY"):
            np.testing.assert_array_equal(q, rq, err_msg=slot)
            np.testing.assert_array_equal(sf, rsf, err_msg=slot)
        else:
            ok, info = requant_ok(q, rq, sf, rsf, ax == "c")
            assert ok, (slot, info)
    np.testing.assert_array_equal(b.rstd.cpu().numpy(), ref["rstd"].astype(np.float32))
    assert row_rel(host_f64(b.H), ref["H"]) < 2e-3
    assert row_rel(host_f64(b.y), ref["y"]) < 2e-3
    assert row_rel(host_f64(b.dH), ref["dH"]) < 5e-3
    assert row_rel(host_f64(b.dN), ref["dN"]) < 5e-3
    assert row_rel(host_f64(b.dX), ref["dX"]) < 5e-3
    assert row_rel(host_f64(b.dW_d), ref["dWd"]) < 5e-3
    assert row_rel(host_f64(b.dW_gu), ref["dWgu"]) < 5e-3
    assert row_rel(host_f64(b.dg)[None, :], ref["dg"][None, :]) < 5e-3
    # a rerun gives the same bits
    y1, dx1, dw1 = b.y.clone(), b.dX.clone(), b.dW_gu.clone()
    fq.mlp_block_fwd(b)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert torch.equal(y1, b.y) and torch.equal(dx1, b.dX) and torch.equal(dw1, b.dW_gu)
