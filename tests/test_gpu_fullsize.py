"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times
(mlp_block_fwd + mlp_block_bwd on the whole workload).

The CPU oracle cannot run a whole 3B/7B/14B-class block in seconds, so:
  * stages whose inputs are the original tensors are checked against the oracle bit for bit
    on the full tensors: W_gu8, W_d8 (+ scales), n8, rstd (+ scale), dY8 (+ scale);
  * H is checked against the oracle on sampled rows (the oracle computes them from its own
    n8 and W_gu8);
  * every later stage depends on a scale that needs the whole tensor, so it is checked through
    properties that hold at any size, computed in numpy from the GPU's own operands: the
    absmax/scale relations of a8 and dH8 (exact), the FP8 codes against their inputs (within
    half an FP8 step), and the GEMM identities of y, dH, dN, dW_d, dW_gu and the RMSNorm
    backward on sampled rows/columns (row-relative 2e-3 outputs, 5e-3 gradients).
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import bf16_np, dev_bf16, fp8_table, row_rel

pytestmark = pytest.mark.gpu

T4, T5 = fp8_table(0), fp8_table(1)


def as_bf16(v):
    """Round a reference to bf16 like the stored tensor it is compared with (via fp32, round to
    nearest even; the double rounding is far inside the tolerance)."""
    return synth.f32_from_bf16_bits(synth.bf16_bits(np.asarray(v, dtype=np.float32))).astype(np.float64)


def sample_rows(n, k, seed):
    r = np.random.default_rng(seed).choice(n, size=min(k, n), replace=False)
    r[0] = n - 1  # the last row sits in the ragged/last tile
    return np.sort(r)


def quant_property(values, codes, table, scale):
    """codes are the RNE FP8 rounding of values*scale: the decoded code is within half a step
    (relative 2^-4 E4M3 / 2^-3 E5M2 in the normal range, half the smallest subnormal below)."""
    p = values.astype(np.float32) * np.float32(scale)
    dq = table[codes]
    frac, sub = (3, 2.0 ** -9) if table is T4 else (2, 2.0 ** -16)
    bound = np.maximum(np.abs(p.astype(np.float64)) * 2.0 ** -(frac + 1), sub / 2) * (1 + 1e-6)
    return np.abs(dq - p) <= bound


@pytest.mark.parametrize("wname", ["3b-mlp-fwd", "7b-mlp-fwd-bwd", "14b-mlp-fwd-bwd"])
def test_full_size_block(wname):
    w = synth.BY_NAME[wname]
    T, d, f = w.T, w.d, w.f
    inp = synth.mlp_inputs(w, seed=0)
    b = fq.MlpBuffers.allocate(T, d, f, backward=w.backward, keep_intermediates=True)
    for k in ("x", "g", "W_gu", "W_d") + (("dY",) if w.backward else ()):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    if w.backward:
        fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    scal = b.scal.cpu().numpy()

    # --- bit-exact against the oracle on full tensors
    wgu8 = b.W_gu8.cpu().numpy()
    wd8 = b.W_d8.cpu().numpy()
    n8 = b.n8.cpu().numpy()
    qo, so, _ = oracle.quantize_absmax(inp["W_gu"], oracle.E4M3)
    np.testing.assert_array_equal(wgu8, qo); np.testing.assert_array_equal(scal[0], so)
    qo, so, _ = oracle.quantize_absmax(inp["W_d"], oracle.E4M3)
    np.testing.assert_array_equal(wd8, qo); np.testing.assert_array_equal(scal[1], so)
    qo, so, ro, _ = oracle.rmsnorm_quant(inp["x"], inp["g"], b.eps)
    np.testing.assert_array_equal(n8, qo); np.testing.assert_array_equal(scal[2], so)
    np.testing.assert_array_equal(b.rstd.cpu().numpy(), ro)

    rows = sample_rows(T, 24, 1)
    # --- H on sampled rows against the oracle (its own n8 = qo and W_gu8)
    H_ref = oracle.gemm_scaled(oracle.NN, qo[rows], 0, oracle.quantize_absmax(inp["W_gu"], 0)[0], 0,
                               float(so[2]), float(scal[0, 2]), out="bf16", nthreads=16)
    H = bf16_np(b.H[torch.from_numpy(rows).cuda()])
    assert row_rel(H, oracle.bf16_to_f64(H_ref)) < 2e-3

    # --- a8: amax / scale / codes (properties of the GPU's H)
    Hf = bf16_np(b.H)
    hg, hu = Hf[:, :f], Hf[:, f:]
    a = hg / (1.0 + np.exp(-hg)) * hu
    del Hf
    amax = np.abs(a).max()
    assert abs(scal[3, 0] / amax - 1) < 1e-5
    assert scal[3, 1] == np.float32(448.0) / np.float32(scal[3, 0])
    a8 = b.a8.cpu().numpy()
    ok = quant_property(a[rows], a8[rows], T4, scal[3, 1])
    assert ok.mean() > 0.9999, ok.mean()          # fp64 vs exp_ref SwiGLU may straddle a midpoint
    del a, hg, hu

    # --- y = bf16(x + alpha2 a8 @ W_d8) on sampled rows
    Wd = T4[wd8]
    y_ref = as_bf16(oracle.bf16_to_f64(inp["x"][rows]) + (scal[3, 2] * scal[1, 2]) * (T4[a8[rows]] @ Wd))
    assert row_rel(bf16_np(b.y[torch.from_numpy(rows).cuda()]), y_ref) < 2e-3
    if not w.backward:
        return

    # --- backward
    dY8 = b.dY8.cpu().numpy()
    qo, so, _ = oracle.quantize_absmax(inp["dY"], oracle.E5M2)
    np.testing.assert_array_equal(dY8, qo); np.testing.assert_array_equal(scal[4], so)
    Hr = bf16_np(b.H[torch.from_numpy(rows).cuda()])
    dA = np.float64(np.float32(scal[4, 2] * scal[1, 2])) * (T5[dY8[rows]] @ Wd.T)
    h, u = Hr[:, :f], Hr[:, f:]
    sg = 1 / (1 + np.exp(-h))
    dH_ref = as_bf16(np.concatenate([dA * u * sg * (1 + h * (1 - sg)), dA * h * sg], axis=1))
    dH = b.dH
    assert row_rel(bf16_np(dH[torch.from_numpy(rows).cuda()]), dH_ref) < 5e-3
    dHa = bf16_np(dH)
    assert scal[5, 0] == np.float32(np.abs(dHa).max())        # exact: max over the stored bf16 values
    assert scal[5, 1] == np.float32(57344.0) / np.float32(scal[5, 0])
    dH8 = b.dH8.cpu().numpy()
    assert quant_property(dHa[rows], dH8[rows], T5, scal[5, 1]).all()
    del dHa
    # dN = alpha5 dH8 @ W_gu8^T
    dN_ref = np.float64(np.float32(scal[5, 2] * scal[0, 2])) * (T5[dH8[rows]] @ T4[wgu8].T)
    dN = b.dN.cpu().numpy().astype(np.float64)
    assert row_rel(dN[rows], dN_ref) < 5e-3
    # dW_d = alpha4 a8^T @ dY8 (sampled rows of dW_d = columns of a8)
    cols = sample_rows(f, 16, 2)
    dWd_ref = np.float64(np.float32(scal[3, 2] * scal[4, 2])) * (T4[a8[:, cols]].T @ T5[dY8])
    assert row_rel(b.dW_d.cpu().numpy().astype(np.float64)[cols], dWd_ref) < 5e-3
    # dW_gu = alpha6 n8^T @ dH8 on sampled rows x columns
    ri, cj = sample_rows(d, 12, 3), sample_rows(2 * f, 48, 4)
    dWgu_ref = np.float64(np.float32(scal[2, 2] * scal[5, 2])) * (T4[n8[:, ri]].T @ T5[dH8[:, cj]])
    got = b.dW_gu.cpu().numpy().astype(np.float64)[np.ix_(ri, cj)]
    assert row_rel(got, dWgu_ref) < 5e-3
    # RMSNorm backward + residual on sampled rows; dg over all rows
    x = oracle.bf16_to_f64(inp["x"])
    g = oracle.bf16_to_f64(inp["g"])
    rstd = b.rstd.cpu().numpy().astype(np.float64)
    nh = x[rows] * rstd[rows, None]
    uu = dN[rows] * g
    dX_ref = as_bf16(oracle.bf16_to_f64(inp["dY"][rows])
                     + rstd[rows, None] * (uu - nh * (uu * nh).mean(axis=1, keepdims=True)))
    assert row_rel(bf16_np(b.dX[torch.from_numpy(rows).cuda()]), dX_ref) < 5e-3
    dg_ref = (dN * (x * rstd[:, None])).sum(axis=0)
    assert row_rel(b.dg.cpu().numpy().astype(np.float64)[None, :], dg_ref[None, :]) < 5e-3
