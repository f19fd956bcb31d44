"""GPU parity: the MLP block forward + backward through the C ABI against the CPU oracle.

Per-tensor FP8 block of the LLMQ pages (§1 dynamic tensor-level scaling, §3/§3.1 fused
RMSNorm / SwiGLU-requant / residual, §5 Fig. 2 E4M3 forward and E5M2 gradients).
  * quantizers whose input is an exact given tensor are bit-exact: W_gu8, W_d8, n8, rstd, dY8
    and their scales;
  * GEMM outputs (H, y) within 2e-3 max row-relative L2 error; gradients (dX, dW_gu, dW_d, dg)
    within 5e-3;
  * quantizers fed by an fp32 GEMM (a8 from H, dH8 from dH) can differ from the fp64 oracle only
    where the bf16 value they quantize differs by an ulp: >= 99.9% identical codes, every
    other code one step away, amax within one bf16 ulp.
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import code_step_diff, dev_bf16, host_bits, host_f64, row_rel

pytestmark = pytest.mark.gpu


def run_block(wname, T, d, f, backward=True, seed=0, grad_e4m3=False):
    w = synth.BY_NAME[wname]
    inp = synth.mlp_inputs(w, seed=seed, T=T, d=d, f=f)
    if backward and "dY" not in inp:
        inp["dY"] = synth.normal_bf16((T, d), 1e-3, seed, synth.TID_DY)
    b = fq.MlpBuffers.allocate(T, d, f, backward=backward, keep_intermediates=True)
    b.grad_e4m3 = grad_e4m3
    for k in ("x", "g", "W_gu", "W_d") + (("dY",) if backward else ()):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    if backward:
        fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    ref = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"] if backward else None,
                       eps=b.eps, nthreads=16, grad_fmt=oracle.E4M3 if grad_e4m3 else oracle.E5M2)
    return b, ref


def check_requant(codes_gpu, codes_ref, amax_gpu, amax_ref):
    same = (codes_gpu == codes_ref).mean()
    assert same >= 0.999, same
    assert code_step_diff(codes_gpu, codes_ref).max() <= 1
    assert abs(amax_gpu / amax_ref - 1) <= 2.0 ** -7


def check_forward(b, ref):
    scal = b.scal.cpu().numpy()
    np.testing.assert_array_equal(b.W_gu8.cpu().numpy(), ref["Wgu8"])
    np.testing.assert_array_equal(b.W_d8.cpu().numpy(), ref["Wd8"])
    np.testing.assert_array_equal(b.n8.cpu().numpy(), ref["n8"])
    np.testing.assert_array_equal(b.rstd.cpu().numpy(), ref["rstd"].astype(np.float32))
    np.testing.assert_array_equal(scal[:3], ref["scal_fwd"][:3])
    assert row_rel(host_f64(b.H), ref["H"]) < 2e-3
    check_requant(b.a8.cpu().numpy(), ref["a8"], scal[3, 0], ref["scal_fwd"][3, 0])
    assert row_rel(host_f64(b.y), ref["y"]) < 2e-3


def check_backward(b, ref):
    scal = b.scal.cpu().numpy()
    np.testing.assert_array_equal(b.dY8.cpu().numpy(), ref["dY8"])
    np.testing.assert_array_equal(scal[4], ref["scal_bwd"][0])
    assert row_rel(host_f64(b.dH), ref["dH"]) < 5e-3
    check_requant(b.dH8.cpu().numpy(), ref["dH8"], scal[5, 0], ref["scal_bwd"][1, 0])
    assert row_rel(host_f64(b.dN), ref["dN"]) < 5e-3
    assert row_rel(host_f64(b.dX), ref["dX"]) < 5e-3
    assert row_rel(host_f64(b.dW_gu), ref["dWgu"]) < 5e-3
    assert row_rel(host_f64(b.dW_d), ref["dWd"]) < 5e-3
    assert row_rel(host_f64(b.dg)[None, :], ref["dg"][None, :]) < 5e-3


# (2048, 256, 256): x is more than a third of the forward prologue's bytes, so the RMSNorm
# statistics take every resident slot of their launch
@pytest.mark.parametrize("T,d,f", [(192, 256, 384), (272, 528, 400), (1, 16, 16), (640, 1024, 1280), (2048, 256, 256)])
def test_block_small_shapes(T, d, f):
    b, ref = run_block("7b-mlp-fwd-bwd", T, d, f)
    check_forward(b, ref)
    check_backward(b, ref)


def test_block_tiny_workload_full_size():
    """The tiny MLP forward workload (T=256, d=512, f=1408) at its full size, all outputs."""
    w = synth.BY_NAME["tiny-mlp-fwd"]
    b, ref = run_block(w.name, w.T, w.d, w.f, backward=False)
    check_forward(b, ref)


def test_block_tiny_workload_with_backward():
    b, ref = run_block("tiny-mlp-fwd", 256, 512, 1408, backward=True)
    check_forward(b, ref)
    check_backward(b, ref)


def test_block_deterministic():
    w = synth.BY_NAME["14b-mlp-fwd-bwd"]
    outs = []
    for _ in range(2):
        b, _ = run_block(w.name, 320, 512, 768)
        outs.append([t.clone() for t in (b.y, b.dX, b.dW_gu, b.dW_d, b.dg, b.a8, b.dH8)])
    for a, c in zip(*outs):
        assert torch.equal(a, c)


@pytest.mark.parametrize("T,d,f", [(272, 528, 400), (640, 1024, 1280)])
def test_block_e4m3_gradients(T, d, f):
    """LLMQ §5 Figure 2's E4M3-everywhere recipe: dY and dH quantized to E4M3."""
    b, ref = run_block("7b-mlp-fwd-bwd", T, d, f, grad_e4m3=True)
    assert float(b.scal[4, 1]) == float(np.float32(448.0) / np.float32(b.scal[4, 0].item()))
    check_forward(b, ref)
    check_backward(b, ref)
