"""GPU: mlp_block_run_steps, the pipelined executor that feeds the block from host memory (step
i+1's inputs copied in and step i-1's outputs copied out while step i computes, two device sets).
Each step's host outputs must equal those of mlp_block_fwd + mlp_block_bwd on the same inputs, bit
for bit (the same kernels in the same order; only the copies are scheduled differently), with
every tensor through the host and with the model state resident on the device."""

import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import synth
from tests._gpu import dev_bf16

pytestmark = pytest.mark.gpu

INPUTS = ("x", "g", "W_gu", "W_d", "dY")
OUTPUTS = ("y", "dX", "dW_gu", "dW_d", "dg")


@pytest.mark.parametrize("n_steps", [1, 2, 5])
def test_run_steps_matches_separate_calls(n_steps):
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = 384, 512, 768
    b0 = fq.MlpBuffers.allocate(T, d, f)
    b1 = fq.MlpBuffers.allocate(T, d, f)
    ref = fq.MlpBuffers.allocate(T, d, f)
    host = []
    for i in range(n_steps):
        inp = synth.mlp_inputs(w, seed=10 + i, T=T, d=d, f=f)
        h = {k: dev_bf16(inp[k]).cpu().pin_memory() for k in INPUTS}
        h.update({k: torch.empty_like(getattr(b0, k), device="cpu").pin_memory() for k in OUTPUTS})
        host.append(h)
    fq.get_status(clear=True)
    fq.mlp_block_run_steps(b0, b1, host)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for i in range(n_steps):
        for k in INPUTS:
            getattr(ref, k).copy_(host[i][k])
        fq.mlp_block_fwd(ref)
        fq.mlp_block_bwd(ref)
        torch.cuda.synchronize()
        for k in OUTPUTS:
            assert torch.equal(host[i][k], getattr(ref, k).cpu()), (i, k)


def test_run_steps_rejects_shared_buffers():
    b0 = fq.MlpBuffers.allocate(128, 256, 256)
    h = {k: torch.empty_like(getattr(b0, k), device="cpu") for k in INPUTS + OUTPUTS}
    with pytest.raises(fq.Fp8qError):
        fq.mlp_block_run_steps(b0, b0, [h])


def test_run_steps_resident_model_state():
    """Weights, gain and weight gradients resident on the device (no host pointer, one buffer
    shared by both sets), only the batch crossing the host link: each step's y and dX equal the
    separate calls' bit for bit, and the shared weight gradients hold the last step's."""
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f, n_steps = 384, 512, 768, 4
    b0 = fq.MlpBuffers.allocate(T, d, f)
    b1 = fq.MlpBuffers.allocate(T, d, f)
    ref = fq.MlpBuffers.allocate(T, d, f)
    state = synth.mlp_inputs(w, seed=30, T=T, d=d, f=f)
    for k in ("g", "W_gu", "W_d"):
        getattr(b0, k).copy_(dev_bf16(state[k]))
        getattr(ref, k).copy_(getattr(b0, k))
    for k in ("g", "W_gu", "W_d", "dW_gu", "dW_d", "dg"):
        setattr(b1, k, getattr(b0, k))
    host = []
    for i in range(n_steps):
        inp = synth.mlp_inputs(w, seed=40 + i, T=T, d=d, f=f)
        h = {k: dev_bf16(inp[k]).cpu().pin_memory() for k in ("x", "dY")}
        h.update({k: torch.empty_like(getattr(b0, k), device="cpu").pin_memory() for k in ("y", "dX")})
        host.append(h)
    fq.get_status(clear=True)
    fq.mlp_block_run_steps(b0, b1, host)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for i in range(n_steps):
        for k in ("x", "dY"):
            getattr(ref, k).copy_(host[i][k])
        fq.mlp_block_fwd(ref)
        fq.mlp_block_bwd(ref)
        torch.cuda.synchronize()
        for k in ("y", "dX"):
            assert torch.equal(host[i][k], getattr(ref, k).cpu()), (i, k)
    for k in ("dW_gu", "dW_d", "dg"):
        assert torch.equal(getattr(b0, k), getattr(ref, k)), k


def test_run_steps_rejects_moving_a_shared_buffer():
    """A buffer the two sets share may not be copied in or out in any step."""
    b0 = fq.MlpBuffers.allocate(128, 256, 256)
    b1 = fq.MlpBuffers.allocate(128, 256, 256)
    b1.W_gu = b0.W_gu
    base = {k: torch.empty_like(getattr(b0, k), device="cpu") for k in ("x", "dY", "y", "dX")}
    moved = dict(base, W_gu=torch.empty_like(b0.W_gu, device="cpu"))
    with pytest.raises(fq.Fp8qError):
        fq.mlp_block_run_steps(b0, b1, [base, moved])
