"""GPU: mlp_block_run_steps, the pipelined executor that feeds the block from host memory (step
i+1's inputs copied in and step i-1's outputs copied out while step i computes, two device sets).
Each step's host outputs must equal those of mlp_block_fwd + mlp_block_bwd on the same inputs, bit
for bit (the same kernels in the same order; only the copies are scheduled differently)."""

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
