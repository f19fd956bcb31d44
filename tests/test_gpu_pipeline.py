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


@pytest.mark.parametrize("n_steps,mx", [(1, False), (2, False), (5, False), (3, True)])
def test_run_steps_matches_separate_calls(n_steps, mx):
    """mx: the block-scaled MXFP8 block through the same executor."""
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = 384, 512, 768
    b0 = fq.MlpBuffers.allocate(T, d, f, mx=mx)
    b1 = fq.MlpBuffers.allocate(T, d, f, mx=mx)
    ref = fq.MlpBuffers.allocate(T, d, f, mx=mx)
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


def test_mlp_fwd_run_steps_matches_separate_calls():
    """Forward-only steps (the inference-style workloads): y of each step equals mlp_block_fwd's,
    the weights resident and shared by both sets."""
    w = synth.BY_NAME["3b-mlp-fwd"]
    T, d, f, n_steps = 320, 512, 768, 3
    b0 = fq.MlpBuffers.allocate(T, d, f, backward=False)
    b1 = fq.MlpBuffers.allocate(T, d, f, backward=False)
    ref = fq.MlpBuffers.allocate(T, d, f, backward=False)
    state = synth.mlp_inputs(w, seed=50, T=T, d=d, f=f)
    for k in ("g", "W_gu", "W_d"):
        getattr(b0, k).copy_(dev_bf16(state[k]))
        getattr(ref, k).copy_(getattr(b0, k))
        setattr(b1, k, getattr(b0, k))
    host = []
    for i in range(n_steps):
        x = synth.mlp_inputs(w, seed=60 + i, T=T, d=d, f=f)["x"]
        host.append({"x": dev_bf16(x).cpu().pin_memory(), "y": torch.empty_like(b0.y, device="cpu").pin_memory()})
    fq.get_status(clear=True)
    fq.mlp_block_fwd_run_steps(b0, b1, host)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for i in range(n_steps):
        ref.x.copy_(host[i]["x"])
        fq.mlp_block_fwd(ref)
        torch.cuda.synchronize()
        assert torch.equal(host[i]["y"], ref.y.cpu()), i
    # a backward tensor in a forward-only run is rejected
    bad = dict(host[0], dX=torch.empty_like(b0.y, device="cpu"))
    with pytest.raises(fq.Fp8qError):
        fq.mlp_block_fwd_run_steps(b0, b1, [bad])


BLOCK_STATE = ("g1", "W_qkv", "W_o", "g", "W_gu", "W_d")
BLOCK_GRADS = ("dW_qkv", "dW_o", "dg1", "dW_gu", "dW_d", "dg")


def _block_get(b, k):
    return getattr(b.mlp, k) if k in ("g", "W_gu", "W_d", "dY", "y", "dW_gu", "dW_d", "dg") else getattr(b, k)


def _block_set(b, k, t):
    setattr(b.mlp if k in ("g", "W_gu", "W_d", "dY", "y", "dW_gu", "dW_d", "dg") else b, k, t)


@pytest.mark.parametrize("core", [None, (4, 2, 128)])
def test_block_run_steps_matches_separate_calls(core):
    """Full-block training steps through block_run_steps, model state resident and shared by the
    two sets, only the batch through the host: every step's y, dX (and d_att without the core)
    equal block_fwd + block_bwd's on the same inputs bit for bit, and the shared weight gradients
    hold the last step's."""
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    T, d, f, nq, n_steps = 256, 512, 640, 1024, 3
    sets = [fq.BlockBuffers.allocate(T, d, f, nq, core=core) for _ in range(3)]
    b0, b1, ref = sets
    state = synth.block_inputs(w, seed=70, T=T, d=d, f=f, n_qkv=nq)
    for k in BLOCK_STATE:
        _block_get(b0, k).copy_(dev_bf16(state[k]))
        _block_get(ref, k).copy_(_block_get(b0, k))
    for k in BLOCK_STATE + BLOCK_GRADS:
        _block_set(b1, k, _block_get(b0, k))
    ins = ("x", "dY") + (() if core else ("att", "dQKV"))
    outs = ("y", "dX") + (() if core else ("d_att",))
    host = []
    for i in range(n_steps):
        inp = synth.block_inputs(w, seed=80 + i, T=T, d=d, f=f, n_qkv=nq)
        h = {k: dev_bf16(inp[k]).cpu().pin_memory() for k in ins}
        h.update({k: torch.empty_like(_block_get(b0, k), device="cpu").pin_memory() for k in outs})
        host.append(h)
    fq.get_status(clear=True)
    fq.block_run_steps(b0, b1, host)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for i in range(n_steps):
        for k in ins:
            _block_get(ref, k).copy_(host[i][k])
        fq.block_fwd(ref)
        fq.block_bwd(ref)
        torch.cuda.synchronize()
        for k in outs:
            assert torch.equal(host[i][k], _block_get(ref, k).cpu()), (i, k)
    for k in BLOCK_GRADS:
        assert torch.equal(_block_get(b0, k), _block_get(ref, k)), k


def test_block_run_steps_rejects_core_inputs():
    """With the attention core inside, att and dQKV are the block's own results."""
    b0 = fq.BlockBuffers.allocate(128, 256, 256, 512, core=(2, 1, 128))
    b1 = fq.BlockBuffers.allocate(128, 256, 256, 512, core=(2, 1, 128))
    h = {"x": torch.empty_like(b0.x, device="cpu"), "att": torch.empty_like(b0.att, device="cpu")}
    with pytest.raises(fq.Fp8qError):
        fq.block_run_steps(b0, b1, [h])
