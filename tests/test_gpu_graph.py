"""GPU: the block as a CUDA graph.  The library never allocates and takes every buffer from the
caller, so a whole training step (mlp_block_fwd + mlp_block_bwd, or the full block with its
attention core) can be captured once with torch.cuda.graph and replayed; the replay must give
the same bits as the direct calls (the same kernels with the same arguments).  The per-launch
trace works inside a captured step too, and on a sample of steps."""

import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import synth
from tests._gpu import dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mx", [False, True])
def test_mlp_step_graph_replay_matches_direct_calls(mx):
    """mx: the block-scaled MXFP8 block."""
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = 384, 512, 768
    b = fq.MlpBuffers.allocate(T, d, f, mx=mx)
    inp = synth.mlp_inputs(w, seed=90, T=T, d=d, f=f)
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (b.y, b.dX, b.dW_gu, b.dW_d, b.dg)]
    for t in (b.y, b.dX, b.dW_gu, b.dW_d, b.dg):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm the launch paths on a side stream before capturing
        fq.mlp_block_fwd(b)
        fq.mlp_block_bwd(b)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fq.mlp_block_fwd(b)
        fq.mlp_block_bwd(b)
    for t in (b.y, b.dX, b.dW_gu, b.dW_d, b.dg):
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for a, r in zip((b.y, b.dX, b.dW_gu, b.dW_d, b.dg), ref):
        assert torch.equal(a, r)


def test_full_block_with_core_graph_replay():
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    T, d, f, nq, core = 256, 512, 640, 1024, (4, 2, 128)
    inp = synth.block_inputs(w, seed=91, T=T, d=d, f=f, n_qkv=nq)
    b = fq.BlockBuffers.allocate(T, d, f, nq, core=core)
    for k in ("x", "g1", "W_qkv", "W_o"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    for k in ("g", "W_gu", "W_d", "dY"):
        getattr(b.mlp, k).copy_(dev_bf16(inp[k]))
    outs = lambda: (b.mlp.y, b.att, b.dX, b.dW_qkv, b.dW_o, b.mlp.dW_gu, b.mlp.dW_d)
    fq.get_status(clear=True)
    fq.block_fwd(b)
    fq.block_bwd(b)
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs()]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fq.block_fwd(b)
        fq.block_bwd(b)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fq.block_fwd(b)
        fq.block_bwd(b)
    for t in outs():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for a, r in zip(outs(), ref):
        assert torch.equal(a, r)


def test_trace_inside_a_captured_step_and_sampled_steps():
    """With the trace on while a step is captured, its events become event-record nodes of the
    graph: after a replay every traced launch has a positive duration and the sum stays inside the
    replay's own time.  fp8q_trace_resume after fp8q_trace_stop keeps the steps recorded so far."""
    import ctypes
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = 512, 512, 1024
    b = fq.MlpBuffers.allocate(T, d, f)
    inp = synth.mlp_inputs(w, seed=91, T=T, d=d, f=f)
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    lib = fq.load_library()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fq.mlp_block_fwd(b)
        fq.mlp_block_bwd(b)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert lib.fp8q_trace_start(64) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fq.mlp_block_fwd(b)
        fq.mlp_block_bwd(b)
    lib.fp8q_trace_stop()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = (ctypes.c_float * 64)()
    kinds = (ctypes.c_int * 64)()
    n = lib.fp8q_trace_read(ms, kinds, 64)
    assert n >= 10
    times = [ms[i] for i in range(n)]
    assert all(t > 0 for t in times) and sum(times) <= e0.elapsed_time(e1) * 1.01
    # a sampled trace: two direct steps traced, one between them not
    assert lib.fp8q_trace_start(64) == 0
    fq.mlp_block_fwd(b)
    lib.fp8q_trace_stop()
    fq.mlp_block_fwd(b)
    assert lib.fp8q_trace_resume() == 0
    fq.mlp_block_fwd(b)
    lib.fp8q_trace_stop()
    torch.cuda.synchronize()
    n2 = lib.fp8q_trace_read(ms, kinds, 64)
    per_fwd = n2 // 2
    assert n2 == 2 * per_fwd and per_fwd >= 3
    assert [kinds[i] for i in range(per_fwd)] == [kinds[per_fwd + i] for i in range(per_fwd)]
