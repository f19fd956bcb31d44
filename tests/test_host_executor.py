"""Host logic of the pipelined executors without a GPU: mlp_block_run_steps,
mlp_block_fwd_run_steps and block_run_steps check their arguments before any device call, so
with fake (aligned, never dereferenced) pointers the rejections are visible on the CPU:
  * a device buffer the two sets share may not be copied in or out in any step;
  * forward-only steps take no backward tensors;
  * with the attention core inside the block, att and dQKV are results, not inputs;
  * sets of different sizes are rejected.
A call that passes every check goes on to the device and, on a machine without one, fails with
the CUDA error code instead -- which shows the check itself let it through."""

import ctypes
import itertools

import pytest

import fp8_absmax_reduce_gb300 as fq

INVALID, CUDA = 1, 3


@pytest.fixture(scope="module")
def lib():
    from fp8_absmax_reduce_gb300 import build as b
    b.build()
    return fq.load_library()


_addr = itertools.count(1 << 24, 1 << 20)  # distinct 1 MiB-aligned fake addresses


def fake():
    return next(_addr)


def mlp_set(T=256, d=256, f=256):
    m = fq.FP8QMlp(T=T, d=d, f=f, eps=1e-6)
    for name in fq._MLP_PTRS:
        setattr(m, name, fake())
    return m


def mlp_io(**kw):
    io = fq.FP8QMlpHostIO()
    for k, v in kw.items():
        setattr(io, k, v)
    return io


def run_mlp(lib, fn, m0, m1, steps, ws_bytes=1 << 40):
    arr = (fq.FP8QMlpHostIO * len(steps))(*steps)
    return getattr(lib, fn)(ctypes.byref(m0), ctypes.byref(m1), arr, len(steps), ctypes.c_void_p(fake()),
                            ws_bytes, None)


def test_mlp_steps_shared_buffer_rules(lib):
    m0, m1 = mlp_set(), mlp_set()
    batch = dict(x=fake(), dY=fake(), y=fake(), dX=fake())
    # weights shared and resident (no host pointer): passes the checks, then needs a device
    m1.W_gu, m1.W_d, m1.g = m0.W_gu, m0.W_d, m0.g
    assert run_mlp(lib, "mlp_block_run_steps", m0, m1, [mlp_io(**batch)]) == CUDA
    # ... but copying into a shared buffer in any step is refused
    assert run_mlp(lib, "mlp_block_run_steps", m0, m1, [mlp_io(**batch), mlp_io(W_gu=fake(), **batch)]) == INVALID
    # a shared output buffer may not be copied out either
    m1.dW_d = m0.dW_d
    assert run_mlp(lib, "mlp_block_run_steps", m0, m1, [mlp_io(dW_d=fake(), **batch)]) == INVALID
    # the batch tensors themselves shared: refused as soon as they move
    m2, m3 = mlp_set(), mlp_set()
    m3.x = m2.x
    assert run_mlp(lib, "mlp_block_run_steps", m2, m3, [mlp_io(**batch)]) == INVALID


def test_mlp_steps_shapes_and_counts(lib):
    m0, m1 = mlp_set(), mlp_set(T=512)
    assert run_mlp(lib, "mlp_block_run_steps", m0, m1, [mlp_io(x=fake())]) == INVALID
    m1 = mlp_set()
    arr = (fq.FP8QMlpHostIO * 1)()
    assert lib.mlp_block_run_steps(ctypes.byref(m0), ctypes.byref(m1), arr, 0, ctypes.c_void_p(fake()), 1 << 40,
                                   None) == INVALID
    # workspace too small
    assert run_mlp(lib, "mlp_block_run_steps", m0, m1, [mlp_io(x=fake())], ws_bytes=16) == 6


def test_mlp_fwd_steps_take_no_backward_tensors(lib):
    m0, m1 = mlp_set(), mlp_set()
    assert run_mlp(lib, "mlp_block_fwd_run_steps", m0, m1, [mlp_io(x=fake(), y=fake())]) == CUDA
    for k in ("dY", "dX", "dW_gu", "dW_d", "dg"):
        assert run_mlp(lib, "mlp_block_fwd_run_steps", m0, m1, [mlp_io(x=fake(), **{k: fake()})]) == INVALID, k


def block_set(T=256, d=256, f=256, nq=512, core=None):
    b = fq.FP8QBlock(T=T, d=d, f=f, n_qkv=nq, eps=1e-6)
    for name, _ in fq.FP8QBlock._fields_:
        if name in ("T", "d", "f", "n_qkv", "eps", "mlp", "n_heads", "n_kv_heads", "seq_len"):
            continue
        setattr(b, name, fake())
    m = mlp_set(T, d, f)
    m.x = b.h
    b.mlp = m
    if core:
        b.n_heads, b.n_kv_heads, b.seq_len = core
    return b


def run_block(lib, b0, b1, steps, backward=1):
    arr = (fq.FP8QBlockHostIO * len(steps))()
    for i, s in enumerate(steps):
        for k, v in s.items():
            setattr(arr[i], k, v)
    return lib.block_run_steps(ctypes.byref(b0), ctypes.byref(b1), arr, len(steps), backward,
                               ctypes.c_void_p(fake()), 1 << 40, None)


def test_block_steps_rules(lib):
    b0, b1 = block_set(), block_set()
    batch = dict(x=fake(), dY=fake(), att=fake(), dQKV=fake(), y=fake(), dX=fake(), d_att=fake())
    assert run_block(lib, b0, b1, [batch]) == CUDA
    # forward only: no backward tensors
    assert run_block(lib, b0, b1, [dict(x=fake(), att=fake(), y=fake())], backward=0) == CUDA
    assert run_block(lib, b0, b1, [dict(x=fake(), dY=fake())], backward=0) == INVALID
    assert run_block(lib, b0, b1, [dict(x=fake(), dW_o=fake())], backward=0) == INVALID
    # a shared weight may not move
    b1.W_o = b0.W_o
    assert run_block(lib, b0, b1, [dict(batch, W_o=fake())]) == INVALID
    # sets of different sizes
    assert run_block(lib, block_set(), block_set(T=512), [batch]) == INVALID


def test_block_steps_with_core_take_no_att_or_dqkv(lib):
    core = (2, 1, 128)
    b0, b1 = block_set(d=256, nq=512, core=core), block_set(d=256, nq=512, core=core)
    assert run_block(lib, b0, b1, [dict(x=fake(), dY=fake(), y=fake(), dX=fake())]) == CUDA
    assert run_block(lib, b0, b1, [dict(x=fake(), att=fake())]) == INVALID
    assert run_block(lib, b0, b1, [dict(x=fake(), dQKV=fake())]) == INVALID
