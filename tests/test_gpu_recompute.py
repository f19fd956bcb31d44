"""Recompute-mode backward (LLMQ §3.1: selective recomputation keeps only what efficient
requantization needs; the retained absmax statistics let quantization fuse with the
nonlinearity during recomputation).

With fp8q_mlp.recompute set, mlp_block_bwd ignores the forward's H and a8, recomputes H from the
retained n8, W_gu8 and scales, and writes a8 = q(SwiGLU(H)) with the retained scale of a straight
from the GEMM epilogue.  The recomputation must reproduce the forward's H and a8 bit for bit (same
operands, deterministic kernels), so the whole backward equals the normal backward bit for bit;
the normal backward is itself checked against the oracle."""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import dev_bf16
from tests.test_gpu_block import check_backward

pytestmark = pytest.mark.gpu


def run(T, d, f, recompute, wname="7b-mlp-fwd-bwd"):
    w = synth.BY_NAME[wname]
    inp = synth.mlp_inputs(w, seed=0, T=T, d=d, f=f)
    b = fq.MlpBuffers.allocate(T, d, f, backward=True, keep_intermediates=True)
    b.recompute = recompute
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    torch.cuda.synchronize()
    saved = (b.H.clone(), b.a8.clone())
    if recompute:
        b.H.fill_(float("nan"))      # the backward must not read what the forward left here
        b.a8.fill_(0x55)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    return b, saved, inp


@pytest.mark.parametrize("T,d,f", [(272, 528, 400), (512, 1024, 1536), (8192, 3584, 18944)])
def test_recompute_backward_bit_identical(T, d, f):
    r, saved, inp = run(T, d, f, True)
    assert torch.equal(r.H, saved[0]), "recomputed H differs from the forward's"
    assert torch.equal(r.a8, saved[1]), "recomputed a8 (fused SwiGLU + E4M3 cast) differs"
    n, _, _ = run(T, d, f, False)
    for k in ("dY8", "dH", "dH8", "dN", "dX", "dW_gu", "dW_d", "dg"):
        assert torch.equal(getattr(r, k), getattr(n, k)), k


def test_recompute_backward_against_oracle():
    T, d, f = 192, 256, 384
    r, _, inp = run(T, d, f, True)
    ref = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], eps=r.eps, nthreads=16)
    check_backward(r, ref)
