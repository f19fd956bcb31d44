"""GPU: guard bands.  Every output the kernels write is placed inside a larger buffer whose
surroundings hold a canary pattern; after the call the canaries must be intact, so no kernel
writes outside its tensor -- past a ragged tile edge, past the end of a row (GEMM outputs with a
padded row stride), before or after the tensor.  A race or an off-by-one tile index that parity
might average away shows up here as a changed canary byte."""

import ctypes

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import synth
from tests._gpu import dev_bf16, dev_u8

pytestmark = pytest.mark.gpu

G = 8192  # guard elements on each side
CANARY = {torch.uint8: 0xA5, torch.bfloat16: 0x7FC1, torch.float32: 0x7FC00001}
INT_VIEW = {torch.uint8: torch.uint8, torch.bfloat16: torch.int16, torch.float32: torch.int32}


class Guarded:
    """A contiguous tensor of `shape` inside a buffer with G canary elements before and after."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.buf = torch.empty(n + 2 * G, dtype=dtype, device="cuda")
        self.buf.view(INT_VIEW[dtype]).fill_(CANARY[dtype] if dtype != torch.bfloat16 else np.int16(CANARY[dtype]))
        self.t = self.buf[G:G + n].view(*shape)
        self.dtype, self.n = dtype, n

    def intact(self):
        iv = self.buf.view(INT_VIEW[self.dtype])
        c = CANARY[self.dtype] if self.dtype != torch.bfloat16 else int(np.int16(CANARY[self.dtype]))
        return bool((iv[:G] == c).all()) and bool((iv[G + self.n:] == c).all())


def test_gemm_padded_rows_and_ragged_tiles():
    """C [M, N] with a row stride of N + 48 inside a guarded buffer: the padding columns and
    the bands before and after stay untouched for every layout, output type and ragged shape."""
    rng = np.random.default_rng(3)
    sinv = torch.ones(2, device="cuda")
    for layout in (fq.NN, fq.NT, fq.TN):
        for (M, N, K) in ((200, 272, 160), (129, 48, 64), (912, 528, 512)):
            for out in (torch.bfloat16, torch.float32):
                if layout == fq.TN and M % 16:
                    continue  # TN keeps A MN-major: M is its leading dimension
                A = rng.integers(0, 126, size=(K, M) if layout == fq.TN else (M, K), dtype=np.uint8)
                B = rng.integers(0, 126, size=(N, K) if layout == fq.NT else (K, N), dtype=np.uint8)
                ldc = N + 48
                Cg = Guarded((M, ldc), out)
                Cg.t.view(INT_VIEW[out]).fill_(CANARY[out] if out != torch.bfloat16 else int(np.int16(CANARY[out])))
                dA, dB = dev_u8(A), dev_u8(B)
                i64 = ctypes.c_int64
                code = fq.BF16 if out == torch.bfloat16 else fq.F32
                rc = fq.lib.fp8_gemm_scaled(layout, i64(M), i64(N), i64(K), fq._ptr(dA), 0, i64(dA.shape[1]),
                                            fq._ptr(dB), 0, i64(dB.shape[1]), fq._ptr(sinv[0:1]), fq._ptr(sinv[1:2]),
                                            fq._ptr(Cg.t), code, i64(ldc), None, i64(0), fq._stream())
                assert rc == 0
                torch.cuda.synchronize()
                assert Cg.intact(), (layout, M, N, K, out)
                pad = Cg.t[:, N:].contiguous().view(INT_VIEW[out])
                c = CANARY[out] if out != torch.bfloat16 else int(np.int16(CANARY[out]))
                assert bool((pad == c).all()), ("row padding written", layout, M, N, K, out)
                body = Cg.t[:, :N].float()
                assert bool(torch.isfinite(body).all())


@pytest.mark.parametrize("n", [1, 17, 4096 + 8, 1 << 20])
def test_quantizer_bands(n):
    x = dev_bf16(synth.normal_bf16((n,), 1.0, n, 5))
    q = Guarded((n,), torch.uint8)
    fq.fp8_quantize_absmax(x, fq.E4M3, q=q.t)
    torch.cuda.synchronize()
    assert q.intact()


def test_rmsnorm_and_swiglu_bands():
    T, d, f = 37, 528, 400
    x = dev_bf16(synth.normal_bf16((T, d), 1.0, 1, 6))
    g = dev_bf16(synth.normal_bf16((d,), 0.1, 1, 7, mean=1.0))
    q, rstd = Guarded((T, d), torch.uint8), Guarded((T,), torch.float32)
    fq.rmsnorm_quant(x, g, 1e-6, q=q.t, rstd=rstd.t)
    H = dev_bf16(synth.normal_bf16((T, 2 * f), 1.0, 1, 8))
    a8 = Guarded((T, f), torch.uint8)
    fq.swiglu_quant(H, fq.E4M3, q=a8.t)
    torch.cuda.synchronize()
    assert q.intact() and rstd.intact() and a8.intact()


def test_mlp_block_bands():
    """Every tensor the MLP block writes, forward and backward, at a ragged shape."""
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = 272, 528, 400
    b = fq.MlpBuffers.allocate(T, d, f, keep_intermediates=True)
    inp = synth.mlp_inputs(w, seed=4, T=T, d=d, f=f)
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    guarded = {}
    for k in ("W_gu8", "W_d8", "n8", "rstd", "H", "a8", "y", "dX", "dW_gu", "dW_d", "dg", "dY8", "dH", "dH8", "dN"):
        t = getattr(b, k, None)
        if t is None:
            continue
        gt = Guarded(tuple(t.shape), t.dtype)
        setattr(b, k, gt.t)
        guarded[k] = gt
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    for k, gt in guarded.items():
        assert gt.intact(), k


def test_attention_bands():
    S, B, Hq, Hkv = 256, 2, 4, 2
    T = S * B
    qkv = dev_bf16(synth.normal_bf16((T, (Hq + 2 * Hkv) * 128), 0.7, 2, 9))
    att, lse = Guarded((T, Hq * 128), torch.bfloat16), Guarded((Hq, T), torch.float32)
    fq.attention_fwd(qkv, S, Hq, Hkv, att=att.t, lse=lse.t)
    dO = dev_bf16(synth.normal_bf16((T, Hq * 128), 1e-3, 2, 10))
    dqkv = Guarded(tuple(qkv.shape), torch.bfloat16)
    fq.attention_bwd(qkv, att.t, lse.t, dO, S, Hq, Hkv, dqkv=dqkv.t)
    torch.cuda.synchronize()
    assert att.intact() and lse.intact() and dqkv.intact()
