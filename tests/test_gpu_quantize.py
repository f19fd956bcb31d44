"""GPU parity: fp8_quantize_absmax, rmsnorm_quant and swiglu_quant against the CPU oracle.

All three are bit-exact by construction (codes, amax, scale, scale_inv, rstd): the quantizer
input is an exact given tensor, every fp32 step is a single IEEE operation in a fixed order
(LLMQ §3.2: deterministic kernels), and the FP8 conversion is round-to-nearest-even with
saturation on both sides.  The codec cross-check runs every rounding-boundary neighbourhood
of the fp32 line through the hardware conversion (scale exactly 1).
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def run_quant(x_host, fmt):
    xd = dev_bf16(x_host) if x_host.dtype == np.uint16 else torch.from_numpy(x_host).cuda()
    q, scal = fq.fp8_quantize_absmax(xd, fmt)
    torch.cuda.synchronize()
    return q.cpu().numpy(), scal.cpu().numpy()


@pytest.mark.parametrize("fmt", [fq.E4M3, fq.E5M2])
@pytest.mark.parametrize("n", [1, 15, 16, 4097, 1 << 20, 3 * (1 << 20) + 7])
def test_quantize_bf16_bit_exact(fmt, n):
    x = synth.normal_bf16((n,), 0.7, seed=n, tensor_id=fmt + 1)
    q, scal = run_quant(x, fmt)
    qo, so, _ = oracle.quantize_absmax(x, fmt)
    np.testing.assert_array_equal(scal, so)
    np.testing.assert_array_equal(q, qo)


@pytest.mark.parametrize("fmt", [fq.E4M3, fq.E5M2])
def test_quantize_fp32_bit_exact(fmt):
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(100003) * np.exp(rng.uniform(-8, 8, 100003))).astype(np.float32)
    q, scal = run_quant(x, fmt)
    qo, so, _ = oracle.quantize_absmax(x, fmt)
    np.testing.assert_array_equal(scal, so)
    np.testing.assert_array_equal(q, qo)


@pytest.mark.parametrize("fmt", [fq.E4M3, fq.E5M2])
def test_hardware_conversion_matches_oracle_codec(fmt):
    # every fp32 high half with low halves around the rounding boundaries, restricted to
    # |v| <= fmax, plus one element equal to fmax: amax = fmax, scale = 1, codes = fp8(v)
    fmax = oracle.FMT_MAX[fmt]
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    v = (hi[:, None] | lows[None, :]).ravel().view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= fmax)]
    v = np.concatenate([v, np.array([fmax], dtype=np.float32)])
    q, scal = run_quant(v, fmt)
    assert scal[1] == 1.0
    want = oracle.fp8_encode(v, fmt)
    bad = np.nonzero(q != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches: v={v[bad[:8]]} gpu={q[bad[:8]]} oracle={want[bad[:8]]}"


def test_quantize_zero_and_nonfinite_status():
    fq.get_status(clear=True)
    q, scal = run_quant(np.zeros(64, np.uint16), fq.E4M3)
    assert (q == 0).all() and list(scal) == [0.0, 1.0, 1.0]
    assert fq.get_status() == 0
    x = np.ones(64, np.float32)
    x[5] = np.nan
    q, scal = run_quant(x, fq.E4M3)
    qo, so, st = oracle.quantize_absmax(x, fq.E4M3)
    assert st == 1 and np.isnan(scal[0])
    assert fq.get_status(clear=True) & fq.STATUS_NONFINITE
    np.testing.assert_array_equal(q, qo)


# d spans every chunk bound of the row kernel (<= 1024, 2048, 4096, 6144, 8192 elements); T = 5000
# gives its warps several rows each.
@pytest.mark.parametrize("T,d", [(1, 16), (37, 528), (256, 512), (1000, 3584), (64, 8192), (5000, 1040),
                                 (150, 2064), (200, 4112), (300, 5120), (100, 6160)])
def test_rmsnorm_quant_bit_exact(T, d):
    w = synth.BY_NAME["3b-mlp-fwd"]
    x = synth.activations(w, T, d, seed=T, tensor_id=synth.TID_X, outlier_id=synth.TID_OUTLIER)
    g = synth.normal_bf16((d,), 0.1, seed=T, tensor_id=synth.TID_G, mean=1.0)
    q, scal, rstd = fq.rmsnorm_quant(dev_bf16(x), dev_bf16(g), 1e-6)
    torch.cuda.synchronize()
    qo, so, ro, _ = oracle.rmsnorm_quant(x, g, 1e-6)
    np.testing.assert_array_equal(rstd.cpu().numpy(), ro)
    np.testing.assert_array_equal(scal.cpu().numpy(), so)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("fmt", [fq.E4M3, fq.E5M2])
@pytest.mark.parametrize("T,f", [(1, 16), (33, 400), (256, 1408), (512, 4096)])
def test_swiglu_quant_bit_exact(fmt, T, f):
    H = synth.normal_bf16((T, 2 * f), 1.5, seed=T + f, tensor_id=7)
    q, scal = fq.swiglu_quant(dev_bf16(H), fmt)
    torch.cuda.synchronize()
    qo, so, _ = oracle.swiglu_quant(H, fmt)
    np.testing.assert_array_equal(scal.cpu().numpy(), so)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
