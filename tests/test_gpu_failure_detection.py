"""Failure detection without a GPU fault.

Every pipelined kernel of the library waits on mbarriers through one bounded wait that gives up
after a time limit, records FP8Q_STATUS_TIMEOUT in the device status word and lets the kernel
return.  Here that wait is made to run out on purpose -- an mbarrier that nothing ever arrives at,
with a 20 ms limit -- and the test checks the status the host reads afterwards and that the CUDA
context is still usable (a quantization afterwards is correct and leaves the status clean).
Argument errors are reported synchronously (no kernel launched).

The GEMM's own abort sequence is exercised the same way: fp8q_selftest_gemm_wait_limit launches the
production GEMM kernels (the 128 x 256 tile with its double-buffered accumulators, the 256 x 256
wide tile for long K) with their pipeline waits limited to a few microseconds, so that ordinary,
finite waits -- the first TMA loads, the accumulator hand-off -- give up.  Each CTA then records
the time-out, stops issuing, drains the copies and MMAs it issued (with the full limit), frees its
tensor memory and exits; the test checks the status bit and that the same GEMM afterwards, and a
different one, still match the oracle on the same context."""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import dev_bf16, row_rel

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    fq.get_status(clear=True)
    fq.selftest_bounded_wait(0.02)
    torch.cuda.synchronize()
    st = fq.get_status(clear=True)
    assert st & fq.STATUS_TIMEOUT
    assert fq.get_status() == 0
    # the context is intact: a normal call still gives the oracle's bits
    x = synth.normal_bf16((1 << 16,), 1.0, seed=3, tensor_id=1)
    q, scal = fq.fp8_quantize_absmax(dev_bf16(x), fq.E4M3)
    torch.cuda.synchronize()
    qo, so, _ = oracle.quantize_absmax(x, fq.E4M3)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(scal.cpu().numpy(), so)
    assert fq.get_status() == 0


def test_selftest_limit_is_validated():
    with pytest.raises(fq.Fp8qError):
        fq.selftest_bounded_wait(1e-6)
    with pytest.raises(fq.Fp8qError):
        fq.selftest_bounded_wait(100.0)


def random_codes(rng, shape, fmt):
    return oracle.fp8_encode(rng.standard_normal(shape).astype(np.float32) * 60.0, fmt)


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 1024),    # 128 x 256 tiles (two accumulators)
                                   (4864, 2048, 8192)])   # the 256 x 256 wide tile (K >= 8192)
def test_gemm_abort_sequence_on_short_waits(M, N, K):
    rng = np.random.default_rng(M + K)
    A, B = random_codes(rng, (M, K), 0), random_codes(rng, (K, N), 0)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    s = torch.tensor([0.01, 0.02], dtype=torch.float32, device="cuda")
    fq.get_status(clear=True)
    fq.selftest_gemm_wait_limit(fq.NN, dA, 0, dB, 0, 2e-6, sinvA=s[0:1], sinvB=s[1:2])
    torch.cuda.synchronize()
    assert fq.get_status(clear=True) & fq.STATUS_TIMEOUT
    # the same GEMM with the normal limit, on the same context: complete and right
    C = fq.fp8_gemm_scaled(fq.NN, dA, 0, dB, 0, s[0:1], s[1:2], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    rows = np.array([0, 1, 127, 128, 255, 256, M // 2 + 3, M - 1])
    ref = oracle.gemm_scaled(oracle.NN, A[rows], 0, B, 0, 0.01, 0.02, out="f64", nthreads=8)
    assert row_rel(C.cpu().numpy()[rows].astype(np.float64), ref) < 2e-3
    # and a different GEMM (another layout and format)
    A2, B2 = random_codes(rng, (256, 512), 1), random_codes(rng, (384, 512), 0)
    C2 = fq.fp8_gemm_scaled(fq.NT, torch.from_numpy(A2).cuda(), 1, torch.from_numpy(B2).cuda(), 0, s[0:1], s[1:2],
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref2 = oracle.gemm_scaled(oracle.NT, A2, 1, B2, 0, 0.01, 0.02, out="f64", nthreads=8)
    assert row_rel(C2.cpu().numpy().astype(np.float64), ref2) < 2e-3
    assert fq.get_status() == 0


def test_mx_gemm_abort_sequence_on_short_waits():
    """The block-scaled kernel (one accumulator, scale chunks staged and copied to tensor memory
    each stage) through the same abort sequence, then a normal block-scaled GEMM on the context."""
    from tests._gpu import mx_sf_to_chunked
    rng = np.random.default_rng(3)
    M, N, K = 2048, 2048, 1024
    A, B = random_codes(rng, (M, K), 0), random_codes(rng, (K, N), 0)
    sfA = rng.integers(120, 134, (M, K // 32)).astype(np.uint8)
    sfB = rng.integers(120, 134, (N, K // 32)).astype(np.uint8)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dsA, dsB = torch.from_numpy(mx_sf_to_chunked(sfA)).cuda(), torch.from_numpy(mx_sf_to_chunked(sfB)).cuda()
    fq.get_status(clear=True)
    fq.selftest_gemm_wait_limit(fq.NN, dA, 0, dB, 0, 2e-6, sfA=dsA, sfB=dsB)
    torch.cuda.synchronize()
    assert fq.get_status(clear=True) & fq.STATUS_TIMEOUT
    C = fq.fp8_gemm_mx(fq.NN, dA, 0, dsA, dB, 0, dsB, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    rows = np.array([0, 127, 128, 1000, M - 1])
    ref = oracle.gemm_mx(oracle.NN, A[rows], 0, sfA[rows], B, 0, sfB, out="f64", nthreads=8)
    assert row_rel(C.cpu().numpy()[rows].astype(np.float64), ref) < 2e-3


def test_gemm_wait_limit_is_validated():
    A = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones(2, dtype=torch.float32, device="cuda")
    with pytest.raises(fq.Fp8qError):
        fq.selftest_gemm_wait_limit(fq.NN, A, 0, A, 0, 1e-7, sinvA=s[0:1], sinvB=s[1:2])
