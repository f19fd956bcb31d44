"""GPU parity: fp8_gemm_scaled (tcgen05 kind::f8f6f4) against the oracle's fp64 GEMM.

Every layout (NN, NT, TN), every operand-format mix (E4M3/E5M2), bf16 and fp32 outputs, the
residual epilogue, and shapes that span several 128x256 tiles with ragged M, N and K tails.
Bar: max row-relative L2 error 2e-3 (fp32 tensor-core accumulation vs fp64).
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
from tests._gpu import dev_bf16, dev_u8, host_bits, host_f64, row_rel

pytestmark = pytest.mark.gpu


def random_codes(rng, shape, fmt):
    v = rng.standard_normal(shape).astype(np.float32) * (100.0 if fmt == 0 else 3000.0)
    return oracle.fp8_encode(v, fmt)


def run_case(layout, M, N, K, fa, fb, out, residual, seed):
    rng = np.random.default_rng(seed)
    A = random_codes(rng, (K, M) if layout == fq.TN else (M, K), fa)
    B = random_codes(rng, (N, K) if layout == fq.NT else (K, N), fb)
    sA, sB = np.float32(0.013), np.float32(0.0071)
    R = oracle.bf16_round(rng.standard_normal((M, N))) if residual else None
    sinv = torch.tensor([sA, sB], dtype=torch.float32, device="cuda")
    C = fq.fp8_gemm_scaled(layout, dev_u8(A), fa, dev_u8(B), fb, sinv[0:1], sinv[1:2],
                           out_dtype=torch.float32 if out == "f32" else torch.bfloat16,
                           residual=None if R is None else dev_bf16(R))
    torch.cuda.synchronize()
    ref = oracle.gemm_scaled(layout, A, fa, B, fb, float(sA), float(sB), out="bf16" if residual else "f64",
                             residual=R, nthreads=8)
    if residual:
        ref = oracle.bf16_to_f64(ref)
    return host_f64(C), ref


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1)])
def test_gemm_layouts_and_formats(layout, fa, fb):
    got, ref = run_case(layout, 272, 528, 400, fa, fb, "f32", False, seed=10 * layout + 3 * fa + fb)
    assert row_rel(got, ref) < 2e-3


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (16, 16, 16), (16, 32, 48), (384, 768, 1024), (144, 272, 144)])
def test_gemm_shapes(layout, M, N, K):
    got, ref = run_case(layout, M, N, K, 0, 0, "f32", False, seed=M + N + K)
    assert row_rel(got, ref) < 2e-3


@pytest.mark.parametrize("layout", [fq.NN, fq.NT])
def test_gemm_bf16_and_residual(layout):
    got, ref = run_case(layout, 300, 512, 256, 0, 0, "bf16", False, seed=5)
    assert row_rel(got, ref) < 2e-3
    got, ref = run_case(layout, 300, 512, 256, 0, 0, "bf16", True, seed=6)
    assert row_rel(got, ref) < 2e-3


def test_gemm_deterministic():
    rng = np.random.default_rng(1)
    A = dev_u8(random_codes(rng, (512, 1024), 0))
    B = dev_u8(random_codes(rng, (1024, 768), 0))
    s = torch.ones(2, device="cuda")
    c1 = fq.fp8_gemm_scaled(fq.NN, A, 0, B, 0, s[0:1], s[1:2], out_dtype=torch.float32)
    c2 = fq.fp8_gemm_scaled(fq.NN, A, 0, B, 0, s[0:1], s[1:2], out_dtype=torch.float32)
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("M,N,K", [(1, 24, 32), (7, 40, 16), (129, 264, 16)])
def test_gemm_nt_ragged_rows(M, N, K):
    # NT keeps both operands K-major, so M and N need no alignment at all
    got, ref = run_case(fq.NT, M, N, K, 1, 0, "f32", False, seed=M * N)
    assert row_rel(got, ref) < 2e-3


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("M,N,K,out,residual", [(400, 528, 8320, "f32", False), (256, 256, 8192, "bf16", False),
                                                (300, 608, 9008, "bf16", True)])
def test_gemm_long_k_wide_tiles(layout, M, N, K, out, residual):
    """K >= 8192 with a plain or residual epilogue: the 256 x 256 tile variant (two 128-row halves
    sharing the B tile), with ragged M (a half-empty second half), N and K tails."""
    if residual and layout == fq.TN:
        pytest.skip("the residual epilogue is used with NN / NT")
    got, ref = run_case(layout, M, N, K, 0, 1 if layout == fq.TN else 0, out, residual, seed=M + K)
    assert row_rel(got, ref) < 2e-3


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("M,N,K", [(912, 528, 512), (2048, 256, 384)])
def test_gemm_many_m_tiles(layout, M, N, K):
    """8 and 16 row tiles of 128 (the first with a 16-row last tile), more tiles than one
    rasterisation group walks at once: every tile must match the oracle, and repeated launches
    must agree bit for bit."""
    got, ref = run_case(layout, M, N, K, 0, 1 if layout == fq.TN else 0, "f32", False, seed=M + N + K + layout)
    assert row_rel(got, ref) < 2e-3
    got2, _ = run_case(layout, M, N, K, 0, 1 if layout == fq.TN else 0, "f32", False, seed=M + N + K + layout)
    assert np.array_equal(got, got2)


@pytest.mark.parametrize("layout", [fq.NN, fq.NT, fq.TN])
@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1)])
def test_gemm_formats_bf16_out(layout, fa, fb):
    """Four row tiles (the last ragged) with every E4M3/E5M2 operand mix and bf16 output."""
    got, ref = run_case(layout, 400, 528, 272, fa, fb, "bf16", False, seed=7 * layout + 3 * fa + fb)
    assert row_rel(got, ref) < 2e-3
