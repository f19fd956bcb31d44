"""The RMSNorm backward kernel (rmsnorm_bwd, the block backward's last step) against the oracle,
element by element, and its abort sequence.

Shapes follow the kernel's cases: d = 16 (one warp, 30 of 32 lanes idle), d = 1040 (130 column
groups: a partly idle last warp), 3584 (two blocks per SM, three row slots each), 4096 (the
largest two-block case), 5120 (one block per SM, five slots) and 8192 (1024 threads, three slots);
T from one row through ragged runs of rows per block up to 8192 rows.

Tolerances, from the arithmetic.  The kernel computes in fp32: nh = x rstd, u = dN g, the row's
sum of u nh in a fixed tree, then dY + rstd (u - nh m); the oracle computes the same in fp64 and
rounds to bf16 once.  The fp32 path is within about 1e-5 of the magnitudes it combines
(|dY| + |rstd u| + |rstd nh| mean|u nh|), so a dX element is the oracle's bf16 value or, where that
error reaches across a rounding boundary, one bf16 step away; where dY and the correction
cancel, the error is bounded by 1e-5 of those magnitudes.  dg sums T products in fp32 (runs of
at most a few hundred rows per block, then the blocks in a fixed order): within 1e-5 of the sum
of the magnitudes of its terms.
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
from tests._gpu import dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def make_inputs(T, d, seed):
    rng = np.random.default_rng(seed)
    x = oracle.bf16_round(rng.standard_normal((T, d)) * 1.5)
    dY = oracle.bf16_round(rng.standard_normal((T, d)) * 0.02)
    g = oracle.bf16_round(1.0 + 0.1 * rng.standard_normal(d))
    dN = (rng.standard_normal((T, d)) * 0.05).astype(np.float32)
    xv = oracle.bf16_to_f64(x)
    rstd = (1.0 / np.sqrt((xv * xv).mean(axis=1) + 1e-6)).astype(np.float32)
    return x, dY, g, dN, rstd


def to_device(x, dY, g, dN, rstd):
    return (torch.from_numpy(dN).cuda(), dev_bf16(x), dev_bf16(dY), dev_bf16(g), torch.from_numpy(rstd).cuda())


def check_rows(dX_bits, x, dY, g, dN, rstd, rows):
    xv, yv, gv = oracle.bf16_to_f64(x[rows]), oracle.bf16_to_f64(dY[rows]), oracle.bf16_to_f64(g)
    dn, rs = dN[rows].astype(np.float64), rstd[rows].astype(np.float64)
    ref, _ = oracle.rmsnorm_bwd(dn, xv, gv, rs, yv)
    exact, _ = oracle.rmsnorm_bwd(dn, xv, gv, rs, yv, exact=True)
    got = oracle.bf16_to_f64(dX_bits[rows])
    nh = xv * rs[:, None]
    u = dn * gv
    # the row mean's fp32 error scales with the mean of |u nh|, not with the (cancelling) mean itself
    m_abs = np.abs(u * nh).mean(axis=1, keepdims=True)
    mag = np.abs(yv) + np.abs(rs[:, None] * u) + np.abs(rs[:, None] * nh) * m_abs
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64) * 2.0 ** 16  # one bf16 step
    err = np.abs(got - ref)
    assert np.all(err <= ulp + 1e-5 * mag), float((err - ulp - 1e-5 * mag).max())
    assert (got == ref).mean() >= 0.995, (got == ref).mean()


def check_dg(dg, x, g, dN, rstd):
    xv = oracle.bf16_to_f64(x)
    terms = dN.astype(np.float64) * xv * rstd.astype(np.float64)[:, None]
    ref = terms.sum(axis=0)
    bound = 1e-5 * np.abs(terms).sum(axis=0) + np.spacing(np.abs(ref).astype(np.float32))
    assert np.all(np.abs(dg.astype(np.float64) - ref) <= bound)


@pytest.mark.parametrize("T,d", [(1, 16), (37, 16), (301, 1040), (2048, 3584), (5000, 4096), (777, 5120),
                                 (96, 8192), (8192, 3584)])
def test_rmsnorm_bwd_matches_oracle(T, d):
    x, dY, g, dN, rstd = make_inputs(T, d, seed=T + d)
    fq.get_status(clear=True)
    dX, dg = fq.rmsnorm_bwd(*to_device(x, dY, g, dN, rstd))
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    dX_bits, dg = host_bits(dX), dg.cpu().numpy()
    rows = np.arange(T) if T * d <= (1 << 22) else np.unique(np.r_[0:3, T // 3, T // 2, T - 3:T])
    check_rows(dX_bits, x, dY, g, dN, rstd, rows)
    check_dg(dg, x, g, dN, rstd)


def test_rmsnorm_bwd_repeats_bit_for_bit():
    T, d = 3000, 3584
    args = to_device(*make_inputs(T, d, seed=5))
    a, ga = fq.rmsnorm_bwd(*args)
    b, gb = fq.rmsnorm_bwd(*args)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(ga, gb)


def test_rmsnorm_bwd_abort_sequence_on_short_waits():
    """With every wait limited to 1 ns the blocks give up on their first rows: the status word
    records the time-out, the blocks drain their copies and exit, and the same call with the
    normal limit afterwards, on the same context, is complete and right."""
    T, d = 16384, 3584
    x, dY, g, dN, rstd = make_inputs(T, d, seed=9)
    args = to_device(x, dY, g, dN, rstd)
    fq.get_status(clear=True)
    fq.selftest_rmsnorm_bwd_wait_limit(*args, 1e-9)
    torch.cuda.synchronize()
    assert fq.get_status(clear=True) & fq.STATUS_TIMEOUT
    dX, dg = fq.rmsnorm_bwd(*args)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    rows = np.array([0, 1, 53, 54, 55, T // 2, T - 1])
    check_rows(host_bits(dX), x, dY, g, dN, rstd, rows)
    check_dg(dg.cpu().numpy(), x, g, dN, rstd)
