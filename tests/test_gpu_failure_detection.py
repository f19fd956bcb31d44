"""Failure detection without a GPU fault.

Every pipelined kernel of the library waits on mbarriers through one bounded wait that gives up
after a time limit, records FP8Q_STATUS_TIMEOUT in the device status word and lets the kernel
return.  Here that wait is made to run out on purpose -- an mbarrier that nothing ever arrives at,
with a 20 ms limit -- and the test checks the status the host reads afterwards and that the CUDA
context is still usable (a quantization afterwards is correct and leaves the status clean).
Argument errors are reported synchronously (no kernel launched)."""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import dev_bf16

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
