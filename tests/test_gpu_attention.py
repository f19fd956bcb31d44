"""GPU parity: the attention core (causal grouped-query softmax attention, bf16, tcgen05
kind::f16) through the C ABI against the oracle's fp64 definition.

The kernel rounds the probabilities P (in (0, 1]) to bf16 before they multiply V (the
tensor-core operand), keeps their fp32 row sum, and rounds att to bf16.  bf16 has 8 significant
bits, so each stored probability is off by at most 2^-8 of itself and an output element moves by
at most 2^-8 sum_k P_ik |v_kc| (the oracle's att_abs); the two bf16 roundings of the output (the
kernel's and the reference's) add at most 2^-8 |att| each.  Bar, elementwise:
|att - ref| <= 2^-8 (att_abs + 2 |ref|) (1 + 2^-6)
(the last factor covers the fp32 arithmetic), and the RMS of the error over that bound below 0.5
(the bound is a worst case); lse within 1e-5 absolute (fp32 log of the fp32 sum).

Backward: the kernels recompute P from S and lse, take D = rowsum(dO * att) from the stored att,
and round P and dS = P (dP - D) to bf16 as tensor-core operands; dqkv is bf16.  The same
first-order argument bounds every gradient element by 2^-8 (abs + 2 |ref|) (1 + 2^-6), with abs
the oracle's dqkv_abs: the size of the gradient's terms with |dS| and the error scale of D
(sum_c |dO| (att_abs + |att|)) in place of the signed values.
"""

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import oracle
import synth
from tests._gpu import dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def check_bound(got, ref, ref_abs):
    bound = 2.0 ** -8 * (ref_abs + 2 * np.abs(ref)) * (1 + 2.0 ** -6)
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:5], float((err / bound).max()))
    assert np.sqrt(np.mean((err / np.maximum(bound, 1e-300)) ** 2)) < 0.5


def check_att(got, ref):
    check_bound(got, ref["att"], ref["att_abs"])


def qkv_input(T, Hq, Hkv, seed=0, std=0.7):
    return synth.normal_bf16((T, (Hq + 2 * Hkv) * 128), std, seed, 50)


# (2176, 2, 2, 1): 17 tiles per sequence -- the odd count takes the one-tile forward, and the CTA
# order's last band is narrower than the others for dQ (bands of 16) and dK/dV (bands of 2)
@pytest.mark.parametrize("S,B,Hq,Hkv", [(128, 1, 1, 1), (256, 2, 4, 2), (384, 1, 5, 1), (512, 2, 2, 2),
                                         (256, 1, 40, 8), (1024, 2, 8, 2), (2176, 2, 2, 1)])
def test_attention_forward(S, B, Hq, Hkv):
    T = S * B
    qkv = qkv_input(T, Hq, Hkv)
    fq.get_status(clear=True)
    att, lse = fq.attention_fwd(dev_bf16(qkv), S, Hq, Hkv)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    ref = oracle.attention(qkv, S, Hq, Hkv, 128, nthreads=16, with_abs=True)
    check_att(host_f64(att), ref)
    np.testing.assert_allclose(lse.cpu().numpy().astype(np.float64), ref["lse"], atol=1e-5, rtol=0)


def test_attention_sharp_and_flat_rows():
    """Large scores (nearly one-hot rows) and q = 0 (uniform rows: prefix means)."""
    S, Hq, Hkv = 256, 2, 1
    qkv = qkv_input(S, Hq, Hkv, seed=3, std=4.0)
    qkv[:, 128:256] = 0   # head 1: q = 0
    att, lse = fq.attention_fwd(dev_bf16(qkv), S, Hq, Hkv)
    ref = oracle.attention(qkv, S, Hq, Hkv, 128, nthreads=16, with_abs=True)
    check_att(host_f64(att), ref)
    np.testing.assert_allclose(lse.cpu().numpy()[1], np.log(np.arange(1, S + 1)), atol=1e-5)


def test_attention_rejects_unsupported():
    qkv = torch.zeros((256, 3 * 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fq.Fp8qError):
        fq.lib and fq._check("attention_fwd", fq.lib.attention_fwd(fq._ptr(qkv), 256, 256, 1, 1, 64, fq._ptr(qkv),
                                                                    fq._ptr(qkv), fq._stream()))
    qkv = torch.zeros((192, 3 * 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fq.Fp8qError):
        fq.attention_fwd(qkv, 192, 1, 1)


def run_bwd(S, B, Hq, Hkv, seed=0):
    T = S * B
    qkv = qkv_input(T, Hq, Hkv, seed=seed)
    dO = synth.normal_bf16((T, Hq * 128), 1e-3, seed, 51)
    fq.get_status(clear=True)
    q = dev_bf16(qkv)
    att, lse = fq.attention_fwd(q, S, Hq, Hkv)
    dqkv = fq.attention_bwd(q, att, lse, dev_bf16(dO), S, Hq, Hkv)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    return qkv, dO, dqkv


# (2176, 2, 2, 1): 17 tiles per sequence -- the odd count takes the one-tile forward, and the CTA
# order's last band is narrower than the others for dQ (bands of 16) and dK/dV (bands of 2)
@pytest.mark.parametrize("S,B,Hq,Hkv", [(128, 1, 1, 1), (256, 2, 4, 2), (384, 1, 5, 1), (512, 2, 2, 2),
                                         (256, 1, 40, 8), (1024, 2, 8, 2), (2176, 2, 2, 1)])
def test_attention_backward(S, B, Hq, Hkv):
    qkv, dO, dqkv = run_bwd(S, B, Hq, Hkv)
    ref = oracle.attention(qkv, S, Hq, Hkv, 128, d_att=dO, nthreads=16, with_abs=True)
    got = host_f64(dqkv)
    for name, lo, hi in (("dq", 0, Hq), ("dk", Hq, Hq + Hkv), ("dv", Hq + Hkv, Hq + 2 * Hkv)):
        sl = slice(lo * 128, hi * 128)
        try:
            check_bound(got[:, sl], ref["dqkv"][:, sl], ref["dqkv_abs"][:, sl])
        except AssertionError as e:
            raise AssertionError(f"{name}: {e}")


def test_attention_backward_deterministic():
    _, _, a = run_bwd(256, 2, 4, 2, seed=1)
    _, _, b = run_bwd(256, 2, 4, 2, seed=1)
    assert torch.equal(a, b)
