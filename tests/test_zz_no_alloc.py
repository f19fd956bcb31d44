"""fp8_quantize_absmax_noalloc: the quantizer for callers that cannot allocate device memory.

Callers such as code whose framework owns every device allocation and gives none to plug-ins,
or latency-critical loops that must not trigger the device synchronisation of cudaMalloc/cudaFree,
cannot hand the regular entry point its workspace.  The no-allocation variant keeps that scratch in a fixed array inside the library.
This test calls it through the C ABI and requires the same bits as the regular entry point
(whose tests require bit-exactness against the CPU oracle), on calls in a row: a large
tensor, then smaller ones that read fewer partials than the earlier call left in the shared array
(the last, 16 elements, a single partial).
It is collected last so that a run stopping at the first failure has run everything else.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def c_lib():
    import fp8_absmax_reduce_gb300 as fq
    L = fq.load_library()
    L.fp8_quantize_absmax_noalloc.restype = ctypes.c_int
    L.fp8_quantize_absmax_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return L


def device_input(n, dtype, seed):
    bits = synth.normal_bf16((n,), 3.0, seed=seed, tensor_id=99)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return t if dtype == torch.bfloat16 else (t.float() * 1.7).contiguous()


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_entry_point(dtype, fmt):
    L = c_lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dcode = 0 if dtype == torch.bfloat16 else 1
    for seed, n in ((1, 3 * (1 << 20) + 5), (2, 40_001), (3, 16)):
        x = device_input(n, dtype, seed + 10 * fmt)
        q_ref = torch.empty(n, dtype=torch.uint8, device="cuda")
        s_ref = torch.empty(3, dtype=torch.float32, device="cuda")
        ws_bytes = L.fp8_quantize_absmax_workspace_size(n)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        rc = L.fp8_quantize_absmax(ctypes.c_void_p(x.data_ptr()), dcode, n, fmt, ctypes.c_void_p(q_ref.data_ptr()),
                                   ctypes.c_void_p(s_ref.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws_bytes,
                                   stream)
        assert rc == 0
        q = torch.empty(n, dtype=torch.uint8, device="cuda")
        s = torch.empty(3, dtype=torch.float32, device="cuda")
        rc = L.fp8_quantize_absmax_noalloc(ctypes.c_void_p(x.data_ptr()), dcode, n, fmt,
                                           ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(s.data_ptr()), stream)
        assert rc == 0
        assert L.fp8q_last_launch_count() == 2  # the absmax pass and the cast pass
        torch.cuda.synchronize()
        assert torch.equal(s, s_ref)
        assert torch.equal(q, q_ref)


def test_noalloc_rejects_bad_arguments():
    L = c_lib()
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(64, dtype=torch.uint8, device="cuda")
    s = torch.empty(3, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert L.fp8_quantize_absmax_noalloc(p(x), 0, 0, 0, p(q), p(s), None) == 1          # n < 1
    assert L.fp8_quantize_absmax_noalloc(p(x), 0, 64, 3, p(q), p(s), None) == 1         # bad format
    assert L.fp8_quantize_absmax_noalloc(ctypes.c_void_p(x.data_ptr() + 2), 0, 60, 0, p(q), p(s), None) == 1
