"""The C ABI without a GPU: libfp8q.so builds, loads, exports every entry point that
include/*.h declares, and rejects bad arguments synchronously with the documented codes
before touching the device."""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_absmax_reduce_gb300 import build as b
    b.build()
    import fp8_absmax_reduce_gb300 as fq
    return fq.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names += re.findall(r"^FP8Q_API\s+[\w\s\*]+?\b(\w+)\s*\(", open(h).read(), flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_workspace_sizes(lib):
    assert lib.fp8q_status_string(0) == b"ok"
    assert lib.fp8q_status_string(1) == b"invalid argument"
    assert lib.fp8_quantize_absmax_workspace_size(1 << 20) >= 4096
    small = lib.mlp_block_workspace_size(16, 16, 16, 0)
    big = lib.mlp_block_workspace_size(8192, 3584, 18944, 1)
    assert 0 < small < big
    # backward workspace holds dY8, dH (bf16), dH8, dN (fp32) and the dg partials
    T, d, f = 8192, 3584, 18944
    assert big >= T * d + T * 2 * f * 2 + T * 2 * f + T * d * 4 + (T // 16) * d * 4


def test_invalid_arguments_rejected_without_device(lib):
    INVALID = 1
    vp = ctypes.c_void_p
    fake = vp(1 << 20)        # 16-byte aligned, never dereferenced
    odd = vp((1 << 20) + 4)   # misaligned
    # quantize: n < 1, misaligned input, bad format
    assert lib.fp8_quantize_absmax(fake, 0, 0, 0, fake, fake, fake, 4096, None) == INVALID
    assert lib.fp8_quantize_absmax(odd, 0, 64, 0, fake, fake, fake, 4096, None) == INVALID
    assert lib.fp8_quantize_absmax(fake, 0, 64, 7, fake, fake, fake, 4096, None) == INVALID
    # GEMM: K-major operand with K not a multiple of 16; residual with fp32 output; bad layout
    i64 = ctypes.c_int64
    assert lib.fp8_gemm_scaled(1, i64(64), i64(64), i64(24), fake, 0, i64(24), fake, 0, i64(24), fake, fake, fake,
                               1, i64(64), None, i64(0), None) == INVALID
    assert lib.fp8_gemm_scaled(0, i64(64), i64(64), i64(32), fake, 0, i64(32), fake, 0, i64(64), fake, fake, fake,
                               1, i64(64), fake, i64(64), None) == INVALID
    assert lib.fp8_gemm_scaled(5, i64(64), i64(64), i64(32), fake, 0, i64(32), fake, 0, i64(64), fake, fake, fake,
                               1, i64(64), None, i64(0), None) == INVALID
    # RMSNorm: d not a multiple of 16, d above the 8192 limit
    assert lib.rmsnorm_quant(fake, fake, 4, 24, ctypes.c_float(1e-6), fake, fake, fake, fake, 4096, None) == INVALID
    assert lib.rmsnorm_quant(fake, fake, 4, 8208, ctypes.c_float(1e-6), fake, fake, fake, fake, 4096, None) == INVALID
    # SwiGLU: f not a multiple of 16
    assert lib.swiglu_quant(fake, 4, 40, 0, fake, fake, fake, 4096, None) == INVALID
    # workspace too small
    assert lib.swiglu_quant(fake, 4, 32, 0, fake, fake, fake, 16, None) == 6
    # block: null descriptor
    assert lib.mlp_block_fwd(None, fake, 1 << 20, None) == INVALID
