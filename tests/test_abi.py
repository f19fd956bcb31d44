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
    # RMSNorm backward: d not a multiple of 16, misaligned x, workspace too small, a zero wait limit
    ws = lib.rmsnorm_bwd_workspace_size(64, 32)
    assert ws == ((64 + 15) // 16 * 32 * 4 + 255) // 256 * 256
    assert lib.rmsnorm_bwd(fake, fake, fake, fake, fake, 64, 24, fake, fake, fake, 4096, None) == INVALID
    assert lib.rmsnorm_bwd(fake, odd, fake, fake, fake, 64, 32, fake, fake, fake, ws, None) == INVALID
    assert lib.rmsnorm_bwd(fake, fake, fake, fake, fake, 64, 32, fake, fake, fake, ws - 256, None) == 6
    assert lib.fp8q_selftest_rmsnorm_bwd_wait_limit(fake, fake, fake, fake, fake, 64, 32, fake, fake, fake, ws,
                                                    0, None) == INVALID


def test_mx_arguments_rejected_without_device(lib):
    INVALID, UNSUPPORTED = 1, 2
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fake = vp(1 << 20)
    # mx_quantize: R or C not a multiple of 128, no output, bad format
    assert lib.mx_quantize(fake, 0, i64(96), i64(128), 0, fake, fake, fake, fake, None) == INVALID
    assert lib.mx_quantize(fake, 0, i64(128), i64(200), 0, fake, fake, None, None, None) == INVALID
    assert lib.mx_quantize(fake, 0, i64(128), i64(128), 0, None, None, None, None, None) == INVALID
    assert lib.mx_quantize(fake, 0, i64(128), i64(128), 3, fake, fake, None, None, None) == INVALID
    # fp8_gemm_mx: K not a multiple of 128, a null scale pointer
    assert lib.fp8_gemm_mx(0, i64(128), i64(256), i64(96), fake, 0, i64(96), fake, fake, 0, i64(256), fake, fake, 1,
                           i64(256), None, i64(0), None) == INVALID
    assert lib.fp8_gemm_mx(0, i64(128), i64(256), i64(128), fake, 0, i64(128), None, fake, 0, i64(256), fake, fake,
                           1, i64(256), None, i64(0), None) == INVALID
    assert lib.mx_scale_bytes(i64(8192), i64(3584)) == 64 * 28 * 512
    assert lib.mx_scale_bytes(i64(130), i64(256)) == 2 * 2 * 512
    # the MXFP8 block: T not a multiple of 128; recompute is not combinable
    import fp8_absmax_reduce_gb300 as fq
    mxs = fq.FP8QMlpMx()
    for slot in fq.MX_SLOTS:
        setattr(mxs, slot, fq.FP8QMxTensor(1 << 20, 1 << 21))
    m = fq.FP8QMlp(T=192, d=256, f=256, eps=1e-6)
    for name in ("x", "g", "W_gu", "W_d", "y", "rstd", "H", "dY", "dX", "dW_gu", "dW_d", "dg"):
        setattr(m, name, 1 << 22)
    m.mx = ctypes.addressof(mxs)
    ws_bytes = lib.mlp_block_workspace_size(256, 256, 256, 1)
    assert lib.mlp_block_fwd(ctypes.byref(m), fake, ws_bytes, None) == INVALID
    m.T = 256
    m.recompute = 1
    assert lib.mlp_block_fwd(ctypes.byref(m), fake, ws_bytes, None) == UNSUPPORTED
    # the GEMM self test validates its wait limit before anything else
    assert lib.fp8q_selftest_gemm_wait_limit(0, i64(128), i64(256), i64(128), fake, 0, i64(128), fake, 0, i64(256),
                                             fake, fake, 0, None, None, fake, 1, i64(256), i64(10), None) == INVALID


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of the C structs have the header's sizes and field offsets (compiled with gcc)."""
    import shutil
    import subprocess
    import fp8_absmax_reduce_gb300 as fq
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    fields = {"fp8q_mlp": (fq.FP8QMlp, ["x", "scal", "dN", "recompute", "bf16", "a16", "mx"]),
              "fp8q_mlp_mx": (fq.FP8QMlpMx, ["W_gu_c", "n_r", "dH_c"]),
              "fp8q_block": (fq.FP8QBlock, ["mlp", "dQKV", "n_heads", "seq_len", "n1_16"]),
              "fp8q_mlp_host_io": (fq.FP8QMlpHostIO, ["dY", "dg"])}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "fp8q.h"', "int main(void) {"]
    for st, (_, names) in fields.items():
        lines.append(f'  printf("%zu\\n", sizeof({st}));')
        lines += [f'  printf("%zu\\n", offsetof({st}, {n}));' for n in names]
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    want = []
    for st, (cls, names) in fields.items():
        want.append(ctypes.sizeof(cls))
        want += [getattr(cls, n).offset for n in names]
    assert got == want
