"""CPU oracle for the FP8 per-tensor-absmax block pipeline.

TEST INFRASTRUCTURE ONLY.  Import this from ``tests/``, from
``__graft_entry__.smoke()`` or from the CPU-baseline leg of ``bench.py``;
nothing in the product path may load it.  It shares no code with the CUDA
library (``fp8_absmax_reduce_gb300``); the two meet only through the seeded
inputs from ``synth``.

The arithmetic lives in ``fp8q_oracle.cpp`` (plain C++17, fp64 GEMM
accumulation, software E4M3/E5M2 with round-to-nearest-even and saturation);
this module compiles it with g++ on first use and marshals numpy arrays.

Sources: "LLMQ: Efficient Lower-Precision Pretraining for Consumer GPUs"
(paperlayer.ai summary), §1 (dynamic tensor-level FP8 scaling), §3/§3.1
(fused non-matmul ops, retained absmax statistics), §5 Figure 2 (E4M3
forward, E5M2 activation gradients); "Periodic Reporting for period 1 -
FastML" (CORDIS), "FP8 training without delayed scaling" (just-in-time
absmax scaling, no clipping); LLMQ §2 (inner-dimension block scaling: the MXFP8 mode, in the
OCP Microscaling block format).

Parity pins: ``tests/test_oracle_*.py``.  Every function here is pinned;
see the header of each test file for what pins it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3, E5M2 = 0, 1
NN, NT, TN = 0, 1, 2
FMT_MAX = {E4M3: 448.0, E5M2: 57344.0}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8q_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfp8q_oracle.so")
_CXXFLAGS = ["-O3", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (g++) if missing or stale; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["g++", *_CXXFLAGS, _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _c(arr):
    return arr.ctypes.data_as(ctypes.c_void_p)


class _BlockIO(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64), ("d", ctypes.c_int64), ("f", ctypes.c_int64),
        ("eps", ctypes.c_float), ("exact", ctypes.c_int), ("nthreads", ctypes.c_int), ("grad_fmt", ctypes.c_int),
        ("x", ctypes.c_void_p), ("g", ctypes.c_void_p), ("Wgu", ctypes.c_void_p),
        ("Wd", ctypes.c_void_p), ("dY", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("H", ctypes.c_void_p), ("rstd", ctypes.c_void_p),
        ("Wgu8", ctypes.c_void_p), ("Wd8", ctypes.c_void_p), ("n8", ctypes.c_void_p),
        ("a8", ctypes.c_void_p), ("scal_fwd", ctypes.c_void_p),
        ("dX", ctypes.c_void_p), ("dWgu", ctypes.c_void_p), ("dWd", ctypes.c_void_p),
        ("dg", ctypes.c_void_p), ("dN", ctypes.c_void_p), ("dH", ctypes.c_void_p),
        ("dY8", ctypes.c_void_p), ("dH8", ctypes.c_void_p), ("scal_bwd", ctypes.c_void_p),
        ("bf16", ctypes.c_int), ("n16", ctypes.c_void_p), ("a16", ctypes.c_void_p),
        ("mx", ctypes.c_int), ("mxq", ctypes.c_void_p * 12), ("mxs", ctypes.c_void_p * 12),
    ]


# MX operand slots of the block (the oracle's MxSlot): tensor, then the direction of its blocks --
# "_r" 32 consecutive columns of a row, "_c" 32 consecutive rows of a column.
MX_SLOTS = ("Wgu_r", "Wgu_c", "Wd_r", "Wd_c", "n_r", "n_c", "a_r", "a_c", "dY_r", "dY_c", "dH_r", "dH_c")
MX_BLOCK = 32


class _FullIO(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64), ("d", ctypes.c_int64), ("f", ctypes.c_int64), ("nq", ctypes.c_int64),
        ("eps", ctypes.c_float), ("exact", ctypes.c_int), ("nthreads", ctypes.c_int),
        ("att", ctypes.c_void_p), ("g1", ctypes.c_void_p), ("Wqkv", ctypes.c_void_p), ("Wo", ctypes.c_void_p),
        ("dQKV", ctypes.c_void_p), ("qkv", ctypes.c_void_p), ("h", ctypes.c_void_p), ("rstd1", ctypes.c_void_p),
        ("Wqkv8", ctypes.c_void_p), ("Wo8", ctypes.c_void_p), ("n1_8", ctypes.c_void_p), ("att8", ctypes.c_void_p),
        ("scal_attn", ctypes.c_void_p), ("dX", ctypes.c_void_p), ("dWqkv", ctypes.c_void_p),
        ("dWo", ctypes.c_void_p), ("dg1", ctypes.c_void_p), ("d_att", ctypes.c_void_p), ("dh", ctypes.c_void_p),
        ("dh8", ctypes.c_void_p), ("dqkv8", ctypes.c_void_p), ("mlp", _BlockIO), ("x", ctypes.c_void_p),
        ("n_heads", ctypes.c_int64), ("n_kv_heads", ctypes.c_int64), ("head_dim", ctypes.c_int64),
        ("seq_len", ctypes.c_int64), ("att_out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("dqkv_out", ctypes.c_void_p), ("n1_16", ctypes.c_void_p),
    ]


class _AttnIO(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("S", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
        ("dh", ctypes.c_int64), ("exact", ctypes.c_int), ("nthreads", ctypes.c_int),
        ("qkv", ctypes.c_void_p), ("att", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("d_att", ctypes.c_void_p), ("dqkv", ctypes.c_void_p), ("att_abs", ctypes.c_void_p),
        ("dqkv_abs", ctypes.c_void_p),
    ]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
            L.fo_fp8_encode.restype = ctypes.c_uint8
            L.fo_fp8_encode.argtypes = [f32, ctypes.c_int]
            L.fo_fp8_decode.restype = ctypes.c_double
            L.fo_fp8_decode.argtypes = [ctypes.c_uint8, ctypes.c_int]
            L.fo_fp8_encode_n.argtypes = [vp, i64, ctypes.c_int, vp]
            L.fo_fp8_decode_n.argtypes = [vp, i64, ctypes.c_int, vp]
            L.fo_bf16_round_n.argtypes = [vp, i64, vp]
            L.fo_exp_ref.restype = f32
            L.fo_exp_ref.argtypes = [f32]
            L.fo_exp_ref_n.argtypes = [vp, i64, vp]
            L.fo_pairwise_sum.restype = f32
            L.fo_pairwise_sum.argtypes = [vp, i64]
            L.fo_quantize_absmax.argtypes = [vp, ctypes.c_int, i64, ctypes.c_int, vp, vp]
            L.fo_rmsnorm_quant.argtypes = [vp, vp, i64, i64, f32, vp, vp, vp]
            L.fo_swiglu_quant.argtypes = [vp, i64, i64, ctypes.c_int, vp, vp]
            L.fo_rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, ctypes.c_int, vp, vp]
            L.fo_gemm_scaled.argtypes = [ctypes.c_int, i64, i64, i64, vp, ctypes.c_int, vp,
                                         ctypes.c_int, f32, f32, vp, ctypes.c_int, vp, ctypes.c_int]
            L.fo_block_forward.argtypes = [ctypes.POINTER(_BlockIO)]
            L.fo_block_forward_backward.argtypes = [ctypes.POINTER(_BlockIO)]
            L.fo_full_block.argtypes = [ctypes.POINTER(_FullIO), ctypes.c_int]
            L.fo_mx_quantize.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp]
            L.fo_gemm_mx.argtypes = [ctypes.c_int, i64, i64, i64, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp,
                                     ctypes.c_int, vp, ctypes.c_int]
            L.fo_attention.argtypes = [ctypes.POINTER(_AttnIO), ctypes.c_int]
            _lib = L
    return _lib


# ----------------------------------------------------------------------------
# bf16 helpers (bf16 tensors travel as uint16 bit patterns)
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """One round-to-nearest-even rounding of real values (float64) to bf16 bits."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().fo_bf16_round_n(_c(v), v.size, _c(out))
    return out


# ----------------------------------------------------------------------------
# FP8 codec and exp_ref
# ----------------------------------------------------------------------------
def fp8_encode(v: np.ndarray, fmt: int) -> np.ndarray:
    """fp32 -> FP8 code, round-to-nearest-even, saturating to +-max, NaN -> 0x7F."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().fo_fp8_encode_n(_c(v), v.size, fmt, _c(out))
    return out


def fp8_decode(codes: np.ndarray, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().fo_fp8_decode_n(_c(c), c.size, fmt, _c(out))
    return out


def exp_ref(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.float32)
    lib().fo_exp_ref_n(_c(x), x.size, _c(out))
    return out


def pairwise_sum_f32(v: np.ndarray) -> np.float32:
    v = np.ascontiguousarray(v, dtype=np.float32)
    return np.float32(lib().fo_pairwise_sum(_c(v), v.size))


# ----------------------------------------------------------------------------
# Standalone operations
# ----------------------------------------------------------------------------
def quantize_absmax(x: np.ndarray, fmt: int):
    """Per-tensor absmax quantization.  x: uint16 (bf16 bits) or float32.

    Returns (codes uint8 same shape, scal float32[3] = amax, scale, scale_inv, status).
    """
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        dtype = 0
    elif x.dtype == np.float32:
        dtype = 1
    else:
        raise TypeError("quantize_absmax takes bf16 bits (uint16) or float32")
    q = np.empty(x.shape, dtype=np.uint8)
    scal = np.zeros(3, dtype=np.float32)
    st = lib().fo_quantize_absmax(_c(x), dtype, x.size, fmt, _c(q), _c(scal))
    return q, scal, st


def rmsnorm_quant(x: np.ndarray, g: np.ndarray, eps: float):
    """x [T,d] bf16 bits, g [d] bf16 bits -> (n8 [T,d], scal[3], rstd[T] fp32, status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    g = np.ascontiguousarray(g, dtype=np.uint16)
    T, d = x.shape
    q = np.empty((T, d), dtype=np.uint8)
    scal = np.zeros(3, dtype=np.float32)
    rstd = np.empty(T, dtype=np.float32)
    st = lib().fo_rmsnorm_quant(_c(x), _c(g), T, d, eps, _c(q), _c(scal), _c(rstd))
    return q, scal, rstd, st


def rmsnorm_bwd(dN: np.ndarray, x: np.ndarray, g: np.ndarray, rstd: np.ndarray, dY: np.ndarray,
                exact: bool = False):
    """RMSNorm backward with the residual gradient dY, on values (float64: dN, x, dY [T,d], g [d],
    rstd [T]): dX = dY + rstd (u - nh mean_j(u nh)), u = dN g, nh = x rstd; dg = sum_t dN nh.
    Returns (dX [T,d], dg [d]) as float64: dX rounded to bf16 and dg to fp32 unless exact."""
    dN, x, dY = (np.ascontiguousarray(a, dtype=np.float64) for a in (dN, x, dY))
    g, rstd = np.ascontiguousarray(g, dtype=np.float64), np.ascontiguousarray(rstd, dtype=np.float64)
    T, d = x.shape
    assert dN.shape == (T, d) and dY.shape == (T, d) and g.shape == (d,) and rstd.shape == (T,)
    dX = np.empty((T, d), dtype=np.float64)
    dg = np.empty(d, dtype=np.float64)
    lib().fo_rmsnorm_bwd(_c(dN), _c(x), _c(g), _c(rstd), _c(dY), T, d, int(exact), _c(dX), _c(dg))
    return dX, dg


def swiglu_quant(H: np.ndarray, fmt: int = E4M3):
    """H [T,2f] bf16 bits (gate | up) -> (a8 [T,f], scal[3], status)."""
    H = np.ascontiguousarray(H, dtype=np.uint16)
    T, f2 = H.shape
    f = f2 // 2
    q = np.empty((T, f), dtype=np.uint8)
    scal = np.zeros(3, dtype=np.float32)
    st = lib().fo_swiglu_quant(_c(H), T, f, fmt, _c(q), _c(scal))
    return q, scal, st


def gemm_scaled(layout: int, A: np.ndarray, fmtA: int, B: np.ndarray, fmtB: int,
                sinvA: float, sinvB: float, out: str = "f32", residual=None, nthreads: int = 1):
    """C = fl32(sinvA*sinvB) * op(A) op(B) [+ residual], fp64 accumulation.

    layout NN: A [M,K], B [K,N];  NT: A [M,K], B [N,K];  TN: A [K,M], B [K,N].
    out: "bf16" (uint16 bits), "f32", or "f64" (alpha * acc before output rounding).
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    if layout == TN:
        K, M = A.shape
    else:
        M, K = A.shape
    N = B.shape[0] if layout == NT else B.shape[1]
    kb = B.shape[1] if layout == NT else B.shape[0]
    if kb != K:
        raise ValueError("inner dimensions differ")
    code = {"bf16": 0, "f32": 1, "f64": 2}[out]
    C = np.empty((M, N), dtype={0: np.uint16, 1: np.float32, 2: np.float64}[code])
    res = None
    if residual is not None:
        if code != 0:
            raise ValueError("residual needs bf16 output")
        res = np.ascontiguousarray(residual, dtype=np.uint16)
    lib().fo_gemm_scaled(layout, M, N, K, _c(A), fmtA, _c(B), fmtB, sinvA, sinvB,
                         None if res is None else _c(res), code, _c(C), nthreads)
    return C


def mx_quantize(x: np.ndarray, fmt: int, along_rows: bool):
    """Block-scaled (MXFP8) quantization of a 2-D tensor (bf16 bits as uint16, or float32).

    along_rows=False: blocks of 32 consecutive columns of a row (the contraction runs along the
    columns); scale codes [R, ceil(C/32)].  along_rows=True: blocks of 32 consecutive rows of a
    column; scale codes [ceil(R/32), C].  Scale code = X + 127 (E8M0), X the smallest integer with
    amax_block <= fmax 2^X; element code = fp8(fl32(v 2^-X)).  Returns (codes, scale codes, status).
    """
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        dtype = 0
    elif x.dtype == np.float32:
        dtype = 1
    else:
        raise TypeError("mx_quantize takes bf16 bits (uint16) or float32")
    R, C = x.shape
    q = np.empty((R, C), dtype=np.uint8)
    sf = np.empty(((R + MX_BLOCK - 1) // MX_BLOCK, C) if along_rows else (R, (C + MX_BLOCK - 1) // MX_BLOCK),
                  dtype=np.uint8)
    st = lib().fo_mx_quantize(_c(x), dtype, R, C, fmt, int(along_rows), _c(q), _c(sf))
    return q, sf, st


def gemm_mx(layout: int, A: np.ndarray, fmtA: int, sfA: np.ndarray, B: np.ndarray, fmtB: int, sfB: np.ndarray,
            out: str = "f32", residual=None, nthreads: int = 1):
    """Block-scaled GEMM C = op(A) op(B) [+ residual] in fp64 (layouts as gemm_scaled).

    sfA [M, ceil(K/32)] holds the scale code of row m's K-block, sfB [N, ceil(K/32)] that of column
    n's, whatever the storage layout of A and B; an element is worth decode(code) 2^(sf - 127).
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    if layout == TN:
        K, M = A.shape
    else:
        M, K = A.shape
    N = B.shape[0] if layout == NT else B.shape[1]
    if (B.shape[1] if layout == NT else B.shape[0]) != K:
        raise ValueError("inner dimensions differ")
    KB = (K + MX_BLOCK - 1) // MX_BLOCK
    sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
    sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
    if sfA.shape != (M, KB) or sfB.shape != (N, KB):
        raise ValueError("scale shapes: sfA [M, K/32], sfB [N, K/32]")
    code = {"bf16": 0, "f32": 1, "f64": 2}[out]
    C = np.empty((M, N), dtype={0: np.uint16, 1: np.float32, 2: np.float64}[code])
    res = None
    if residual is not None:
        if code != 0:
            raise ValueError("residual needs bf16 output")
        res = np.ascontiguousarray(residual, dtype=np.uint16)
    lib().fo_gemm_mx(layout, M, N, K, _c(A), fmtA, _c(sfA), _c(B), fmtB, _c(sfB),
                     None if res is None else _c(res), code, _c(C), nthreads)
    return C


# ----------------------------------------------------------------------------
# The MLP block
# ----------------------------------------------------------------------------
def _as_f64(a, exact):
    if exact:
        return np.ascontiguousarray(a, dtype=np.float64)
    return bf16_to_f64(a)


def block(x, g, Wgu, Wd, dY=None, eps: float = 1e-6, exact: bool = False, nthreads: int = 1,
          grad_fmt: int = E5M2, bf16: bool = False, mx: bool = False):
    """MLP block forward (and backward when dY is given).

    Quantized mode (exact=False): x, g, Wgu, Wd, dY are bf16 bit patterns
    (uint16) of shapes [T,d], [d], [d,2f], [f,d], [T,d].  Returned float arrays
    hold the stored values (bf16 tensors as their exact value, fp32 tensors as
    fp32); codes are uint8.  scal_fwd rows: W_gu, W_d, n, a; scal_bwd rows: dY, dH.

    Exact mode (exact=True): float64 inputs, no quantization and no rounding;
    the backward is then the exact gradient of the forward.

    BF16 baseline (bf16=True, bf16 inputs): no quantization; n and a are stored
    as bf16 (returned as "n16", "a16") and every GEMM multiplies the bf16
    operands unscaled; the storage points are those of the FP8 block.

    Block-scaled MXFP8 (mx=True, bf16 inputs): every GEMM operand is quantized in blocks of 32
    along that GEMM's contraction dimension (mx_quantize), no per-tensor scales; the results hold
    "mx_<slot>" (codes) and "mx_<slot>_sf" (E8M0 scale codes) for every slot of MX_SLOTS (the
    backward's dY / dH slots only with dY).
    """
    if (bf16 or mx) and exact:
        raise ValueError("bf16, mx and exact are separate modes")
    if bf16 and mx:
        raise ValueError("bf16 and mx are separate modes")
    x64, g64, Wgu64, Wd64 = (_as_f64(a, exact) for a in (x, g, Wgu, Wd))
    T, d = x64.shape
    f = Wd64.shape[0]
    if Wgu64.shape != (d, 2 * f) or g64.shape != (d,):
        raise ValueError("block shapes: x [T,d], g [d], Wgu [d,2f], Wd [f,d]")
    out = {
        "y": np.empty((T, d)), "H": np.empty((T, 2 * f)), "rstd": np.empty(T),
        "Wgu8": np.empty((d, 2 * f), np.uint8), "Wd8": np.empty((f, d), np.uint8),
        "n8": np.empty((T, d), np.uint8), "a8": np.empty((T, f), np.uint8),
        "scal_fwd": np.zeros((4, 3), np.float32),
    }
    io = _BlockIO(T=T, d=d, f=f, eps=eps, exact=int(exact), nthreads=int(nthreads), grad_fmt=int(grad_fmt),
                  bf16=int(bf16), mx=int(mx))
    keep = [x64, g64, Wgu64, Wd64]
    if mx:
        shapes = {"Wgu": (d, 2 * f), "Wd": (f, d), "n": (T, d), "a": (T, f), "dY": (T, d), "dH": (T, 2 * f)}
        for i, slot in enumerate(MX_SLOTS):
            name, axis = slot.rsplit("_", 1)
            if name in ("dY", "dH") and dY is None:
                continue
            R, C = shapes[name]
            sfs = ((R + MX_BLOCK - 1) // MX_BLOCK, C) if axis == "c" else (R, (C + MX_BLOCK - 1) // MX_BLOCK)
            out["mx_" + slot] = np.empty((R, C), np.uint8)
            out["mx_" + slot + "_sf"] = np.empty(sfs, np.uint8)
            io.mxq[i] = out["mx_" + slot].ctypes.data
            io.mxs[i] = out["mx_" + slot + "_sf"].ctypes.data
    io.x, io.g, io.Wgu, io.Wd = (a.ctypes.data for a in keep)
    if bf16:
        out.update({"n16": np.empty((T, d)), "a16": np.empty((T, f))})
        io.n16, io.a16 = out["n16"].ctypes.data, out["a16"].ctypes.data
    for k in ("y", "H", "rstd", "Wgu8", "Wd8", "n8", "a8", "scal_fwd"):
        setattr(io, k, out[k].ctypes.data)
    if dY is None:
        st = lib().fo_block_forward(ctypes.byref(io))
    else:
        dY64 = _as_f64(dY, exact)
        keep.append(dY64)
        io.dY = dY64.ctypes.data
        out.update({
            "dX": np.empty((T, d)), "dWgu": np.empty((d, 2 * f)), "dWd": np.empty((f, d)),
            "dg": np.empty(d), "dN": np.empty((T, d)), "dH": np.empty((T, 2 * f)),
            "dY8": np.empty((T, d), np.uint8), "dH8": np.empty((T, 2 * f), np.uint8),
            "scal_bwd": np.zeros((2, 3), np.float32),
        })
        for k in ("dX", "dWgu", "dWd", "dg", "dN", "dH", "dY8", "dH8", "scal_bwd"):
            setattr(io, k, out[k].ctypes.data)
        st = lib().fo_block_forward_backward(ctypes.byref(io))
    out["status"] = st
    return out


def attention(qkv, S: int, Hq: int, Hkv: int, dh: int, d_att=None, exact: bool = False, nthreads: int = 1,
              with_abs: bool = False):
    """Causal grouped-query softmax attention (the core between the QKV and O projections).

    qkv [T, (Hq + 2 Hkv) dh] (bf16 bits, or float64 in exact mode) holds B = T / S sequences of S
    consecutive tokens; returns att [T, Hq dh] (bf16 values; exact mode unrounded), lse [Hq, T]
    (natural log of each softmax denominator, relative to no shift), and with d_att [T, Hq dh]
    the input gradient dqkv [T, (Hq + 2 Hkv) dh].  with_abs: also "att_abs" = sum_k P_ik |v_k|, the
    size of the terms of each output (the scale of an error bound for rounded probabilities), and
    with d_att "dqkv_abs", the same for each gradient (see the oracle's AttnIO)."""
    q64 = _as_f64(qkv, exact)
    T, nq = q64.shape
    if T % S or nq != (Hq + 2 * Hkv) * dh or Hq % Hkv:
        raise ValueError("attention shapes")
    out = {"att": np.empty((T, Hq * dh)), "lse": np.empty((Hq, T))}
    io = _AttnIO(B=T // S, S=S, Hq=Hq, Hkv=Hkv, dh=dh, exact=int(exact), nthreads=int(nthreads))
    keep = [q64]
    io.qkv = q64.ctypes.data
    io.att, io.lse = out["att"].ctypes.data, out["lse"].ctypes.data
    if with_abs:
        out["att_abs"] = np.empty((T, Hq * dh))
        io.att_abs = out["att_abs"].ctypes.data
    if d_att is not None:
        da64 = _as_f64(d_att, exact)
        keep.append(da64)
        out["dqkv"] = np.empty((T, nq))
        io.d_att, io.dqkv = da64.ctypes.data, out["dqkv"].ctypes.data
        if with_abs:
            out["dqkv_abs"] = np.empty((T, nq))
            io.dqkv_abs = out["dqkv_abs"].ctypes.data
    st = lib().fo_attention(ctypes.byref(io), int(d_att is not None))
    if st:
        raise ValueError(f"fo_attention status {st}")
    return out


def full_block(x, g1, Wqkv, Wo, att, g2, Wgu, Wd, dY=None, dQKV=None, eps: float = 1e-6, exact: bool = False,
               nthreads: int = 1, grad_fmt: int = E5M2, core=None, bf16: bool = False):
    """The full transformer block's matmuls around a given attention core.

    core = (n_heads, n_kv_heads, head_dim, seq_len): the attention core (attention()) computes att
    from qkv and, in the backward, dQKV from d_att; att and dQKV are then not read (may be None)
    and the results hold "att", "lse" and "dqkv" as well.  bf16: the BF16 baseline (every operand
    stored as bf16 instead of quantized, see block()); the results then hold "n1_16", "n16", "a16".

    Forward: qkv = bf16(alpha n1_8 @ W_qkv8) with n1 = RMSNorm(x) g1; h = bf16(x + alpha att8 @ W_o8);
    y = MLP block on h (gain g2).  Backward (with dY [T,d] and the core's input gradient dQKV
    [T,nq]): dh from the MLP; d_att = bf16(alpha dh8 @ W_o8^T); dW_o; dW_qkv; dX = bf16(dh +
    RMSNorm'(alpha dQKV8 @ W_qkv8^T)); dg1.  Returned keys: the attention-side tensors plus every
    key of block() for the MLP part; scal_attn rows: W_qkv, W_o, n1, att, dh, dQKV.
    Inputs are bf16 bit patterns (quantized mode) or float64 (exact mode)."""
    x64, g164, Wqkv64, Wo64 = (_as_f64(a, exact) for a in (x, g1, Wqkv, Wo))
    att64 = _as_f64(att, exact) if att is not None else np.zeros(x64.shape)
    g264, Wgu64, Wd64 = (_as_f64(a, exact) for a in (g2, Wgu, Wd))
    T, d = x64.shape
    nq = Wqkv64.shape[1]
    f = Wd64.shape[0]
    backward = dY is not None
    out = {
        "qkv": np.empty((T, nq)), "h": np.empty((T, d)), "rstd1": np.empty(T),
        "Wqkv8": np.empty((d, nq), np.uint8), "Wo8": np.empty((d, d), np.uint8),
        "n1_8": np.empty((T, d), np.uint8), "att8": np.empty((T, d), np.uint8),
        "scal_attn": np.zeros((6, 3), np.float32),
        "y": np.empty((T, d)), "H": np.empty((T, 2 * f)), "rstd": np.empty(T),
        "Wgu8": np.empty((d, 2 * f), np.uint8), "Wd8": np.empty((f, d), np.uint8),
        "n8": np.empty((T, d), np.uint8), "a8": np.empty((T, f), np.uint8),
        "scal_fwd": np.zeros((4, 3), np.float32),
    }
    keep = [x64, g164, Wqkv64, Wo64, att64, g264, Wgu64, Wd64]
    io = _FullIO(T=T, d=d, f=f, nq=nq, eps=eps, exact=int(exact), nthreads=int(nthreads))
    io.x, io.g1, io.Wqkv, io.Wo, io.att = (a.ctypes.data for a in keep[:5])
    if core is not None:
        io.n_heads, io.n_kv_heads, io.head_dim, io.seq_len = (int(v) for v in core)
        out.update({"att": np.empty((T, d)), "lse": np.empty((io.n_heads, T))})
        io.att_out, io.lse = out["att"].ctypes.data, out["lse"].ctypes.data
    m = _BlockIO(T=T, d=d, f=f, eps=eps, exact=int(exact), nthreads=int(nthreads), grad_fmt=int(grad_fmt),
                 bf16=int(bf16))
    m.g, m.Wgu, m.Wd = (a.ctypes.data for a in keep[5:])
    if bf16:
        out.update({"n1_16": np.empty((T, d)), "n16": np.empty((T, d)), "a16": np.empty((T, f))})
        io.n1_16 = out["n1_16"].ctypes.data
        m.n16, m.a16 = out["n16"].ctypes.data, out["a16"].ctypes.data
    for k in ("qkv", "h", "rstd1", "Wqkv8", "Wo8", "n1_8", "att8", "scal_attn"):
        setattr(io, k, out[k].ctypes.data)
    for k in ("y", "H", "rstd", "Wgu8", "Wd8", "n8", "a8", "scal_fwd"):
        setattr(m, k, out[k].ctypes.data)
    if backward:
        dY64 = _as_f64(dY, exact)
        dQKV64 = _as_f64(dQKV, exact) if dQKV is not None else np.zeros((T, nq))
        keep += [dY64, dQKV64]
        m.dY = dY64.ctypes.data
        io.dQKV = dQKV64.ctypes.data
        if core is not None:
            out["dqkv"] = np.empty((T, nq))
            io.dqkv_out = out["dqkv"].ctypes.data
        out.update({
            "dX": np.empty((T, d)), "dWqkv": np.empty((d, nq)), "dWo": np.empty((d, d)), "dg1": np.empty(d),
            "d_att": np.empty((T, d)), "dh": np.empty((T, d)), "dh8": np.empty((T, d), np.uint8),
            "dqkv8": np.empty((T, nq), np.uint8),
            "dWgu": np.empty((d, 2 * f)), "dWd": np.empty((f, d)), "dg": np.empty(d), "dN": np.empty((T, d)),
            "dH": np.empty((T, 2 * f)), "dY8": np.empty((T, d), np.uint8), "dH8": np.empty((T, 2 * f), np.uint8),
            "scal_bwd": np.zeros((2, 3), np.float32),
        })
        for k in ("dX", "dWqkv", "dWo", "dg1", "d_att", "dh", "dh8", "dqkv8"):
            setattr(io, k, out[k].ctypes.data)
        for k in ("dWgu", "dWd", "dg", "dN", "dH", "dY8", "dH8", "scal_bwd"):
            setattr(m, k, out[k].ctypes.data)
    io.mlp = m
    out["status"] = lib().fo_full_block(ctypes.byref(io), int(backward))
    if out["status"] & 2:
        raise ValueError("full_block: inconsistent attention core shapes")
    return out
