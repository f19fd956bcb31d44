"""GB300 (sm_103a) FP8 transformer-block pipeline with just-in-time per-tensor absmax scaling.

Thin Python binding of the C-ABI library ``libfp8q.so`` (``include/fp8q.h``).
Every function here only marshals torch tensors (device memory, the current
stream) into the C calls; all arithmetic runs in the library's CUDA kernels.
There is no CPU fallback: without the built library, the first call raises.

Build the library with ``python -m fp8_absmax_reduce_gb300.build``.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

from . import build as _build_mod

E4M3, E5M2 = 0, 1
BF16, F32 = 0, 1
NN, NT, TN = 0, 1, 2
STATUS_NONFINITE, STATUS_TIMEOUT = 0x1, 0x2

_LIB_PATH = _build_mod.LIB


class Fp8qError(RuntimeError):
    pass


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libfp8q.so is not built ({_LIB_PATH}); run python -m fp8_absmax_reduce_gb300.build")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, f32, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
    L.fp8_quantize_absmax_workspace_size.restype = sz
    L.fp8_quantize_absmax_workspace_size.argtypes = [i64]
    L.fp8_quantize_absmax.argtypes = [vp, i32, i64, i32, vp, vp, vp, sz, vp]
    L.fp8_gemm_scaled.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, i32, i64, vp, vp, vp, i32, i64, vp, i64, vp]
    L.rmsnorm_quant_workspace_size.restype = sz
    L.rmsnorm_quant_workspace_size.argtypes = [i64, i64]
    L.rmsnorm_quant.argtypes = [vp, vp, i64, i64, f32, vp, vp, vp, vp, sz, vp]
    L.rmsnorm_bwd_workspace_size.restype = sz
    L.rmsnorm_bwd_workspace_size.argtypes = [i64, i64]
    L.rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, sz, vp]
    L.fp8q_selftest_rmsnorm_bwd_wait_limit.argtypes = [vp, vp, vp, vp, vp, i64, i64, vp, vp, vp, sz, i64, vp]
    L.swiglu_quant_workspace_size.restype = sz
    L.swiglu_quant_workspace_size.argtypes = [i64, i64]
    L.swiglu_quant.argtypes = [vp, i64, i64, i32, vp, vp, vp, sz, vp]
    L.mlp_block_workspace_size.restype = sz
    L.mlp_block_workspace_size.argtypes = [i64, i64, i64, i32]
    L.mlp_block_fwd.argtypes = [ctypes.POINTER(FP8QMlp), vp, sz, vp]
    L.mx_scale_bytes.restype = sz
    L.mx_scale_bytes.argtypes = [i64, i64]
    L.mx_quantize.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp, vp, vp]
    L.fp8_gemm_mx.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, vp, i32, i64, vp, vp, i32, i64, vp, i64, vp]
    L.attention_fwd.argtypes = [vp, i64, i64, i32, i32, i32, vp, vp, vp]
    L.attention_bwd_workspace_size.restype = sz
    L.attention_bwd_workspace_size.argtypes = [i64, i32]
    L.attention_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32, vp, vp, sz, vp]
    L.mlp_block_bwd.argtypes = [ctypes.POINTER(FP8QMlp), vp, sz, vp]
    L.mlp_block_run_steps.argtypes = [ctypes.POINTER(FP8QMlp), ctypes.POINTER(FP8QMlp), ctypes.POINTER(FP8QMlpHostIO),
                                      i32, vp, sz, vp]
    L.mlp_block_fwd_run_steps.argtypes = L.mlp_block_run_steps.argtypes
    L.fp8q_get_status.argtypes = [i32]
    L.fp8q_status_string.restype = ctypes.c_char_p
    L.fp8q_status_string.argtypes = [i32]
    L.fp8q_last_launch_count.restype = i32
    L.block_workspace_size.restype = sz
    L.block_workspace_size.argtypes = [i64, i64, i64, i64, i32]
    L.block_fwd.argtypes = [ctypes.POINTER(FP8QBlock), vp, sz, vp]
    L.block_bwd.argtypes = [ctypes.POINTER(FP8QBlock), vp, sz, vp]
    L.block_run_steps.argtypes = [ctypes.POINTER(FP8QBlock), ctypes.POINTER(FP8QBlock),
                                  ctypes.POINTER(FP8QBlockHostIO), i32, i32, vp, sz, vp]
    L.fp8q_selftest_bounded_wait.argtypes = [i64, vp]
    L.fp8q_selftest_gemm_wait_limit.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, i32, i64, vp, vp, i32, vp, vp,
                                                vp, i32, i64, i64, vp]
    L.fp8q_trace_start.argtypes = [i32]
    L.fp8q_trace_read.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), i32]
    L.fp8q_kernel_name.restype = ctypes.c_char_p
    L.fp8q_kernel_name.argtypes = [i32]
    return L


_MLP_PTRS = ("x", "g", "W_gu", "W_d", "y", "W_gu8", "W_d8", "n8", "rstd", "H", "a8", "scal",
             "dY", "dX", "dW_gu", "dW_d", "dg", "dY8", "dH", "dH8", "dN")


class FP8QMlp(ctypes.Structure):
    """Mirror of ``fp8q_mlp`` in include/fp8q.h."""
    _fields_ = ([("T", ctypes.c_int64), ("d", ctypes.c_int64), ("f", ctypes.c_int64), ("eps", ctypes.c_float)]
                + [(name, ctypes.c_void_p) for name in _MLP_PTRS]
                + [("recompute", ctypes.c_int), ("grad_e4m3", ctypes.c_int), ("bf16", ctypes.c_int),
                   ("n16", ctypes.c_void_p), ("a16", ctypes.c_void_p), ("mx", ctypes.c_void_p)])


class FP8QMxTensor(ctypes.Structure):
    """Mirror of ``fp8q_mx_tensor``: codes and chunked E8M0 scales."""
    _fields_ = [("q", ctypes.c_void_p), ("sf", ctypes.c_void_p)]


# The block-scaled operands of the MXFP8 block, in the order of fp8q_mlp_mx.
MX_SLOTS = ("W_gu_r", "W_gu_c", "W_d_r", "W_d_c", "n_r", "n_c", "a_r", "a_c", "dY_r", "dY_c", "dH_r", "dH_c")


class FP8QMlpMx(ctypes.Structure):
    """Mirror of ``fp8q_mlp_mx`` in include/fp8q.h."""
    _fields_ = [(n, FP8QMxTensor) for n in MX_SLOTS]


class FP8QMlpHostIO(ctypes.Structure):
    """Mirror of ``fp8q_mlp_host_io`` in include/fp8q.h."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "g", "W_gu", "W_d", "dY", "y", "dX", "dW_gu", "dW_d", "dg")]


class FP8QBlockHostIO(ctypes.Structure):
    """Mirror of ``fp8q_block_host_io`` in include/fp8q.h."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "g1", "W_qkv", "W_o", "att", "g", "W_gu", "W_d", "dY", "dQKV",
                                               "y", "dX", "d_att", "dW_qkv", "dW_o", "dg1", "dW_gu", "dW_d", "dg")]


class FP8QBlock(ctypes.Structure):
    """Mirror of ``fp8q_block`` in include/fp8q.h."""
    _fields_ = ([("T", ctypes.c_int64), ("d", ctypes.c_int64), ("f", ctypes.c_int64), ("n_qkv", ctypes.c_int64),
                 ("eps", ctypes.c_float)]
                + [(n, ctypes.c_void_p) for n in ("x", "g1", "W_qkv", "W_o", "att", "qkv", "h", "W_qkv8", "W_o8",
                                                  "n1_8", "rstd1", "att8", "scal")]
                + [("mlp", FP8QMlp)]
                + [(n, ctypes.c_void_p) for n in ("dQKV", "d_att", "dX", "dW_qkv", "dW_o", "dg1", "dh8", "dQKV8",
                                                  "dN1")]
                + [("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("seq_len", ctypes.c_int64),
                   ("lse", ctypes.c_void_p), ("n1_16", ctypes.c_void_p)])


_lib_handle = None


def load_library() -> ctypes.CDLL:
    """Load libfp8q.so (once).  Raises ImportError when it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load()
    return _lib_handle


class _LazyLib:
    def __getattr__(self, name):
        return getattr(load_library(), name)


lib = _LazyLib()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(name: str, rc: int):
    if rc != 0:
        raise Fp8qError(f"{name}: {lib.fp8q_status_string(rc).decode()} (status {rc})")


def _ws(nbytes: int, device, ws=None):
    if nbytes == 0:
        return None
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t: torch.Tensor):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return t.device


# ---------------------------------------------------------------------------
def fp8_quantize_absmax(x: torch.Tensor, fmt: int = E4M3, q=None, scal=None, ws=None, stream=None):
    """Per-tensor absmax quantization. Returns (codes uint8 like x, scal float32[3] = amax, scale, scale_inv)."""
    dev = _dev(x)
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev) if q is None else q
    scal = torch.empty(3, dtype=torch.float32, device=dev) if scal is None else scal
    nb = lib.fp8_quantize_absmax_workspace_size(x.numel())
    w = _ws(nb, dev, ws)
    _check("fp8_quantize_absmax", lib.fp8_quantize_absmax(_ptr(x), _dtype_code(x), x.numel(), fmt, _ptr(q),
                                                          _ptr(scal), _ptr(w), nb, _stream(stream)))
    return q, scal


def fp8_gemm_scaled(layout: int, A: torch.Tensor, fmtA: int, B: torch.Tensor, fmtB: int, sinvA: torch.Tensor,
                    sinvB: torch.Tensor, out_dtype=torch.bfloat16, residual=None, C=None, stream=None):
    """C = (sinvA*sinvB) op(A) op(B) (+ residual).  NN: A [M,K], B [K,N]; NT: A [M,K], B [N,K];
    TN: A [K,M], B [K,N].  sinvA/sinvB: one-element float32 device tensors (a scal[2:3] slice)."""
    dev = _dev(A)
    _dev(B)
    if layout == TN:
        K, M = A.shape
    else:
        M, K = A.shape
    N = B.shape[0] if layout == NT else B.shape[1]
    lda, ldb = A.shape[1], B.shape[1]
    out_code = {torch.bfloat16: BF16, torch.float32: F32}[out_dtype]
    C = torch.empty((M, N), dtype=out_dtype, device=dev) if C is None else C
    ldr = residual.shape[1] if residual is not None else 0
    _check("fp8_gemm_scaled", lib.fp8_gemm_scaled(layout, M, N, K, _ptr(A), fmtA, lda, _ptr(B), fmtB, ldb,
                                                  _ptr(sinvA), _ptr(sinvB), _ptr(C), out_code, C.shape[1],
                                                  _ptr(residual), ldr, _stream(stream)))
    return C


def mx_scale_bytes(rows: int, K: int) -> int:
    """Bytes of the chunked E8M0 scales of an operand with `rows` rows and contraction length K."""
    return lib.mx_scale_bytes(rows, K)


def mx_quantize(x: torch.Tensor, fmt: int = E4M3, rows: bool = True, cols: bool = True, stream=None):
    """Block-scaled (MXFP8) quantization of x [R, C] (bf16 or fp32; R, C multiples of 128).
    Returns ((q_r, sf_r) or None, (q_c, sf_c) or None): blocks of 32 along each row (the operand of a
    GEMM contracting over C) and down each column (contracting over R), scales in the chunked layout."""
    dev = _dev(x)
    R, C = x.shape
    r = (torch.empty((R, C), dtype=torch.uint8, device=dev),
         torch.empty(mx_scale_bytes(R, C), dtype=torch.uint8, device=dev)) if rows else None
    c = (torch.empty((R, C), dtype=torch.uint8, device=dev),
         torch.empty(mx_scale_bytes(C, R), dtype=torch.uint8, device=dev)) if cols else None
    _check("mx_quantize", lib.mx_quantize(_ptr(x), _dtype_code(x), R, C, fmt, _ptr(r[0]) if r else None,
                                          _ptr(r[1]) if r else None, _ptr(c[0]) if c else None,
                                          _ptr(c[1]) if c else None, _stream(stream)))
    return r, c


def fp8_gemm_mx(layout: int, A: torch.Tensor, fmtA: int, sfA: torch.Tensor, B: torch.Tensor, fmtB: int,
                sfB: torch.Tensor, out_dtype=torch.bfloat16, residual=None, C=None, stream=None):
    """Block-scaled GEMM C = op(A) op(B) (+ residual); layouts as fp8_gemm_scaled, sfA / sfB the
    operands' chunked scales (see fp8_gemm_mx in include/fp8q.h); K a multiple of 128."""
    dev = _dev(A)
    _dev(B)
    if layout == TN:
        K, M = A.shape
    else:
        M, K = A.shape
    N = B.shape[0] if layout == NT else B.shape[1]
    out_code = {torch.bfloat16: BF16, torch.float32: F32}[out_dtype]
    C = torch.empty((M, N), dtype=out_dtype, device=dev) if C is None else C
    ldr = residual.shape[1] if residual is not None else 0
    _check("fp8_gemm_mx", lib.fp8_gemm_mx(layout, M, N, K, _ptr(A), fmtA, A.shape[1], _ptr(sfA), _ptr(B), fmtB,
                                          B.shape[1], _ptr(sfB), _ptr(C), out_code, C.shape[1], _ptr(residual), ldr,
                                          _stream(stream)))
    return C


def rmsnorm_quant(x: torch.Tensor, g: torch.Tensor, eps: float = 1e-6, q=None, scal=None, rstd=None, ws=None,
                  stream=None):
    """RMSNorm + E4M3 quantization. Returns (codes [T,d], scal[3], rstd[T])."""
    dev = _dev(x)
    T, d = x.shape
    q = torch.empty((T, d), dtype=torch.uint8, device=dev) if q is None else q
    scal = torch.empty(3, dtype=torch.float32, device=dev) if scal is None else scal
    rstd = torch.empty(T, dtype=torch.float32, device=dev) if rstd is None else rstd
    nb = lib.rmsnorm_quant_workspace_size(T, d)
    w = _ws(nb, dev, ws)
    _check("rmsnorm_quant", lib.rmsnorm_quant(_ptr(x), _ptr(g), T, d, eps, _ptr(q), _ptr(scal), _ptr(rstd),
                                              _ptr(w), nb, _stream(stream)))
    return q, scal, rstd


def _rmsnorm_bwd_call(name, dN, x, dY, g, rstd, dX, dg, ws, stream, *limit):
    dev = _dev(x)
    T, d = x.shape
    dX = torch.empty((T, d), dtype=torch.bfloat16, device=dev) if dX is None else dX
    dg = torch.empty(d, dtype=torch.float32, device=dev) if dg is None else dg
    nb = lib.rmsnorm_bwd_workspace_size(T, d)
    w = _ws(nb, dev, ws)
    _check(name, getattr(lib, name)(_ptr(dN), _ptr(x), _ptr(dY), _ptr(g), _ptr(rstd), T, d, _ptr(dX), _ptr(dg),
                                    _ptr(w), nb, *limit, _stream(stream)))
    return dX, dg


def rmsnorm_bwd(dN: torch.Tensor, x: torch.Tensor, dY: torch.Tensor, g: torch.Tensor, rstd: torch.Tensor, dX=None,
                dg=None, ws=None, stream=None):
    """RMSNorm backward with the residual gradient: dN [T,d] fp32, x, dY [T,d] bf16, g [d] bf16,
    rstd [T] fp32 -> (dX [T,d] bf16, dg [d] fp32)."""
    return _rmsnorm_bwd_call("rmsnorm_bwd", dN, x, dY, g, rstd, dX, dg, ws, stream)


def selftest_rmsnorm_bwd_wait_limit(dN, x, dY, g, rstd, limit_s: float, dX=None, dg=None, ws=None, stream=None):
    """rmsnorm_bwd with every wait on a row's copies limited to limit_s
    (fp8q_selftest_rmsnorm_bwd_wait_limit in include/fp8q.h).  Returns (dX, dg), incomplete on a time-out."""
    return _rmsnorm_bwd_call("fp8q_selftest_rmsnorm_bwd_wait_limit", dN, x, dY, g, rstd, dX, dg, ws, stream,
                             max(1, int(limit_s * 1e9)))


def swiglu_quant(H: torch.Tensor, fmt: int = E4M3, q=None, scal=None, ws=None, stream=None):
    """SwiGLU of H [T,2f] (gate | up) + per-tensor quantization. Returns (codes [T,f], scal[3])."""
    dev = _dev(H)
    T, f2 = H.shape
    f = f2 // 2
    q = torch.empty((T, f), dtype=torch.uint8, device=dev) if q is None else q
    scal = torch.empty(3, dtype=torch.float32, device=dev) if scal is None else scal
    nb = lib.swiglu_quant_workspace_size(T, f)
    w = _ws(nb, dev, ws)
    _check("swiglu_quant", lib.swiglu_quant(_ptr(H), T, f, fmt, _ptr(q), _ptr(scal), _ptr(w), nb, _stream(stream)))
    return q, scal


def attention_fwd(qkv: torch.Tensor, seq_len: int, n_heads: int, n_kv_heads: int, att=None, lse=None,
                  stream=None):
    """Causal grouped-query attention of qkv [T, (n_heads + 2 n_kv_heads) 128] (bf16).
    Returns (att [T, n_heads 128] bf16, lse [n_heads, T] fp32)."""
    dev = _dev(qkv)
    T = qkv.shape[0]
    att = torch.empty((T, n_heads * 128), dtype=torch.bfloat16, device=dev) if att is None else att
    lse = torch.empty((n_heads, T), dtype=torch.float32, device=dev) if lse is None else lse
    _check("attention_fwd", lib.attention_fwd(_ptr(qkv), T, seq_len, n_heads, n_kv_heads, 128, _ptr(att), _ptr(lse),
                                              _stream(stream)))
    return att, lse


def attention_bwd(qkv: torch.Tensor, att: torch.Tensor, lse: torch.Tensor, d_att: torch.Tensor, seq_len: int,
                  n_heads: int, n_kv_heads: int, dqkv=None, ws=None, stream=None):
    """Input gradient dqkv [T, (n_heads + 2 n_kv_heads) 128] (bf16) of attention_fwd for d_att."""
    dev = _dev(qkv)
    T = qkv.shape[0]
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    nb = lib.attention_bwd_workspace_size(T, n_heads)
    w = _ws(nb, dev, ws)
    _check("attention_bwd", lib.attention_bwd(_ptr(qkv), _ptr(att), _ptr(lse), _ptr(d_att), T, seq_len, n_heads,
                                              n_kv_heads, 128, _ptr(dqkv), _ptr(w), nb, _stream(stream)))
    return dqkv


# ---------------------------------------------------------------------------
@dataclasses.dataclass
class MlpBuffers:
    """Caller-owned device buffers of one MLP block (see fp8q_mlp in include/fp8q.h)."""
    T: int
    d: int
    f: int
    eps: float
    x: torch.Tensor
    g: torch.Tensor
    W_gu: torch.Tensor
    W_d: torch.Tensor
    y: torch.Tensor
    W_gu8: torch.Tensor | None
    W_d8: torch.Tensor | None
    n8: torch.Tensor | None
    rstd: torch.Tensor
    H: torch.Tensor
    a8: torch.Tensor | None
    scal: torch.Tensor | None
    dY: torch.Tensor | None = None
    dX: torch.Tensor | None = None
    dW_gu: torch.Tensor | None = None
    dW_d: torch.Tensor | None = None
    dg: torch.Tensor | None = None
    dY8: torch.Tensor | None = None
    dH: torch.Tensor | None = None
    dH8: torch.Tensor | None = None
    dN: torch.Tensor | None = None
    ws: torch.Tensor | None = None
    recompute: bool = False
    grad_e4m3: bool = False
    bf16: bool = False
    n16: torch.Tensor | None = None
    a16: torch.Tensor | None = None
    mx: dict | None = None  # MXFP8 block: slot name -> (codes, chunked scales), see MX_SLOTS
    _mx_struct: FP8QMlpMx | None = None

    @staticmethod
    def allocate(T: int, d: int, f: int, device="cuda", backward: bool = True, eps: float = 1e-6,
                 keep_intermediates: bool = False, bf16: bool = False, mx: bool = False) -> "MlpBuffers":
        """bf16=True: buffers of the BF16 baseline (n16, a16 instead of the FP8 codes and scales).
        mx=True: the block-scaled MXFP8 block (the codes and scales of every slot of MX_SLOTS)."""
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        q8 = (lambda shape: None) if (bf16 or mx) else (lambda shape: e(shape, torch.uint8))
        b = MlpBuffers(
            T=T, d=d, f=f, eps=eps,
            x=e((T, d), torch.bfloat16), g=e((d,), torch.bfloat16), W_gu=e((d, 2 * f), torch.bfloat16),
            W_d=e((f, d), torch.bfloat16), y=e((T, d), torch.bfloat16), W_gu8=q8((d, 2 * f)),
            W_d8=q8((f, d)), n8=q8((T, d)), rstd=e((T,), torch.float32),
            H=e((T, 2 * f), torch.bfloat16), a8=q8((T, f)),
            scal=None if (bf16 or mx) else torch.zeros((6, 3), device=device), bf16=bf16)
        if mx:
            shape = {"W_gu": (d, 2 * f), "W_d": (f, d), "n": (T, d), "a": (T, f), "dY": (T, d), "dH": (T, 2 * f)}
            b.mx = {}
            for slot in MX_SLOTS:
                name, ax = slot.rsplit("_", 1)
                if name in ("dY", "dH") and not backward:
                    continue
                R, C = shape[name]
                b.mx[slot] = (e((R, C), torch.uint8),
                              e((mx_scale_bytes(R, C) if ax == "r" else mx_scale_bytes(C, R),), torch.uint8))
        if bf16:
            b.n16 = e((T, d), torch.bfloat16)
            b.a16 = e((T, f), torch.bfloat16)
        if backward:
            b.dY = e((T, d), torch.bfloat16)
            b.dX = e((T, d), torch.bfloat16)
            b.dW_gu = e((d, 2 * f), torch.float32)
            b.dW_d = e((f, d), torch.float32)
            b.dg = e((d,), torch.float32)
            if keep_intermediates:
                b.dY8 = None if mx else q8((T, d))
                b.dH = e((T, 2 * f), torch.bfloat16)
                b.dH8 = None if mx else q8((T, 2 * f))
                b.dN = e((T, d), torch.float32)
        nb = lib.mlp_block_workspace_size(T, d, f, int(backward))
        b.ws = torch.empty(nb, dtype=torch.uint8, device=device)
        return b

    def struct(self) -> FP8QMlp:
        s = FP8QMlp(T=self.T, d=self.d, f=self.f, eps=self.eps, recompute=int(self.recompute),
                    grad_e4m3=int(self.grad_e4m3), bf16=int(self.bf16))
        for name in _MLP_PTRS + ("n16", "a16"):
            t = getattr(self, name)
            setattr(s, name, None if t is None else t.data_ptr())
        if self.mx is not None:
            if self._mx_struct is None:
                m = FP8QMlpMx()
                for slot, (q, sf) in self.mx.items():
                    setattr(m, slot, FP8QMxTensor(q.data_ptr(), sf.data_ptr()))
                self._mx_struct = m
            s.mx = ctypes.addressof(self._mx_struct)
        return s


def mlp_block_fwd(b: MlpBuffers, stream=None):
    s = b.struct()
    _check("mlp_block_fwd", lib.mlp_block_fwd(ctypes.byref(s), _ptr(b.ws), b.ws.numel(), _stream(stream)))


def mlp_block_bwd(b: MlpBuffers, stream=None):
    s = b.struct()
    _check("mlp_block_bwd", lib.mlp_block_bwd(ctypes.byref(s), _ptr(b.ws), b.ws.numel(), _stream(stream)))


def mlp_block_run_steps(b0: MlpBuffers, b1: MlpBuffers, host: list, stream=None):
    """Pipelined training steps from and to host memory (mlp_block_run_steps in include/fp8q.h).
    host: one dict per step with CPU tensors x, g, W_gu, W_d, dY (inputs) and y, dX, dW_gu, dW_d,
    dg (outputs), ideally pinned; a missing (or None) entry stays on the device in that step.
    Device sets b0, b1 alternate; b0's workspace is used."""
    _check("mlp_block_run_steps", lib.mlp_block_run_steps(*_steps_args(b0, b1, host, FP8QMlpHostIO), _ptr(b0.ws),
                                                          b0.ws.numel(), _stream(stream)))


def mlp_block_fwd_run_steps(b0: MlpBuffers, b1: MlpBuffers, host: list, stream=None):
    """Pipelined forward-only steps from and to host memory (mlp_block_fwd_run_steps in
    include/fp8q.h): x, g, W_gu, W_d in, y out; entries that are missing stay on the device."""
    _check("mlp_block_fwd_run_steps", lib.mlp_block_fwd_run_steps(*_steps_args(b0, b1, host, FP8QMlpHostIO),
                                                                  _ptr(b0.ws), b0.ws.numel(), _stream(stream)))


def _steps_args(b0, b1, host, io_type):
    """(set 0, set 1, host array, step count) for the pipelined executors; a host dict's missing or
    None entries become null pointers (the tensor stays on the device)."""
    n = len(host)
    arr = (io_type * n)()
    for i, h in enumerate(host):
        for name, _ in io_type._fields_:
            t = h.get(name)
            setattr(arr[i], name, t.data_ptr() if t is not None else None)
    s0, s1 = b0.struct(), b1.struct()
    # (each byref keeps its struct alive for the call)
    return ctypes.byref(s0), ctypes.byref(s1), arr, n


def get_status(clear: bool = False) -> int:
    """Device status bits (STATUS_NONFINITE, STATUS_TIMEOUT); synchronize the stream first."""
    v = lib.fp8q_get_status(int(clear))
    if v < 0:
        raise Fp8qError("fp8q_get_status failed")
    return v


def last_launch_count() -> int:
    return lib.fp8q_last_launch_count()


# ---------------------------------------------------------------------------
@dataclasses.dataclass
class BlockBuffers:
    """Caller-owned device buffers of the full block (see fp8q_block in include/fp8q.h).
    ``mlp`` holds the MLP sub-block's buffers; its ``x`` is the attention residual output h and,
    in the backward, its ``dX`` receives dh."""
    T: int
    d: int
    f: int
    n_qkv: int
    eps: float
    x: torch.Tensor
    g1: torch.Tensor
    W_qkv: torch.Tensor
    W_o: torch.Tensor
    att: torch.Tensor
    qkv: torch.Tensor
    W_qkv8: torch.Tensor
    W_o8: torch.Tensor
    n1_8: torch.Tensor
    rstd1: torch.Tensor
    att8: torch.Tensor
    scal: torch.Tensor
    mlp: MlpBuffers
    dQKV: torch.Tensor | None = None
    d_att: torch.Tensor | None = None
    dX: torch.Tensor | None = None
    dW_qkv: torch.Tensor | None = None
    dW_o: torch.Tensor | None = None
    dg1: torch.Tensor | None = None
    dh8: torch.Tensor | None = None
    dQKV8: torch.Tensor | None = None
    dN1: torch.Tensor | None = None
    ws: torch.Tensor | None = None
    n_heads: int = 0
    n_kv_heads: int = 0
    seq_len: int = 0
    lse: torch.Tensor | None = None
    n1_16: torch.Tensor | None = None

    @staticmethod
    def allocate(T: int, d: int, f: int, n_qkv: int, device="cuda", backward: bool = True, eps: float = 1e-6,
                 keep_intermediates: bool = False, core=None, bf16: bool = False) -> "BlockBuffers":
        """core = (n_heads, n_kv_heads, seq_len): the attention core runs inside the block (att and
        dQKV become outputs); None: att and dQKV are given.  bf16: the BF16 baseline's buffers."""
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        q8 = (lambda shape: None) if bf16 else (lambda shape: e(shape, torch.uint8))
        m = MlpBuffers.allocate(T, d, f, device=device, backward=backward, eps=eps,
                                keep_intermediates=keep_intermediates, bf16=bf16)
        m.ws = None  # the block's workspace holds the MLP's
        b = BlockBuffers(
            T=T, d=d, f=f, n_qkv=n_qkv, eps=eps, x=e((T, d), torch.bfloat16), g1=e((d,), torch.bfloat16),
            W_qkv=e((d, n_qkv), torch.bfloat16), W_o=e((d, d), torch.bfloat16), att=e((T, d), torch.bfloat16),
            qkv=e((T, n_qkv), torch.bfloat16), W_qkv8=q8((d, n_qkv)), W_o8=q8((d, d)),
            n1_8=q8((T, d)), rstd1=e((T,), torch.float32), att8=q8((T, d)),
            scal=None if bf16 else torch.zeros((6, 3), device=device), mlp=m)
        if bf16:
            b.n1_16 = e((T, d), torch.bfloat16)
        if backward:
            b.dQKV = e((T, n_qkv), torch.bfloat16)
            b.d_att = e((T, d), torch.bfloat16)
            b.dX = e((T, d), torch.bfloat16)
            b.dW_qkv = e((d, n_qkv), torch.float32)
            b.dW_o = e((d, d), torch.float32)
            b.dg1 = e((d,), torch.float32)
            if keep_intermediates:
                b.dh8 = q8((T, d))
                b.dQKV8 = q8((T, n_qkv))
                b.dN1 = e((T, d), torch.float32)
        if core is not None:
            b.n_heads, b.n_kv_heads, b.seq_len = (int(v) for v in core)
            b.lse = e((b.n_heads, T), torch.float32)
        nb = lib.block_workspace_size(T, d, f, n_qkv, int(backward))
        b.ws = torch.empty(nb, dtype=torch.uint8, device=device)
        return b

    @property
    def h(self) -> torch.Tensor:
        return self.mlp.x

    @property
    def dh(self) -> torch.Tensor:
        return self.mlp.dX

    def struct(self) -> FP8QBlock:
        s = FP8QBlock(T=self.T, d=self.d, f=self.f, n_qkv=self.n_qkv, eps=self.eps, n_heads=self.n_heads,
                      n_kv_heads=self.n_kv_heads, seq_len=self.seq_len)
        s.lse = None if self.lse is None else self.lse.data_ptr()
        s.n1_16 = None if self.n1_16 is None else self.n1_16.data_ptr()
        for name in ("x", "g1", "W_qkv", "W_o", "att", "qkv", "W_qkv8", "W_o8", "n1_8", "rstd1", "att8", "scal",
                     "dQKV", "d_att", "dX", "dW_qkv", "dW_o", "dg1", "dh8", "dQKV8", "dN1"):
            t = getattr(self, name)
            setattr(s, name, None if t is None else t.data_ptr())
        s.h = self.mlp.x.data_ptr()
        s.mlp = self.mlp.struct()
        return s


def block_fwd(b: BlockBuffers, stream=None):
    s = b.struct()
    _check("block_fwd", lib.block_fwd(ctypes.byref(s), _ptr(b.ws), b.ws.numel(), _stream(stream)))


def block_bwd(b: BlockBuffers, stream=None):
    s = b.struct()
    _check("block_bwd", lib.block_bwd(ctypes.byref(s), _ptr(b.ws), b.ws.numel(), _stream(stream)))


def block_run_steps(b0: BlockBuffers, b1: BlockBuffers, host: list, backward: bool = True, stream=None):
    """Pipelined full-block steps from and to host memory (block_run_steps in include/fp8q.h).
    host: one dict per step, keys as fp8q_block_host_io (x, g1, W_qkv, W_o, att, g, W_gu, W_d, dY,
    dQKV in; y, dX, d_att, dW_qkv, dW_o, dg1, dW_gu, dW_d, dg out); missing entries stay on the
    device.  Device sets b0, b1 alternate; b0's workspace is used."""
    _check("block_run_steps", lib.block_run_steps(*_steps_args(b0, b1, host, FP8QBlockHostIO), int(bool(backward)),
                                                  _ptr(b0.ws), b0.ws.numel(), _stream(stream)))


def selftest_gemm_wait_limit(layout: int, A: torch.Tensor, fmtA: int, B: torch.Tensor, fmtB: int, limit_s: float,
                             sinvA=None, sinvB=None, sfA=None, sfB=None, out_dtype=torch.float32, C=None,
                             stream=None):
    """fp8_gemm_scaled (sinvA/sinvB given) or fp8_gemm_mx (sfA/sfB given) with every pipeline wait of
    the kernel limited to limit_s (fp8q_selftest_gemm_wait_limit in include/fp8q.h).  Returns C."""
    dev = _dev(A)
    if layout == TN:
        K, M = A.shape
    else:
        M, K = A.shape
    N = B.shape[0] if layout == NT else B.shape[1]
    out_code = {torch.bfloat16: BF16, torch.float32: F32}[out_dtype]
    C = torch.empty((M, N), dtype=out_dtype, device=dev) if C is None else C
    mx = sfA is not None
    _check("fp8q_selftest_gemm_wait_limit",
           lib.fp8q_selftest_gemm_wait_limit(layout, M, N, K, _ptr(A), fmtA, A.shape[1], _ptr(B), fmtB, B.shape[1],
                                             _ptr(sinvA), _ptr(sinvB), int(mx), _ptr(sfA), _ptr(sfB), _ptr(C),
                                             out_code, C.shape[1], int(limit_s * 1e9), _stream(stream)))
    return C


def selftest_bounded_wait(limit_s: float = 0.02, stream=None):
    """Make the library's bounded wait run out on purpose (an mbarrier nothing arrives at);
    afterwards the device status carries STATUS_TIMEOUT.  Diagnostics only."""
    _check("fp8q_selftest_bounded_wait", lib.fp8q_selftest_bounded_wait(int(limit_s * 1e9), _stream(stream)))
