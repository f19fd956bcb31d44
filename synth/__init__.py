"""Seeded synthetic inputs for the FP8 MLP-block workloads.

This module is the only code that both the CUDA path's tests/benchmark and
the CPU oracle consume.  It holds no arithmetic of the method itself: it draws
random tensors, rounds them once to bf16, and describes the five workloads.

Generator: numpy's counter-based Philox bit generator (Salmon et al.,
"Parallel random numbers: as easy as 1, 2, 3", SC'11), keyed by
(seed, tensor id) so every tensor has its own independent stream; normals
from numpy's ``standard_normal``.  Values are produced in fp32 (outlier
channel scaling applied there) and rounded once, round-to-nearest-even, to
bf16.  bf16 tensors travel as uint16 bit patterns.

Workloads (the pages name no public dataset for this path; these synthetic
shapes and value distributions stand in for LLM activations, weights and
gradients):

  tiny-mlp-fwd         T=256,   d=512,  f=1408   forward only
  3b-mlp-fwd           T=4096,  d=2048, f=11008  forward only, 1% outlier channels x20
  7b-mlp-fwd-bwd       T=8192,  d=3584, f=18944  forward+backward, 1% outlier channels x20
  14b-mlp-fwd-bwd      T=8192,  d=5120, f=13824  forward+backward, x = 0.5 * Student-t(4)
  32b-block-fwd-bwd    T=16384, d=5120, f=27648  forward+backward, QKV 7168, 0.5% outliers x30
  32b-block-attn-fwd-bwd  the same block with its attention core computed inside: 40 query heads,
                       8 K/V heads of 128, 4 sequences of 4096 tokens (causal)
"""

from __future__ import annotations

import dataclasses

import numpy as np

# tensor ids (part of each stream's Philox key)
TID_X, TID_G, TID_WGU, TID_WD, TID_DY, TID_OUTLIER = 1, 2, 3, 4, 5, 6
TID_WQKV, TID_WO, TID_G1, TID_ATT, TID_DQKV, TID_OUTLIER_ATT = 7, 8, 9, 10, 11, 12


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    x_kind: str            # "normal" | "student_t4"
    x_scale: float         # std of normal x, or the multiplier of Student-t
    outlier_frac: float    # fraction of channels scaled as outliers (0: none)
    outlier_mult: float
    w_std: float
    dy_std: float          # 0: forward only
    qkv: int = 0           # QKV output width (full-block workload), 0: MLP only
    n_heads: int = 0       # attention core inside the block (0: att / dQKV are given tensors)
    n_kv_heads: int = 0
    seq_len: int = 0

    @property
    def backward(self) -> bool:
        return self.dy_std > 0

    def gemm_flops(self) -> float:
        """Algorithmic GEMM FLOPs of one step: 6Tdf forward, 18Tdf forward+backward
        (plus the QKV and O projections for the full-block workload)."""
        per = 6.0 * self.T * self.d * self.f
        if self.qkv:
            per += 2.0 * self.T * self.d * self.qkv + 2.0 * self.T * self.d * self.d
        return per * (3.0 if self.backward else 1.0)

    def attention_flops(self) -> float:
        """Algorithmic FLOPs of the causal attention core (0 without it): S(S+1)/2 query-key pairs
        per sequence and head, 2 products (Q K^T, P V) forward and 5 (S, dP, dV, dK, dQ) backward,
        2 * 128 FLOPs per pair and product."""
        if not self.n_heads:
            return 0.0
        pairs = (self.T // self.seq_len) * self.seq_len * (self.seq_len + 1) / 2
        return pairs * self.n_heads * 2.0 * 128 * (7 if self.backward else 2)


WORKLOADS = [
    Workload("tiny-mlp-fwd", 256, 512, 1408, "normal", 1.0, 0.0, 1.0, 0.02, 0.0),
    Workload("3b-mlp-fwd", 4096, 2048, 11008, "normal", 1.0, 0.01, 20.0, 0.02, 0.0),
    Workload("7b-mlp-fwd-bwd", 8192, 3584, 18944, "normal", 1.0, 0.01, 20.0, 0.02, 1e-3),
    Workload("14b-mlp-fwd-bwd", 8192, 5120, 13824, "student_t4", 0.5, 0.0, 1.0, 0.015, 1e-3),
    Workload("32b-block-fwd-bwd", 16384, 5120, 27648, "normal", 1.0, 0.005, 30.0, 0.01, 1e-3, qkv=7168),
    Workload("32b-block-attn-fwd-bwd", 16384, 5120, 27648, "normal", 1.0, 0.005, 30.0, 0.01, 1e-3, qkv=7168,
             n_heads=40, n_kv_heads=8, seq_len=4096),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=(int(seed) << 32) | int(tensor_id)))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(shape, std: float, seed: int, tensor_id: int, mean: float = 0.0) -> np.ndarray:
    v = rng(seed, tensor_id).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    if mean != 0.0:
        v += np.float32(mean)
    return bf16_bits(v)


def outlier_channels(d: int, frac: float, seed: int, tensor_id: int) -> np.ndarray:
    k = int(round(frac * d))
    if k == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(rng(seed, tensor_id).permutation(d)[:k])


def activations(w: Workload, T: int, d: int, seed: int, tensor_id: int, outlier_id: int) -> np.ndarray:
    """[T,d] activations with the workload's distribution, as bf16 bits."""
    r = rng(seed, tensor_id)
    if w.x_kind == "student_t4":
        v = (r.standard_t(4.0, (T, d)) * w.x_scale).astype(np.float32)
    else:
        v = r.standard_normal((T, d), dtype=np.float32)
        if w.x_scale != 1.0:
            v *= np.float32(w.x_scale)
    ch = outlier_channels(d, w.outlier_frac, seed, outlier_id)
    if ch.size:
        v[:, ch] *= np.float32(w.outlier_mult)
    return bf16_bits(v)


def mlp_inputs(w: Workload, seed: int = 0, T: int | None = None, d: int | None = None,
               f: int | None = None) -> dict:
    """Inputs of the MLP block: x [T,d], g [d], W_gu [d,2f] (gate | up), W_d [f,d],
    and dY [T,d] for backward workloads.  T, d, f override the workload's sizes
    (same distributions) for small parity cases."""
    T = w.T if T is None else T
    d = w.d if d is None else d
    f = w.f if f is None else f
    out = {
        "x": activations(w, T, d, seed, TID_X, TID_OUTLIER),
        "g": normal_bf16((d,), 0.1, seed, TID_G, mean=1.0),
        "W_gu": normal_bf16((d, 2 * f), w.w_std, seed, TID_WGU),
        "W_d": normal_bf16((f, d), w.w_std, seed, TID_WD),
    }
    if w.backward:
        out["dY"] = normal_bf16((T, d), w.dy_std, seed, TID_DY)
    return out


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Exact fp32 value of bf16 bit patterns (for building device tensors)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def block_inputs(w: Workload, seed: int = 0, T: int | None = None, d: int | None = None, f: int | None = None,
                 n_qkv: int | None = None) -> dict:
    """Inputs of the full block: the MLP's (x, g = the MLP gain, W_gu, W_d, dY) plus g1 [d],
    W_qkv [d, n_qkv], W_o [d, d], the attention core's output att [T, d] (same distribution as x,
    its own outlier channels) and the gradient arriving at the core's input dQKV [T, n_qkv]."""
    out = mlp_inputs(w, seed, T, d, f)
    T, d = out["x"].shape
    nq = w.qkv if n_qkv is None else n_qkv
    out["g1"] = normal_bf16((d,), 0.1, seed, TID_G1, mean=1.0)
    out["W_qkv"] = normal_bf16((d, nq), w.w_std, seed, TID_WQKV)
    out["W_o"] = normal_bf16((d, d), w.w_std, seed, TID_WO)
    out["att"] = activations(w, T, d, seed, TID_ATT, TID_OUTLIER_ATT)
    if w.backward:
        out["dQKV"] = normal_bf16((T, nq), w.dy_std, seed, TID_DQKV)
    return out
