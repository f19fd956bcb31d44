"""Helpers shared by the GPU parity tests: host <-> device conversion and the error metrics."""

import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bfloat16 tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """CUDA bf16 tensor -> uint16 bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def row_rel(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of ||got_i - ref_i||_2 / ||ref_i||_2 (rows with a zero reference are skipped
    unless got is non-zero there)."""
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, dtype=np.float64).reshape(ref.shape[0], -1)
    num = np.linalg.norm(got - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    zero = den == 0
    if (num[zero] > 0).any():
        return float("inf")
    return float((num[~zero] / den[~zero]).max()) if (~zero).any() else 0.0


def code_step_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable steps between FP8 codes of the same format (sign-magnitude)."""
    def ordinal(c):
        c = c.astype(np.int32)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordinal(a) - ordinal(b))


def fp8_table(fmt: int) -> np.ndarray:
    """Values of all 256 FP8 codes, built for property checks without the oracle: the positive
    finite values are the multiples of the smallest subnormal whose multiplier has at most
    1 + frac significant bits, up to the format's maximum, in increasing code order."""
    frac, lsub, vmax = (3, -9, 448.0) if fmt == 0 else (2, -16, 57344.0)
    kmax = int(vmax / 2.0 ** lsub)
    ks = sorted({m << j for m in range(1 << (frac + 1)) for j in range(64) if (m << j) <= kmax})
    pos = np.array([k * 2.0 ** lsub for k in ks])
    t = np.full(256, np.nan)
    t[: pos.size] = pos
    t[128: 128 + pos.size] = -pos
    if fmt == 1:
        t[0x7C], t[0xFC] = np.inf, -np.inf
    return t


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """CUDA bf16 tensor -> float64 values."""
    return host_f64(t)


def _mx_offsets(rows: int, nb: int) -> np.ndarray:
    """Byte offsets of (row r, K block b) in the chunked scale layout of include/fp8q.h: 512-byte
    chunks of 128 rows x 4 blocks, row-chunk-major; inside a chunk (r % 32) * 16 + (r / 32) * 4 + b."""
    nkc = (nb + 3) // 4
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    return ((r // 128) * nkc + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4


def mx_sf_to_chunked(plain: np.ndarray) -> np.ndarray:
    """Scale codes [rows, K/32] -> the chunked byte layout (padding rows / blocks hold 127, i.e. 1.0)."""
    rows, nb = plain.shape
    out = np.full(((rows + 127) // 128) * ((nb + 3) // 4) * 512, 127, dtype=np.uint8)
    out[_mx_offsets(rows, nb)] = plain
    return out


def mx_sf_from_chunked(chunked: np.ndarray, rows: int, K: int) -> np.ndarray:
    """The chunked layout -> scale codes [rows, K/32]."""
    return np.asarray(chunked).ravel()[_mx_offsets(rows, (K + 31) // 32)]
