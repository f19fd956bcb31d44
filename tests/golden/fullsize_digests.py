"""Writes the oracle's results for the full-size workloads, as compact digests, into
``tests/golden/fullsize/<workload>.npz``.

The GPU tests of the 3B-, 7B- and 14B-class MLP blocks and of the 32B-class full block compare the
CUDA library's full-size outputs with these files.  Every value stored here comes from the CPU
oracle (``oracle/``) run on the seeded inputs of ``synth/``; nothing is taken from the CUDA path.

What a file holds (row indices are stored beside the rows):
  * ``sha_in_<name>``: SHA-256 of each input tensor, so a test can tell that the inputs it rebuilt
    on its own machine are the ones these results were computed from;
  * every {amax, scale, scale_inv} triple (``scal_fwd``, ``scal_bwd``, ``scal_attn``);
  * ``sha_<name>``: SHA-256 of the tensors the GPU must reproduce bit for bit (quantizer codes
    and RMSNorm statistics whose input is a given tensor);
  * sampled token rows of every per-token output (bf16 tensors as bit patterns, FP8 tensors as
    codes, fp32 tensors as fp32), chosen on both sides of the 128- and 256-row tile edges, the
    2048-row rasterisation-group edge and the last row;
  * sampled rows of every weight gradient, and every gain gradient in full;
  * for ``<workload>-mx`` (the block-scaled MXFP8 block): SHA-256 of every block quantization of a
    given tensor (codes and E8M0 scales), and the sampled rows (and their column blocks' scales) of
    the requantized a and dH in both block directions.

Usage: ``python tests/golden/fullsize_digests.py [--threads N] [workload ...]`` (default: all five
entries, one thread per core; the 32B-class block needs about 40 GB of host memory).
"""

from __future__ import annotations

import argparse
import hashlib
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

OUT_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fullsize")
WORKLOADS = ("3b-mlp-fwd", "7b-mlp-fwd-bwd", "14b-mlp-fwd-bwd", "32b-block-fwd-bwd", "7b-mlp-fwd-bwd-mx")
MX_SUFFIX = "-mx"  # <workload>-mx: the block-scaled MXFP8 block on that workload's inputs


def sha(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def token_rows(T: int) -> np.ndarray:
    """Both sides of the 128- and 256-row tile edges and of the 2048-row rasterisation-group edge,
    one row inside the second half, the last row."""
    r = {0, 127, 128, 255, 256, 2047, 2048, T // 2 + 77, T - 129, T - 1}
    return np.array(sorted(i for i in r if 0 <= i < T), dtype=np.int64)


def weight_rows(n: int) -> np.ndarray:
    r = {0, 127, 128, 256, n // 2 + 3, n - 1}
    return np.array(sorted(i for i in r if 0 <= i < n), dtype=np.int64)


def bits(v: np.ndarray) -> np.ndarray:
    """bf16 values (float64, exactly representable) -> their bf16 bit patterns."""
    b = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32).view(np.uint32)
    assert not (b & 0xFFFF).any(), "not a bf16 value"
    return (b >> 16).astype(np.uint16)


def f32(v: np.ndarray) -> np.ndarray:
    out = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32)
    assert np.array_equal(out.astype(np.float64), np.asarray(v)), "not an fp32 value"
    return out


def mlp_digest(w, threads: int) -> dict:
    inp = synth.mlp_inputs(w, seed=0)
    t0 = time.time()
    r = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp.get("dY"), nthreads=threads)
    secs = time.time() - t0
    assert r["status"] == 0
    rows = token_rows(w.T)
    out = {f"sha_in_{k}": sha(v) for k, v in inp.items()}
    out.update(rows=rows, scal_fwd=r["scal_fwd"], sha_Wgu8=sha(r["Wgu8"]), sha_Wd8=sha(r["Wd8"]),
               sha_n8=sha(r["n8"]), sha_rstd=sha(f32(r["rstd"])),
               H=bits(r["H"][rows]), a8=r["a8"][rows], y=bits(r["y"][rows]))
    if w.backward:
        rd, rg = weight_rows(w.f), weight_rows(w.d)
        out.update(scal_bwd=r["scal_bwd"], sha_dY8=sha(r["dY8"]), dH=bits(r["dH"][rows]), dH8=r["dH8"][rows],
                   dN=f32(r["dN"][rows]), dX=bits(r["dX"][rows]), rows_dWd=rd, dWd=f32(r["dWd"][rd]),
                   rows_dWgu=rg, dWgu=f32(r["dWgu"][rg]), dg=f32(r["dg"]))
    out["oracle_seconds"] = np.float64(secs)
    out["oracle_threads"] = np.int64(threads)
    return out


def mlp_mx_digest(w, threads: int) -> dict:
    """The block-scaled MXFP8 block (oracle.block(..., mx=True)) on the workload's inputs."""
    inp = synth.mlp_inputs(w, seed=0)
    t0 = time.time()
    r = oracle.block(inp["x"], inp["g"], inp["W_gu"], inp["W_d"], dY=inp["dY"], nthreads=threads, mx=True)
    secs = time.time() - t0
    assert r["status"] == 0
    rows = token_rows(w.T)
    blocks = np.unique(rows // oracle.MX_BLOCK)  # the column blocks (32 tokens) holding the sampled rows
    rd, rg = weight_rows(w.f), weight_rows(w.d)
    out = {f"sha_in_{k}": sha(v) for k, v in inp.items()}
    out.update(rows=rows, col_blocks=blocks, rows_dWd=rd, rows_dWgu=rg, sha_rstd=sha(f32(r["rstd"])),
               H=bits(r["H"][rows]), y=bits(r["y"][rows]), dH=bits(r["dH"][rows]), dN=f32(r["dN"][rows]),
               dX=bits(r["dX"][rows]), dWd=f32(r["dWd"][rd]), dWgu=f32(r["dWgu"][rg]), dg=f32(r["dg"]))
    for slot in oracle.MX_SLOTS:
        q, sf = r["mx_" + slot], r["mx_" + slot + "_sf"]
        if slot.split("_")[0] in ("Wgu", "Wd", "n", "dY"):   # quantizers of given tensors: bit for bit
            out["sha_mx_" + slot] = sha(q)
            out["sha_mx_" + slot + "_sf"] = sha(sf)
        else:                                                 # requantizations of GEMM outputs: sampled
            out["mx_" + slot] = q[rows]
            out["mx_" + slot + "_sf"] = sf[rows] if slot.endswith("_r") else sf[blocks]
    out["oracle_seconds"] = np.float64(secs)
    out["oracle_threads"] = np.int64(threads)
    return out


def block_digest(w, threads: int) -> dict:
    inp = synth.block_inputs(w, seed=0)
    t0 = time.time()
    r = oracle.full_block(inp["x"], inp["g1"], inp["W_qkv"], inp["W_o"], inp["att"], inp["g"], inp["W_gu"],
                          inp["W_d"], dY=inp["dY"], dQKV=inp["dQKV"], nthreads=threads)
    secs = time.time() - t0
    assert r["status"] == 0
    rows = token_rows(w.T)
    rd, rg = weight_rows(w.f), weight_rows(w.d)
    out = {f"sha_in_{k}": sha(v) for k, v in inp.items()}
    out.update(rows=rows, rows_dWd=rd, rows_dW=rg,
               scal_attn=r["scal_attn"], scal_fwd=r["scal_fwd"], scal_bwd=r["scal_bwd"],
               sha_Wqkv8=sha(r["Wqkv8"]), sha_Wo8=sha(r["Wo8"]), sha_n1_8=sha(r["n1_8"]), sha_att8=sha(r["att8"]),
               sha_rstd1=sha(f32(r["rstd1"])), sha_Wgu8=sha(r["Wgu8"]), sha_Wd8=sha(r["Wd8"]),
               sha_dY8=sha(r["dY8"]), sha_dqkv8=sha(r["dqkv8"]),
               qkv=bits(r["qkv"][rows]), h=bits(r["h"][rows]), n8=r["n8"][rows], H=bits(r["H"][rows]),
               a8=r["a8"][rows], y=bits(r["y"][rows]),
               dH=bits(r["dH"][rows]), dH8=r["dH8"][rows], dN=f32(r["dN"][rows]), dh=bits(r["dh"][rows]),
               dh8=r["dh8"][rows], d_att=bits(r["d_att"][rows]), dX=bits(r["dX"][rows]),
               dWd=f32(r["dWd"][rd]), dWgu=f32(r["dWgu"][rg]), dWo=f32(r["dWo"][rg]), dWqkv=f32(r["dWqkv"][rg]),
               dg=f32(r["dg"]), dg1=f32(r["dg1"]))
    out["oracle_seconds"] = np.float64(secs)
    out["oracle_threads"] = np.int64(threads)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--threads", type=int, default=os.cpu_count() or 1)
    ap.add_argument("workloads", nargs="*", default=list(WORKLOADS))
    args = ap.parse_args()
    os.makedirs(OUT_DIR, exist_ok=True)
    for name in args.workloads:
        mx = name.endswith(MX_SUFFIX)
        w = synth.BY_NAME[name[: -len(MX_SUFFIX)] if mx else name]
        t0 = time.time()
        if mx:
            dig = mlp_mx_digest(w, args.threads)
        else:
            dig = block_digest(w, args.threads) if w.qkv else mlp_digest(w, args.threads)
        dig["numpy_version"] = np.array(np.__version__)
        path = os.path.join(OUT_DIR, name + ".npz")
        np.savez_compressed(path, **dig)
        print(f"{name}: oracle {float(dig['oracle_seconds']):.0f} s on {args.threads} threads, total "
              f"{time.time() - t0:.0f} s -> {os.path.relpath(path, ROOT)} ({os.path.getsize(path) / 1e6:.1f} MB)",
              flush=True)


if __name__ == "__main__":
    main()
