#!/usr/bin/env python
"""Benchmark of the FP8 MLP block (forward + backward) on GB300.

One step = mlp_block_fwd + mlp_block_bwd of the chosen workload (default: the
7B-class MLP, T=8192, d=3584, f=18944) through the C ABI: weight / activation
/ gradient quantization, RMSNorm, the six FP8 GEMMs with their fused
epilogues, SwiGLU requantization and the RMSNorm backward.

Prints one JSON line.  value = algorithmic GEMM TFLOP/s of the whole job
(18*T*d*f per step, summed over ranks); e2e = the same metric with each
step's batch (activations and upstream gradients in, block output and input
gradients out) copied between pinned host memory and the device inside the
timed region, the model state resident in HBM; e2e_all_io = the same with
every input and output, weights and weight gradients included, through the
host.  The roofline object is for the dominant kernel (the
tcgen05 GEMM), timed live with CUDA events recorded by the library around each
of its launches in the first --trace-steps steps of the timed region (the
event pairs are stream work of their own, ~2 % of a step when every step is
traced).

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl ours|reference]

N > 1 (under torchrun): independent replicas, one per GPU (the block has no
exchange step in the forward/backward pass itself); weak scaling.
--impl reference: the CPU oracle, timed on this machine's host cores on a
bounded token sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "FP8 MLP-block fwd+bwd TFLOP/s & tokens/s, % of GB300 dense FP8 peak (1 GPU)"
FP8_PER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor throughput on GB300 (4.5 : 2.25 PFLOP/s)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b-mlp-fwd-bwd", choices=[w.name for w in synth.WORKLOADS])
    ap.add_argument("--cpu-sample-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay figure")
    ap.add_argument("--recompute", action="store_true",
                    help="recompute-mode backward (H and a8 recomputed from n8 with the retained scale)")
    ap.add_argument("--grad-e4m3", action="store_true",
                    help="E4M3 gradients (dY, dH; dh, dQKV in the full block) instead of E5M2")
    ap.add_argument("--bf16", action="store_true",
                    help="the BF16 baseline (same block, bf16 operands, tcgen05 kind::f16) for the FP8/BF16 speedup")
    ap.add_argument("--mxfp8", action="store_true",
                    help="the block-scaled MXFP8 MLP block (E8M0 scale per 32 elements, tcgen05 block_scale GEMMs)")
    ap.add_argument("--measure-fp8-peak", action="store_true",
                    help="time cuBLASLt FP8 (torch._scaled_mm) 8192^3, burst and sustained, and exit")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's T (same d, f, distributions); for small profiling runs")
    ap.add_argument("--trace-steps", type=int, default=10,
                    help="timed steps whose kernel launches the per-launch trace brackets with CUDA events "
                         "(the first ones of the timed region)")
    ap.add_argument("--launch-log", default="",
                    help="write the mean time of every launch position of the step (kernel, bytes, flops, us) "
                         "to this JSON file")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            m = json.load(fh)
        return {"hbm_gbs": m["hbm_gbs"], "bf16": m["bf16_tflops"], "bf16_sustained": m["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
            os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][1]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------
# replicas across ranks (one process per GPU; no exchange in the data path)
# ---------------------------------------------------------------------------
def max_over_ranks(v: float, device=None) -> float:
    """The largest value of v over all ranks (a time: the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / (max_ms * 1e-3)


# ---------------------------------------------------------------------------
# per-launch algorithmic work of one step (order = the library's launch order)
# ---------------------------------------------------------------------------
def step_work(w: synth.Workload, recompute: bool = False, bf16: bool = False, mx: bool = False):
    """(kernel kind, algorithmic bytes, flops) of every traced launch of one step (the recompute
    GEMM's flops are executed work on top of the algorithmic 18Tdf)."""
    T, d, f = w.T, w.d, w.f
    if mx:  # the MXFP8 MLP block: each quantizer pass reads its input once and writes both code
        # tensors (2 B per element) and both scale sets (2 / 32 B per element)
        q = lambda n, rd: ("mx_quant", n * (rd + 2 + 2 / 32), 0)
        sf = lambda n: n / 32   # scale bytes of one operand
        fwd = [
            q(d * 2 * f, 2), q(f * d, 2),
            ("rmsnorm_stats", 2 * T * d + 2 * d + 4 * T, 0), ("mx_quant", T * d * (2 + 2 + 2 / 32) + 4 * T + 2 * d, 0),
            ("gemm_gate_up_swiglu", T * d + d * 2 * f + sf(T * d) + sf(d * 2 * f) + 2 * T * 2 * f, 2.0 * T * d * 2 * f),
            q(T * f, 4),
            ("gemm_down_residual", T * f + f * d + sf(T * f) + sf(f * d) + 4 * T * d, 2.0 * T * f * d),
        ]
        bwd = [
            q(T * d, 2),
            ("gemm_down_dgrad_swiglu_bwd", T * d + f * d + sf(T * d) + sf(f * d) + 2 * T * 2 * f * 2, 2.0 * T * d * f),
            q(T * 2 * f, 2),
            ("gemm_down_wgrad", T * f + T * d + sf(T * f) + sf(T * d) + 4 * f * d, 2.0 * f * T * d),
            ("gemm_gate_up_dgrad", T * 2 * f + d * 2 * f + sf(T * 2 * f) + sf(d * 2 * f) + 4 * T * d, 2.0 * T * 2 * f * d),
            ("gemm_gate_up_wgrad", T * d + T * 2 * f + sf(T * d) + sf(T * 2 * f) + 4 * d * 2 * f, 2.0 * d * T * 2 * f),
            ("rmsnorm_bwd", 10 * T * d, 0),
        ]
        return fwd + (bwd if w.backward else [])
    if bf16:  # the BF16 baseline: 2-byte operands, no casts
        fwd = [
            ("rmsnorm_bf16", 4 * T * d + 2 * d + 4 * T, 0),
            ("gemm_gate_up_swiglu", 2 * T * d + 2 * d * 2 * f + 2 * T * 2 * f + 2 * T * f, 2.0 * T * d * 2 * f),
            ("gemm_down_residual", 2 * T * f + 2 * f * d + 4 * T * d, 2.0 * T * f * d),
        ]
        bwd = [
            ("gemm_down_dgrad_swiglu_bwd", 2 * T * d + 2 * f * d + 2 * T * 2 * f * 2, 2.0 * T * d * f),
            ("gemm_down_wgrad", 2 * T * f + 2 * T * d + 4 * f * d, 2.0 * f * T * d),
            ("gemm_gate_up_dgrad", 2 * T * 2 * f + 2 * d * 2 * f + 4 * T * d, 2.0 * T * 2 * f * d),
            ("gemm_gate_up_wgrad", 2 * T * d + 2 * T * 2 * f + 4 * d * 2 * f, 2.0 * d * T * 2 * f),
            ("rmsnorm_bwd", 10 * T * d, 0),
        ]
        if not w.qkv:
            return fwd + (bwd if w.backward else [])
        q = w.qkv
        core_f, core_b = [], []
        if w.n_heads:
            hq, hkv = w.n_heads, w.n_kv_heads
            pairs = (T // w.seq_len) * w.seq_len * (w.seq_len + 1) / 2 * hq
            core_f = [("attn_fwd", 2 * T * q + 2 * T * d + 4 * T * hq, 4.0 * 128 * pairs)]
            core_b = [("attn_bwd_delta", 4 * T * d + 12 * T * hq, 0),
                      ("attn_bwd_dkdv", 2 * T * q + 2 * T * d + 8 * T * hq + 4 * T * hkv * 128, 8.0 * 128 * pairs),
                      ("attn_bwd_dq", 2 * T * q + 4 * T * d + 8 * T * hq, 6.0 * 128 * pairs)]
        a_fwd = [("rmsnorm_bf16", 4 * T * d + 2 * d + 4 * T, 0),
                 ("gemm_qkv", 2 * T * d + 2 * d * q + 2 * T * q, 2.0 * T * d * q), *core_f,
                 ("gemm_o_residual", 2 * T * d + 2 * d * d + 4 * T * d, 2.0 * T * d * d)]
        a_bwd = [("gemm_o_dgrad", 2 * T * d + 2 * d * d + 2 * T * d, 2.0 * T * d * d),
                 ("gemm_o_wgrad", 4 * T * d + 4 * d * d, 2.0 * T * d * d), *core_b,
                 ("gemm_qkv_dgrad", 2 * T * q + 2 * d * q + 4 * T * d, 2.0 * T * q * d),
                 ("gemm_qkv_wgrad", 2 * T * d + 2 * T * q + 4 * d * q, 2.0 * T * d * q),
                 ("rmsnorm_bwd", 10 * T * d, 0)]
        return a_fwd + fwd + (bwd + a_bwd if w.backward else [])
    mlp_fwd = [
        # the quantizer prologue: RMSNorm statistics beside the two weight absmax passes, then the casts
        ("prologue_stats", 2 * d * 2 * f + 2 * f * d + 2 * T * d + 2 * d + 4 * T, 0),
        ("prologue_cast", 3 * d * 2 * f + 3 * f * d + 3 * T * d + 4 * T + 2 * d, 0),
        ("gemm_gate_up_swiglu", T * d + d * 2 * f + 2 * T * 2 * f, 2.0 * T * d * 2 * f),
        ("swiglu_cast", 4 * T * f + T * f, 0),
        ("gemm_down_residual", T * f + f * d + 4 * T * d, 2.0 * T * f * d),
    ]
    mlp_bwd = [
        ("absmax_partial", 2 * T * d, 0), ("quant_cast", 3 * T * d, 0),
        ("gemm_down_dgrad_swiglu_bwd", T * d + f * d + 2 * T * 2 * f * 2, 2.0 * T * d * f),
        ("quant_cast", 3 * T * 2 * f, 0),
        ("gemm_down_wgrad", T * f + T * d + 4 * f * d, 2.0 * f * T * d),
        ("gemm_gate_up_dgrad", T * 2 * f + d * 2 * f + 4 * T * d, 2.0 * T * 2 * f * d),
        ("gemm_gate_up_wgrad", T * d + T * 2 * f + 4 * d * 2 * f, 2.0 * d * T * 2 * f),
        ("rmsnorm_bwd", 10 * T * d, 0),
    ]
    if recompute:
        mlp_bwd = [("gemm_gate_up_recompute", T * d + d * 2 * f + 2 * T * 2 * f + T * f, 2.0 * T * d * 2 * f)] + mlp_bwd
    if not w.qkv:
        return mlp_fwd + (mlp_bwd if w.backward else [])
    q = w.qkv
    attn_fwd = [
        # the attention side's quantizer prologue: RMSNorm statistics beside the W_qkv and W_o
        # absmax passes, then the three casts
        ("prologue_stats", 2 * d * q + 2 * d * d + 2 * T * d + 2 * d + 4 * T, 0),
        ("prologue_cast", 3 * d * q + 3 * d * d + 3 * T * d + 4 * T + 2 * d, 0),
        ("gemm_qkv", T * d + d * q + 2 * T * q, 2.0 * T * d * q),
        ("absmax_partial", 2 * T * d, 0), ("quant_cast", 3 * T * d, 0),
        ("gemm_o_residual", T * d + d * d + 4 * T * d, 2.0 * T * d * d),
    ]
    core_fwd, core_bwd = [], []
    if w.n_heads:
        # the attention core: bytes read/written once; FLOPs executed (2 * 128 per causal pair and
        # product: 2 products forward; dK/dV recomputes S and forms dP, dV, dK (4), dQ recomputes
        # S and dP and forms dQ (3) -- the algorithmic count in the headline uses 5)
        hq, hkv = w.n_heads, w.n_kv_heads
        pairs = (T // w.seq_len) * w.seq_len * (w.seq_len + 1) / 2 * hq
        core_fwd = [("attn_fwd", 2 * T * q + 2 * T * d + 4 * T * hq, 4.0 * 128 * pairs)]
        core_bwd = [
            ("attn_bwd_delta", 4 * T * d + 12 * T * hq, 0),
            ("attn_bwd_dkdv", 2 * T * q + 2 * T * d + 8 * T * hq + 4 * T * hkv * 128, 8.0 * 128 * pairs),
            ("attn_bwd_dq", 2 * T * q + 4 * T * d + 8 * T * hq, 6.0 * 128 * pairs),
        ]
        attn_fwd = attn_fwd[:3] + core_fwd + attn_fwd[3:]
    attn_bwd = [
        ("absmax_partial", 2 * T * d, 0), ("quant_cast", 3 * T * d, 0),
        ("gemm_o_dgrad", T * d + d * d + 2 * T * d, 2.0 * T * d * d),
        ("gemm_o_wgrad", 2 * T * d + 4 * d * d, 2.0 * T * d * d),
        *core_bwd,
        ("absmax_partial", 2 * T * q, 0), ("quant_cast", 3 * T * q, 0),
        ("gemm_qkv_dgrad", T * q + d * q + 4 * T * d, 2.0 * T * q * d),
        ("gemm_qkv_wgrad", T * d + T * q + 4 * d * q, 2.0 * T * d * q),
        ("rmsnorm_bwd", 10 * T * d, 0),
    ]
    return attn_fwd + mlp_fwd + (mlp_bwd + attn_bwd if w.backward else [])


# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import fp8_absmax_reduce_gb300 as fq

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = args.w
    flops = w.gemm_flops() + w.attention_flops()
    if w.qkv:
        inp = synth.block_inputs(w, seed=rank)
        core = (w.n_heads, w.n_kv_heads, w.seq_len) if w.n_heads else None
        b = fq.BlockBuffers.allocate(w.T, w.d, w.f, w.qkv, device=dev, backward=w.backward, core=core,
                                     bf16=args.bf16)
        dev_in = {"x": b.x, "g1": b.g1, "W_qkv": b.W_qkv, "W_o": b.W_o, "g": b.mlp.g,
                  "W_gu": b.mlp.W_gu, "W_d": b.mlp.W_d}
        if not core:
            dev_in["att"] = b.att    # the attention core's output is given
        if w.backward:
            dev_in["dY"] = b.mlp.dY
            if not core:
                dev_in["dQKV"] = b.dQKV
        dev_out = {"y": b.mlp.y}
        if w.backward:
            dev_out.update(dX=b.dX, dW_qkv=b.dW_qkv, dW_o=b.dW_o, dg1=b.dg1, dW_gu=b.mlp.dW_gu, dW_d=b.mlp.dW_d,
                           dg=b.mlp.dg, d_att=b.d_att)
        fwd, bwd = fq.block_fwd, fq.block_bwd
    else:
        inp = synth.mlp_inputs(w, seed=rank)
        b = fq.MlpBuffers.allocate(w.T, w.d, w.f, device=dev, backward=w.backward, bf16=args.bf16, mx=args.mxfp8)
        dev_in = {k: getattr(b, k) for k in ["x", "g", "W_gu", "W_d"] + (["dY"] if w.backward else [])}
        dev_out = {"y": b.y}
        if w.backward:
            dev_out.update(dX=b.dX, dW_gu=b.dW_gu, dW_d=b.dW_d, dg=b.dg)
        fwd, bwd = fq.mlp_block_fwd, fq.mlp_block_bwd
    (b.mlp if w.qkv else b).recompute = bool(args.recompute)
    (b.mlp if w.qkv else b).grad_e4m3 = bool(args.grad_e4m3)
    host_in = {k: torch.from_numpy(inp[k].view(np.int16)).view(torch.bfloat16).pin_memory() for k in dev_in}
    for k, t in dev_in.items():
        t.copy_(host_in[k])
    del inp
    stream = torch.cuda.current_stream()
    lib = fq.load_library()

    def step():
        fwd(b)
        n = lib.fp8q_last_launch_count()
        if w.backward:
            bwd(b)
            n += lib.fp8q_last_launch_count()
        return n

    fq.get_status(clear=True)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    K = args.steps
    plan = step_work(w, args.recompute, args.bf16, args.mxfp8)
    # the per-launch CUDA events bracket every launch of a sample of the timed steps, spread evenly
    # over the region (steps 0, stride, 2 stride, ...): an event pair is about 2 us of stream work,
    # so tracing every step would itself lengthen the step by ~2 %
    traced_steps = max(1, min(K, args.trace_steps))
    stride = K // traced_steps
    if lib.fp8q_trace_start(traced_steps * len(plan)) != 0:
        raise RuntimeError("fp8q_trace_start failed")
    lib.fp8q_trace_stop()
    count = [0]

    def timed_step():
        i = count[0]
        count[0] += 1
        on = i % stride == 0 and i // stride < traced_steps
        if on:
            lib.fp8q_trace_resume()
        n = step()
        if on:
            lib.fp8q_trace_stop()
        return n

    launches = 0
    if flush_l2(w):
        # weights that fit (nearly) in L2: a 256 MB write between steps, outside the timed spans
        scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        with ClockSampler(local_rank) as clk:
            for e0, e1 in evs:
                scratch.fill_(1)
                e0.record(stream)
                launches += timed_step()
                e1.record(stream)
            torch.cuda.synchronize()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
        del scratch
    else:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local_rank) as clk:
            ev0.record(stream)
            for _ in range(K):
                launches += timed_step()
            ev1.record(stream)
            torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
    lib.fp8q_trace_stop()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    status = fq.get_status()

    import ctypes
    cap = K * len(plan)
    tms = (ctypes.c_float * cap)()
    kinds = (ctypes.c_int * cap)()
    n = lib.fp8q_trace_read(tms, kinds, cap)
    traced = [(lib.fp8q_kernel_name(kinds[i]).decode(), tms[i]) for i in range(max(n, 0))]

    ms = max_over_ranks(ms, dev)

    # ---- e2e: each step's inputs in from pinned host memory and its outputs back out, inside
    # the timed region.  "batch": the tensors a training step exchanges with the host -- the
    # activations and upstream gradients in, the block output and input gradients out -- with the
    # model state (weights, gains, weight gradients) resident in HBM; "all": every input and
    # output through the host, weights and fp32 weight gradients included.
    # ---- the same step captured once as a CUDA graph and replayed (the library takes every buffer
    # from the caller and never allocates, so a step is capturable); an extra figure, not the value
    graph = None
    if not args.no_graph and world == 1:
        try:
            graph = graph_replay(step, stream, K, flops, world)
        except Exception as exc:  # a capture the runtime refuses leaves the measured value untouched
            graph = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
            torch.cuda.synchronize()

    e2e = e2e_all = None
    if not args.no_e2e:
        batch_in = [k for k in ("x", "dY", "att", "dQKV") if k in dev_in]
        batch_out = [k for k in ("y", "dX", "d_att") if k in dev_out]
        host_out = {k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in dev_out.items()}
        Ke = max(3, K)  # as many steps as the device-timed region, under the same clocks
        # the second device set of the library's pipelined executor (step i+1's inputs arrive and
        # step i-1's outputs leave while step i computes); tensors that stay in HBM are shared
        if w.qkv:
            b2 = fq.BlockBuffers.allocate(w.T, w.d, w.f, w.qkv, device=dev, backward=w.backward, core=core,
                                          bf16=args.bf16)
            run, run_name = (lambda bb, steps: fq.block_run_steps(bb[0], bb[1], steps, backward=w.backward)), \
                "block_run_steps"
            state = ("g1", "W_qkv", "W_o", "g", "W_gu", "W_d") + (
                ("dW_qkv", "dW_o", "dg1", "dW_gu", "dW_d", "dg") if w.backward else ())
        else:
            b2 = fq.MlpBuffers.allocate(w.T, w.d, w.f, device=dev, backward=w.backward, bf16=args.bf16,
                                        mx=args.mxfp8)
            if w.backward:
                run, run_name = (lambda bb, steps: fq.mlp_block_run_steps(bb[0], bb[1], steps)), "mlp_block_run_steps"
            else:
                run, run_name = (lambda bb, steps: fq.mlp_block_fwd_run_steps(bb[0], bb[1], steps)), \
                    "mlp_block_fwd_run_steps"
            state = ("g", "W_gu", "W_d") + (("dW_gu", "dW_d", "dg") if w.backward else ())
        (b2.mlp if w.qkv else b2).recompute = bool(args.recompute)
        (b2.mlp if w.qkv else b2).grad_e4m3 = bool(args.grad_e4m3)
        b2_own = {k: buf_get(b2, k) for k in state}

        def measure(keys_in, keys_out):
            h2d = sum(host_in[k].numel() * host_in[k].element_size() for k in keys_in)
            d2h = sum(host_out[k].numel() * host_out[k].element_size() for k in keys_out)
            for k in state:
                buf_set(b2, k, b2_own[k] if k in keys_in or k in keys_out else buf_get(b, k))
            hio = {k: host_in[k] for k in keys_in}
            hio.update({k: host_out[k] for k in keys_out})
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            run((b, b2), [hio] * 2)
            torch.cuda.synchronize()
            e0.record(stream)
            run((b, b2), [hio] * Ke)
            e1.record(stream)
            torch.cuda.synchronize()
            ems = max_over_ranks(e0.elapsed_time(e1) / Ke, dev)
            return {"value": job_throughput(flops, world, ems) / 1e12, "unit": "TFLOP/s", "ms_per_step": ems,
                    "tokens_per_s": world * w.T / (ems * 1e-3), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "h2d": keys_in, "d2h": keys_out,
                    "mode": f"pipelined: {run_name} (step i+1's inputs in and step i-1's outputs out during step i)",
                    "steps": Ke}

        e2e = measure(batch_in, batch_out)
        e2e["resident"] = "model state (weights, gains, weight gradients) in HBM across steps"
        e2e_all = measure(list(dev_in), list(dev_out))
        del b2, b2_own
    return {"ms": ms, "K": K, "launches": launches, "traced": traced, "plan": plan, "clocks": clk.summary(),
            "status": status, "e2e": e2e, "e2e_all": e2e_all, "graph": graph, "w": w, "flops": flops}


def graph_replay(step, stream, K, flops, world):
    """The step captured once as a CUDA graph and replayed K times back to back."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg):
        step()
    cg.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(K):
        cg.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    gms = g0.elapsed_time(g1) / K
    return {"value": job_throughput(flops, world, gms) / 1e12, "unit": "TFLOP/s", "ms_per_step": gms, "steps": K,
            "note": "one step captured with torch.cuda.graph, replayed back to back (no L2 flush between replays)"}


L2_BYTES = 129e6


def weight_bytes(w):
    """bf16 weight bytes one step reads: W_gu, W_d (and W_qkv, W_o in the full block)."""
    return 2.0 * (3 * w.d * w.f + (w.d * w.qkv + w.d * w.d if w.qkv else 0))


def flush_l2(w):
    """Whether the timed steps flush L2 between them: when the weights alone would not keep the
    next step's reads out of L2 (less than twice its 129 MB)."""
    return weight_bytes(w) < 2 * L2_BYTES


_MLP_KEYS = ("g", "W_gu", "W_d", "dY", "y", "dW_gu", "dW_d", "dg")


def buf_get(b, k):
    """A tensor of MlpBuffers or BlockBuffers by its host-IO name (the block's MLP-side ones live
    in b.mlp)."""
    return getattr(b.mlp, k) if hasattr(b, "n_qkv") and k in _MLP_KEYS else getattr(b, k)


def buf_set(b, k, t):
    setattr(b.mlp if hasattr(b, "n_qkv") and k in _MLP_KEYS else b, k, t)


def kernel_table(traced, plan, K, pk):
    """Aggregate the traced launches by kernel and attach their algorithmic work."""
    rows = {}
    per = len(plan)
    total = sum(t for _, t in traced)
    for i, (name, t) in enumerate(traced):
        pname, pbytes, pflops = plan[i % per]
        r = rows.setdefault(name, {"launches": 0, "ms": 0.0, "bytes": 0.0, "flops": 0.0})
        r["launches"] += 1
        r["ms"] += t
        r["bytes"] += pbytes
        r["flops"] += pflops
    out = {}
    for name, r in rows.items():
        e = {"launches": r["launches"], "total_ms": round(r["ms"], 4), "share": round(r["ms"] / total, 4),
             "avg_us": round(1e3 * r["ms"] / r["launches"], 2)}
        if r["flops"]:
            e["tflops"] = round(r["flops"] / (r["ms"] * 1e-3) / 1e12, 1)
        else:
            e["gbs"] = round(r["bytes"] / (r["ms"] * 1e-3) / 1e9, 1)
            e["hbm_frac"] = round(e["gbs"] / pk["hbm_gbs"], 3)
        out[name] = e
    return out, total


def launch_positions(traced, plan):
    """Mean time of each launch position of the step over the timed steps, with its planned work."""
    per = len(plan)
    out = []
    for i, (pname, pbytes, pflops) in enumerate(plan):
        ts = [t for k, (_, t) in enumerate(traced) if k % per == i]
        us = 1e3 * sum(ts) / len(ts) if ts else 0.0
        out.append({"pos": i, "kernel": pname, "bytes": pbytes, "flops": pflops, "us": round(us, 2),
                    "gbs": round(pbytes / (us * 1e-6) / 1e9, 1) if us and not pflops else None,
                    "tflops": round(pflops / (us * 1e-6) / 1e12, 1) if us and pflops else None})
    return out


def precision_name(args) -> str:
    return "bf16 baseline" if args.bf16 else ("mxfp8 (block-scaled)" if args.mxfp8 else "fp8")


def cpu_baseline(w, tokens, grad_e4m3=False, bf16=False, mx=False):
    import oracle
    oracle.build()
    gf = oracle.E4M3 if grad_e4m3 else oracle.E5M2
    if w.qkv:
        inp = synth.block_inputs(w, seed=0)
        sl = {k: inp[k][:tokens] for k in ("x", "att", "dY", "dQKV") if k in inp}
        # with the attention core the sample is one sequence of `tokens` tokens
        core = (w.n_heads, w.n_kv_heads, 128, tokens) if w.n_heads else None
        t0 = time.perf_counter()
        oracle.full_block(sl["x"], inp["g1"], inp["W_qkv"], inp["W_o"], None if core else sl["att"], inp["g"],
                          inp["W_gu"], inp["W_d"], dY=sl.get("dY"), dQKV=None if core else sl.get("dQKV"),
                          nthreads=1, grad_fmt=gf, core=core, bf16=bf16)
        dt = time.perf_counter() - t0
    else:
        inp = synth.mlp_inputs(w, seed=0)
        x = inp["x"][:tokens]
        dY = inp["dY"][:tokens] if w.backward else None
        t0 = time.perf_counter()
        oracle.block(x, inp["g"], inp["W_gu"], inp["W_d"], dY=dY, nthreads=1, grad_fmt=gf, bf16=bf16, mx=mx)
        dt = time.perf_counter() - t0
    import dataclasses
    sub = dataclasses.replace(w, T=tokens, seq_len=tokens if w.n_heads else 0)
    core_note = f"; attention over one sequence of {tokens} tokens" if w.n_heads else ""
    return {"value": (sub.gemm_flops() + sub.attention_flops()) / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle", "seconds": round(dt, 2), "tokens_per_s": tokens / dt,
            "sample": f"{tokens} of {w.T} tokens of {w.name} with the full weights "
                      f"({'forward+backward' if w.backward else 'forward'}{core_note}), single-threaded oracle"}


def measure_fp8_peak():
    """Dense FP8 tensor throughput of the vendor library on this GPU, for context next to the
    derived peak: torch._scaled_mm (cuBLASLt) E4M3 x E4M3 -> bf16, 8192^3, tensor-wise scales.
    Burst: best of 10 single timed calls; sustained: back-to-back calls for 4 s."""
    import torch
    n = 8192
    g = torch.Generator(device="cuda").manual_seed(0)
    a = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device="cuda")
    mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    flop = 2.0 * n ** 3
    reps = max(1, int(4000.0 / best))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record()
        for _ in range(reps):
            mm()
        e1.record()
        torch.cuda.synchronize()
    sus = e0.elapsed_time(e1) / reps
    print(json.dumps({"fp8_cublaslt_tflops_burst": flop / (best * 1e-3) / 1e12,
                      "fp8_cublaslt_tflops_sustained": flop / (sus * 1e-3) / 1e12, "n": n, "reps": reps,
                      "clocks": clk.summary(), "torch": torch.__version__}))


def main():
    args = parse_args()
    if args.measure_fp8_peak:
        measure_fp8_peak()
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.BY_NAME[args.workload]
    if args.tokens:
        import dataclasses
        w = dataclasses.replace(w, T=args.tokens)
    if args.bf16 and (args.recompute or args.grad_e4m3):
        raise SystemExit("--bf16: without --recompute / --grad-e4m3")
    if args.mxfp8 and (args.bf16 or args.recompute or w.qkv):
        raise SystemExit("--mxfp8: an MLP workload, without --bf16 / --recompute")
    pk = peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        tokens = 2
        for _ in range(args.warmup):
            cpu_baseline(w, tokens, args.grad_e4m3, args.bf16, args.mxfp8)
        t0 = time.perf_counter()
        res = [cpu_baseline(w, tokens, args.grad_e4m3, args.bf16, args.mxfp8) for _ in range(args.steps)]
        dt = time.perf_counter() - t0
        import dataclasses
        sub = dataclasses.replace(w, T=tokens, seq_len=tokens if w.n_heads else 0)
        sub_flops = sub.gemm_flops() + sub.attention_flops()  # the work the sample does
        value = sub_flops * args.steps / dt / 1e12
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded Philox, bf16)",
                "config": {"workload": w.name, "T": w.T, "d": w.d, "f": w.f,
                           "gradients": "e4m3" if args.grad_e4m3 else "e5m2",
                           "precision": precision_name(args)},
                "cpu_baseline": {"kind": "oracle", "cores": 1, "value": value, "unit": "TFLOP/s",
                                 "sample": res[0]["sample"]},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    args.w = w
    r = run_ours(args, rank, world, local_rank)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    ms_step = r["ms"] / r["K"]
    value = job_throughput(r["flops"], world, ms_step) / 1e12
    kernels, traced_total = kernel_table(r["traced"], r["plan"], r["K"], pk)
    if args.launch_log:
        with open(args.launch_log, "w") as fh:
            json.dump(launch_positions(r["traced"], r["plan"]), fh, indent=1)
    gemm = {k: v for k, v in kernels.items() if k.startswith("gemm")}
    g_ms = sum(v["total_ms"] for v in gemm.values())
    g_launch = sum(v["launches"] for v in gemm.values())
    t_steps = len(r["traced"]) // len(r["plan"])  # the timed steps the trace bracketed
    g_flops = sum(fl for (name, _, fl) in r["plan"] if name.startswith("gemm")) * t_steps
    achieved = g_flops / (g_ms * 1e-3) / 1e12
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as fh:
            tj = json.load(fh)
        if tj.get("workload") == w.name and tj.get("T") == w.T and tj.get("kernel_hash") == kernel_hash() and not args.bf16 and not args.mxfp8:
            traffic = tj.get("bytes_per_launch")
    pick = choose_peak(pk, r["ms"], r["clocks"], bf16=args.bf16)
    peak = pick["peak"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": r["K"],
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 (bf16 operands, fp32 accumulation)" if args.bf16 else
                  "mxfp8 (e4m3/e5m2 operands with e8m0 scales per 32 elements, fp32 accumulation)" if args.mxfp8 else
                  "fp8 (e4m3/e5m2 operands, fp32 accumulation)"),
        "data": "synthetic (seeded Philox, bf16 inputs)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "f": w.f, "gemm_flops_per_step": w.gemm_flops(),
                   "attention_flops_per_step": w.attention_flops(),
                   "backward": "recompute H and a8 from n8 with the retained scale" if args.recompute else "stored H and a8",
                   "gradients": "bf16" if args.bf16 else ("e4m3" if args.grad_e4m3 else "e5m2"),
                   "precision": precision_name(args),
                   "l2": (f"L2 flushed between steps (a 256 MB write outside the timed spans; bf16 weights "
                          f"{weight_bytes(w) / 1e6:.0f} MB)" if flush_l2(w) else
                          f"inputs larger than L2 (bf16 weights {weight_bytes(w) / 1e6:.0f} MB read per step), no flush"),
                   "parallelism": "replicas" if world > 1 else "single"},
        "tokens_per_s": world * w.T / (ms_step * 1e-3),
        "pct_fp8_peak": round(100.0 * value / world / pick["fp8_peak"], 2),
        "roofline": {"kernel": "k_gemm_f8 / k_gemm_f8_wide (the six block GEMMs)", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "launches_per_step": g_launch // t_steps, "traced_steps": t_steps,
                     "share_of_step": round(g_ms / traced_total, 4),
                     "peak_kind": pick["kind"], "peak_source": pick["source"],
                     "frac_burst": round(achieved / pick["burst"], 4),
                     "frac_sustained": round(achieved / pick["sustained"], 4)},
        "kernels": kernels,
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "device_status": r["status"],
    }
    if r["e2e"]:
        line["e2e"] = r["e2e"]
        line["e2e_all_io"] = r["e2e_all"]
    if r["graph"]:
        line["graph_replay"] = r["graph"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_sample_tokens, args.grad_e4m3, args.bf16, args.mxfp8)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def choose_peak(pk, timed_ms, clocks, bf16=False):
    """The tensor peak that matches how the timed region ran.

    MEASURED_PEAKS.json holds a burst figure (a GEMM timed alone on a cool GPU) and a sustained one
    (seconds of back-to-back GEMMs under the power cap, at a lower clock).  A timed region shorter
    than a second, or one whose median SM clock stayed within 3 % of the maximum, ran at burst
    conditions and is held to the burst peak; a longer region that settled lower is held to the
    sustained peak.  FP8 peaks are the measured bf16 figures times the nominal dense FP8:BF16 ratio.
    """
    mult = 1.0 if bf16 else FP8_PER_BF16
    burst, sustained = pk["bf16"] * mult, pk["bf16_sustained"] * mult
    sm, sm_max = (clocks or {}).get("sm_mhz"), (clocks or {}).get("sm_max_mhz")
    at_max = sm is not None and sm_max and sm >= 0.97 * sm_max
    kind = "burst" if (timed_ms < 1000.0 or at_max) else "sustained"
    peak = burst if kind == "burst" else sustained
    what = "bf16" if bf16 else "bf16 x nominal fp8/bf16 2"
    src = (f"{pk['source']} {kind}: {what} = {peak:.1f} TFLOP/s (timed region {timed_ms:.0f} ms, "
           f"median SM clock {sm} of {sm_max} MHz)")
    return {"peak": peak, "kind": kind, "burst": burst, "sustained": sustained, "source": src,
            "fp8_peak": (pk["bf16"] if kind == "burst" else pk["bf16_sustained"]) * FP8_PER_BF16}


def kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for name in ("fp8q_gemm.cu", "fp8q_common.cuh"):
        with open(os.path.join(ROOT, "fp8_absmax_reduce_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
