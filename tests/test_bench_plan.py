"""bench.py's per-launch work plan (CPU, no GPU): the plan maps every traced launch of a step to
its algorithmic bytes and FLOPs, from which the bench derives the roofline and the per-kernel
table, so it must stay in step with the library and the workloads.
  * every plan entry names a kernel kind the library's trace reports;
  * the GEMM FLOPs of a step add up to the workload's algorithmic count (6Tdf forward, 18Tdf
    forward + backward, plus the QKV and O projections), in every precision mode (per-tensor FP8,
    BF16, block-scaled MXFP8 for the MLP workloads); the recompute
    mode adds exactly one gate/up GEMM of executed work;
  * --launch-log folds the traced launches of K steps onto the plan's positions;
  * the attention kernels' executed FLOPs are 18 products per causal pair and head against the
    algorithmic 14 (the backward kernels recompute S and dP), 128 x 2 FLOPs each.
"""

import dataclasses

import pytest

import bench
import synth


@pytest.fixture(scope="module")
def kernel_names():
    from fp8_absmax_reduce_gb300 import build as b
    b.build()
    import fp8_absmax_reduce_gb300 as fq
    lib = fq.load_library()
    names = set()
    for k in range(64):
        n = lib.fp8q_kernel_name(k).decode()
        if n != "unknown":
            names.add(n)
    return names


def modes(w):
    out = [dict()]
    if w.backward:
        out += [dict(recompute=True)]
    out += [dict(bf16=True)]
    if not w.qkv:
        out += [dict(mx=True)]
    return out


@pytest.mark.parametrize("w", synth.WORKLOADS, ids=lambda w: w.name)
def test_plan_names_are_library_kernels(w, kernel_names):
    for m in modes(w):
        plan = bench.step_work(w, **m)
        assert plan
        for name, nbytes, flops in plan:
            assert name in kernel_names, (w.name, m, name)
            assert nbytes > 0 and flops >= 0


@pytest.mark.parametrize("w", synth.WORKLOADS, ids=lambda w: w.name)
def test_plan_gemm_flops_match_the_workload(w):
    T, d, f = w.T, w.d, w.f
    for m in modes(w):
        plan = bench.step_work(w, **m)
        gemm = sum(fl for name, _, fl in plan if name.startswith("gemm"))
        want = w.gemm_flops() + (2.0 * T * d * 2 * f if m.get("recompute") else 0.0)
        assert gemm == pytest.approx(want, rel=1e-12), (w.name, m)


def test_plan_attention_flops():
    w = synth.BY_NAME["32b-block-attn-fwd-bwd"]
    for m in (dict(), dict(bf16=True)):
        plan = bench.step_work(w, **m)
        attn = sum(fl for name, _, fl in plan if name.startswith("attn"))
        assert attn == pytest.approx(w.attention_flops() * 18 / 14, rel=1e-12)
    fwd_only = dataclasses.replace(w, dy_std=0.0)
    plan = bench.step_work(fwd_only)
    attn = sum(fl for name, _, fl in plan if name.startswith("attn"))
    assert attn == pytest.approx(fwd_only.attention_flops(), rel=1e-12)


def test_attention_flops_closed_form():
    """S(S+1)/2 causal pairs per sequence and head, 128 x 2 FLOPs per pair and product."""
    w = dataclasses.replace(synth.BY_NAME["32b-block-attn-fwd-bwd"], T=8, seq_len=4, n_heads=2)
    pairs = 2 * (4 * 5 // 2)  # two sequences of 4 tokens
    assert w.attention_flops() == pairs * 2 * 256 * 7
    assert dataclasses.replace(w, dy_std=0.0).attention_flops() == pairs * 2 * 256 * 2


def test_peak_follows_the_run():
    """A short timed region, or one held at the maximum clock, is held to the burst peak; a long
    one that settled lower to the sustained peak; FP8 peaks are twice the bf16 ones."""
    import bench
    pk = {"bf16": 1900.0, "bf16_sustained": 1700.0, "source": "measured"}
    short = bench.choose_peak(pk, 300.0, {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0})
    assert short["kind"] == "burst" and short["peak"] == 3800.0 and short["fp8_peak"] == 3800.0
    at_max = bench.choose_peak(pk, 5000.0, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert at_max["kind"] == "burst"
    capped = bench.choose_peak(pk, 5000.0, {"sm_mhz": 1700.0, "sm_max_mhz": 2070.0})
    assert capped["kind"] == "sustained" and capped["peak"] == 3400.0
    assert bench.choose_peak(pk, 5000.0, {"sm_mhz": 1700.0, "sm_max_mhz": 2070.0}, bf16=True)["peak"] == 1700.0
    assert bench.choose_peak(pk, 5000.0, None)["kind"] == "sustained"


def test_launch_positions_average_each_position():
    """--launch-log: the traced launches of K steps fold onto the plan's positions, one mean per
    position, with the rates from the plan's bytes or FLOPs."""
    plan = [("quant_cast", 2e9, 0), ("gemm_x", 1e9, 4e12)]
    traced = [("quant_cast", 1.0), ("gemm_x", 2.0), ("quant_cast", 3.0), ("gemm_x", 4.0)]  # ms, two steps
    out = bench.launch_positions(traced, plan)
    assert [o["pos"] for o in out] == [0, 1]
    assert out[0]["us"] == 2000.0 and out[1]["us"] == 3000.0
    assert out[0]["gbs"] == pytest.approx(2e9 / 2e-3 / 1e9, abs=0.1) and out[0]["tflops"] is None
    assert out[1]["tflops"] == pytest.approx(4e12 / 3e-3 / 1e12, abs=0.1) and out[1]["gbs"] is None
