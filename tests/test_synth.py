"""The seeded input generator: determinism, independence of streams, bf16 rounding, workload shapes."""

import numpy as np

import synth


def test_deterministic_and_independent():
    a = synth.normal_bf16((64, 32), 0.02, seed=0, tensor_id=synth.TID_WGU)
    b = synth.normal_bf16((64, 32), 0.02, seed=0, tensor_id=synth.TID_WGU)
    c = synth.normal_bf16((64, 32), 0.02, seed=0, tensor_id=synth.TID_WD)
    d = synth.normal_bf16((64, 32), 0.02, seed=1, tensor_id=synth.TID_WGU)
    assert (a == b).all() and (a != c).mean() > 0.9 and (a != d).mean() > 0.9


def test_bf16_rounding_is_nearest_even():
    v = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20, -2.5, 0.0], dtype=np.float32)
    assert list(synth.bf16_bits(v)) == [0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000]
    back = synth.f32_from_bf16_bits(synth.bf16_bits(v))
    assert back[3] == -2.5


def test_workload_inputs():
    w = synth.BY_NAME["3b-mlp-fwd"]
    inp = synth.mlp_inputs(w, T=64, d=2048, f=128)
    assert inp["x"].shape == (64, 2048) and inp["W_gu"].shape == (2048, 256) and "dY" not in inp
    x = synth.f32_from_bf16_bits(inp["x"]).astype(np.float64)
    ch = synth.outlier_channels(2048, 0.01, 0, synth.TID_OUTLIER)
    assert ch.size == 20
    big = np.abs(x[:, ch]).mean() / np.abs(np.delete(x, ch, axis=1)).mean()
    assert 15 < big < 25
    g = synth.f32_from_bf16_bits(inp["g"])
    assert abs(g.mean() - 1) < 0.02 and 0.08 < g.std() < 0.12
    assert synth.WORKLOADS[2].gemm_flops() == 18.0 * 8192 * 3584 * 18944
