"""GPU parity at the workloads' full sizes against the oracle, in the launch configuration bench.py
times (mlp_block_fwd + mlp_block_bwd, or block_fwd + block_bwd, on the whole workload).

The oracle's results for these sizes come from tests/golden/fullsize/<workload>.npz, written by
tests/golden/fullsize_digests.py from the oracle alone (multi-threaded over output rows; the
same bits as one thread).  The test first checks that the seeded inputs it rebuilt are the ones
the digest was computed from (SHA-256 of every input tensor), then compares:
  * bit for bit on the full tensors (SHA-256): every quantizer whose input is a given tensor --
    W_gu8, W_d8, n8 and rstd of the MLP workloads, dY8; in the 32B-class block W_qkv8, W_o8, n1_8,
    rstd1, att8, W_gu8, W_d8, dY8, dQKV8 -- and their scale triples;
  * the in-block requantizations (a8, dH8; in the 32B block also n8 of h and dh8) on sampled rows:
    >= 99.9 % identical codes, every other one a step away, amax within one bf16 step;
  * every GEMM output and gradient on sampled rows (token rows on both sides of the tile and
    rasterisation-group edges; rows of each weight gradient) and the full gain gradients: max
    row-relative L2 error 2e-3 for block outputs, 5e-3 for gradients;
  * the block-scaled MXFP8 7B-class block: its quantizations of given tensors (weights, n, dY, both
    block directions) bit for bit with their E8M0 scales; the requantized a and dH per block:
    >= 99.9 % equal scales, and inside those >= 99.9 % identical codes, the rest a step away or,
    for values small against their block, within 2.5e-3 of the format's maximum in units of the
    block scale;
plus two whole-tensor relations only the GPU's own tensors can give: the scale of dH (and dh) is
fmax over the absmax of the stored bf16 tensor.
"""

import hashlib
import os

import numpy as np
import pytest
import torch

import fp8_absmax_reduce_gb300 as fq
import synth
from tests._gpu import code_step_diff, dev_bf16, fp8_table, row_rel

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fullsize")


def sha(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def digest(name, inp):
    D = np.load(os.path.join(GOLD, name + ".npz"))
    for k, v in inp.items():
        assert sha(v) == str(D[f"sha_in_{k}"]), (
            f"input {k} is not the one the digest was computed from (numpy {np.__version__} here, "
            f"{D['numpy_version']} there)")
    return D


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_vals(b: np.ndarray) -> np.ndarray:
    return synth.f32_from_bf16_bits(b).astype(np.float64)


def rows_of(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    return t[torch.from_numpy(rows).to(t.device)]


def requant(got, ref, got_amax, ref_amax, second_level=False):
    """In-block requantization: the amax within one bf16 step (the GEMM-produced input may differ in
    its last bit); with equal scales >= 99.9 % identical codes, every other one step away.  A second
    level (codes of a tensor computed from first-level codes: a8 of the 32B block, whose H comes
    from n8 of h) keeps >= 99.9 % identical codes, the others free."""
    assert abs(float(got_amax) / float(ref_amax) - 1.0) <= 2.0 ** -7, (got_amax, ref_amax)
    steps = code_step_diff(got, ref)
    same = (steps == 0).mean()
    if second_level:
        assert same >= 0.999, same
    elif got_amax == ref_amax:
        assert same >= 0.999 and steps.max() <= 1, (same, steps.max())
    else:  # every code shifts by at most a step when the scale moved by a bf16 ulp
        assert steps.max() <= 1, steps.max()


def bf16_absmax(b: np.ndarray) -> float:
    """Exact max |v| of bf16 bit patterns (integer max of the magnitude bits: non-negative floats
    order like their bit patterns)."""
    m = int((b.reshape(-1) & np.uint16(0x7FFF)).max())
    return float(synth.f32_from_bf16_bits(np.array([m], np.uint16))[0])


@pytest.mark.parametrize("wname", ["3b-mlp-fwd", "7b-mlp-fwd-bwd", "14b-mlp-fwd-bwd"])
def test_full_size_mlp_block(wname):
    w = synth.BY_NAME[wname]
    T, d, f = w.T, w.d, w.f
    inp = synth.mlp_inputs(w, seed=0)
    D = digest(wname, inp)
    b = fq.MlpBuffers.allocate(T, d, f, backward=w.backward, keep_intermediates=True)
    for k in ("x", "g", "W_gu", "W_d") + (("dY",) if w.backward else ()):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    if w.backward:
        fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    scal = b.scal.cpu().numpy()
    rows = D["rows"]

    # bit-exact on full tensors
    assert sha(b.W_gu8.cpu().numpy()) == str(D["sha_Wgu8"])
    assert sha(b.W_d8.cpu().numpy()) == str(D["sha_Wd8"])
    assert sha(b.n8.cpu().numpy()) == str(D["sha_n8"])
    assert sha(b.rstd.cpu().numpy()) == str(D["sha_rstd"])
    np.testing.assert_array_equal(scal[:3], D["scal_fwd"][:3])
    # the gate/up GEMM, SwiGLU requantization, the down GEMM + residual
    assert row_rel(bf16_vals(bits(rows_of(b.H, rows))), bf16_vals(D["H"])) < 2e-3
    requant(rows_of(b.a8, rows).cpu().numpy(), D["a8"], scal[3, 0], D["scal_fwd"][3, 0])
    assert row_rel(bf16_vals(bits(rows_of(b.y, rows))), bf16_vals(D["y"])) < 2e-3
    if not w.backward:
        return
    assert sha(b.dY8.cpu().numpy()) == str(D["sha_dY8"])
    np.testing.assert_array_equal(scal[4], D["scal_bwd"][0])
    assert row_rel(bf16_vals(bits(rows_of(b.dH, rows))), bf16_vals(D["dH"])) < 5e-3
    dH_bits = bits(b.dH)
    assert scal[5, 0] == np.float32(bf16_absmax(dH_bits))            # exact: the stored bf16 dH
    assert scal[5, 1] == np.float32(57344.0) / np.float32(scal[5, 0])
    del dH_bits
    requant(rows_of(b.dH8, rows).cpu().numpy(), D["dH8"], scal[5, 0], D["scal_bwd"][1, 0])
    assert row_rel(rows_of(b.dN, rows).cpu().numpy().astype(np.float64), D["dN"].astype(np.float64)) < 5e-3
    assert row_rel(bf16_vals(bits(rows_of(b.dX, rows))), bf16_vals(D["dX"])) < 5e-3
    assert row_rel(rows_of(b.dW_d, D["rows_dWd"]).cpu().numpy().astype(np.float64),
                   D["dWd"].astype(np.float64)) < 5e-3
    assert row_rel(rows_of(b.dW_gu, D["rows_dWgu"]).cpu().numpy().astype(np.float64),
                   D["dWgu"].astype(np.float64)) < 5e-3
    assert row_rel(b.dg.cpu().numpy()[None, :].astype(np.float64), D["dg"][None, :].astype(np.float64)) < 5e-3


def test_full_size_32b_block():
    w = synth.BY_NAME["32b-block-fwd-bwd"]
    T, d, f, nq = w.T, w.d, w.f, w.qkv
    inp = synth.block_inputs(w, seed=0)
    D = digest(w.name, inp)
    b = fq.BlockBuffers.allocate(T, d, f, nq, keep_intermediates=True)
    for k, t in (("x", b.x), ("g1", b.g1), ("W_qkv", b.W_qkv), ("W_o", b.W_o), ("att", b.att), ("g", b.mlp.g),
                 ("W_gu", b.mlp.W_gu), ("W_d", b.mlp.W_d), ("dY", b.mlp.dY), ("dQKV", b.dQKV)):
        t.copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.block_fwd(b)
    fq.block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    sa, sm = b.scal.cpu().numpy(), b.mlp.scal.cpu().numpy()
    rows, rd, rg = D["rows"], D["rows_dWd"], D["rows_dW"]
    # bit-exact on full tensors: quantizers of given tensors, the attention-side RMSNorm
    for name, t in (("Wqkv8", b.W_qkv8), ("Wo8", b.W_o8), ("n1_8", b.n1_8), ("att8", b.att8), ("rstd1", b.rstd1),
                    ("Wgu8", b.mlp.W_gu8), ("Wd8", b.mlp.W_d8), ("dY8", b.mlp.dY8), ("dqkv8", b.dQKV8)):
        assert sha(t.cpu().numpy()) == str(D["sha_" + name]), name
    np.testing.assert_array_equal(sa[[0, 1, 2, 3, 5]], D["scal_attn"][[0, 1, 2, 3, 5]])
    np.testing.assert_array_equal(sm[[0, 1, 4]], np.concatenate([D["scal_fwd"][:2], D["scal_bwd"][:1]]))
    f32 = lambda t, r: rows_of(t, r).cpu().numpy().astype(np.float64)
    # attention side forward
    assert row_rel(bf16_vals(bits(rows_of(b.qkv, rows))), bf16_vals(D["qkv"])) < 2e-3
    assert row_rel(bf16_vals(bits(rows_of(b.h, rows))), bf16_vals(D["h"])) < 2e-3
    # the MLP on h (a GEMM output: n8 and a8 are requantizations of it)
    requant(rows_of(b.mlp.n8, rows).cpu().numpy(), D["n8"], sm[2, 0], D["scal_fwd"][2, 0])
    assert row_rel(bf16_vals(bits(rows_of(b.mlp.H, rows))), bf16_vals(D["H"])) < 5e-3
    requant(rows_of(b.mlp.a8, rows).cpu().numpy(), D["a8"], sm[3, 0], D["scal_fwd"][3, 0], second_level=True)
    assert row_rel(bf16_vals(bits(rows_of(b.mlp.y, rows))), bf16_vals(D["y"])) < 2e-3
    # backward
    assert row_rel(bf16_vals(bits(rows_of(b.mlp.dH, rows))), bf16_vals(D["dH"])) < 5e-3
    requant(rows_of(b.mlp.dH8, rows).cpu().numpy(), D["dH8"], sm[5, 0], D["scal_bwd"][1, 0])
    assert row_rel(f32(b.mlp.dN, rows), D["dN"].astype(np.float64)) < 5e-3
    assert row_rel(bf16_vals(bits(rows_of(b.dh, rows))), bf16_vals(D["dh"])) < 5e-3
    dh_bits = bits(b.dh)
    assert sa[4, 0] == np.float32(bf16_absmax(dh_bits))
    assert sa[4, 1] == np.float32(57344.0) / np.float32(sa[4, 0])
    del dh_bits
    requant(rows_of(b.dh8, rows).cpu().numpy(), D["dh8"], sa[4, 0], D["scal_attn"][4, 0])
    assert row_rel(bf16_vals(bits(rows_of(b.d_att, rows))), bf16_vals(D["d_att"])) < 5e-3
    assert row_rel(bf16_vals(bits(rows_of(b.dX, rows))), bf16_vals(D["dX"])) < 5e-3
    # weight gradients fed by a requantized operand: one flipped code of relative step <= 2^-3
    # moves a row (a sum over T tokens) by about 2^-3 / sqrt(T)
    tol_w = max(5e-3, 2.0 ** -3 / np.sqrt(T))
    assert row_rel(f32(b.mlp.dW_d, rd), D["dWd"].astype(np.float64)) < tol_w
    assert row_rel(f32(b.mlp.dW_gu, rg), D["dWgu"].astype(np.float64)) < tol_w
    assert row_rel(f32(b.dW_o, rg), D["dWo"].astype(np.float64)) < tol_w
    assert row_rel(f32(b.dW_qkv, rg), D["dWqkv"].astype(np.float64)) < 5e-3
    assert row_rel(b.mlp.dg.cpu().numpy()[None, :].astype(np.float64), D["dg"][None, :].astype(np.float64)) < 5e-3
    assert row_rel(b.dg1.cpu().numpy()[None, :].astype(np.float64), D["dg1"][None, :].astype(np.float64)) < 5e-3


def mx_plain_sf(sf_chunked: torch.Tensor, R: int, C: int, along_rows: bool) -> np.ndarray:
    """GPU scales (chunked layout) -> the oracle's plain layout: [R, C/32] for blocks along a row,
    [R/32, C] for blocks down a column."""
    from tests._gpu import mx_sf_from_chunked
    sf = sf_chunked.cpu().numpy()
    return mx_sf_from_chunked(sf, C, R).T if along_rows else mx_sf_from_chunked(sf, R, C)


def mx_requant(q, rq, sf, rsf, block_of, fmt):
    """Requantized MX codes (their input is a GEMM output): >= 99.9 % of the blocks have the oracle's
    scale (the others one power of two away); inside the blocks whose scales agree >= 99.9 % identical
    codes, and the others a step away or, for small values, within 2.5e-3 of the format's maximum in
    units of the block scale.  The bound follows the GEMM's own tolerance: its output is right to
    5e-3 of a row's magnitude, not of each element (the tensor core's accumulation is not the
    oracle's fp64 sum), and a block's maximum is at least half the format's maximum, so a value
    much smaller than its block's maximum can land several codes away.  block_of maps each code to
    its block's index in sf."""
    sd = np.abs(sf.astype(int) - rsf.astype(int))
    assert (sd == 0).mean() >= 0.999 and sd.max() <= 1, ((sd == 0).mean(), sd.max())
    agree = (sd == 0).ravel()[block_of]
    qa, ra = q.ravel()[agree], np.asarray(rq).ravel()[agree]
    steps = code_step_diff(qa, ra)
    assert (steps == 0).mean() >= 0.999, (steps == 0).mean()
    tab = fp8_table(fmt)
    far = steps > 1
    gap = np.abs(tab[qa[far]] - tab[ra[far]])
    fmax = 448.0 if fmt == 0 else 57344.0
    assert np.all(gap <= 2.5e-3 * fmax), (int(steps.max()), float(gap.max()) if gap.size else 0.0)


def test_full_size_mlp_block_mxfp8():
    """The block-scaled MXFP8 7B-class block against the oracle's full-size MX results."""
    w = synth.BY_NAME["7b-mlp-fwd-bwd"]
    T, d, f = w.T, w.d, w.f
    inp = synth.mlp_inputs(w, seed=0)
    D = digest("7b-mlp-fwd-bwd-mx", inp)
    b = fq.MlpBuffers.allocate(T, d, f, backward=True, keep_intermediates=True, mx=True)
    for k in ("x", "g", "W_gu", "W_d", "dY"):
        getattr(b, k).copy_(dev_bf16(inp[k]))
    fq.get_status(clear=True)
    fq.mlp_block_fwd(b)
    fq.mlp_block_bwd(b)
    torch.cuda.synchronize()
    assert fq.get_status() == 0
    assert sha(b.rstd.cpu().numpy()) == str(D["sha_rstd"])
    shapes = {"W_gu": (d, 2 * f), "W_d": (f, d), "n": (T, d), "a": (T, f), "dY": (T, d), "dH": (T, 2 * f)}
    okey = {"W_gu": "Wgu", "W_d": "Wd", "n": "n", "a": "a", "dY": "dY", "dH": "dH"}
    fmts = {"a": 0, "dH": 1}  # E4M3 activations, E5M2 gradients
    rows, blocks = D["rows"], D["col_blocks"]
    for slot in fq.MX_SLOTS:
        name, ax = slot.rsplit("_", 1)
        R, C = shapes[name]
        q, sfc = b.mx[slot]
        key = f"mx_{okey[name]}_{ax}"
        if name in ("W_gu", "W_d", "n", "dY"):
            assert sha(q.cpu().numpy()) == str(D["sha_" + key]), slot
            assert sha(mx_plain_sf(sfc, R, C, ax == "c")) == str(D["sha_" + key + "_sf"]), slot
            continue
        sf = mx_plain_sf(sfc, R, C, ax == "c")
        qr = rows_of(q, rows).cpu().numpy()
        if ax == "r":   # blocks along the row: block (i, j // 32) of sampled row i
            block_of = (np.arange(len(rows))[:, None] * (C // 32) + np.arange(C)[None, :] // 32).ravel()
            mx_requant(qr, D[key], sf[rows], D[key + "_sf"], block_of, fmts[name])
        else:           # blocks down a column: block (row // 32, j)
            pos = np.searchsorted(blocks, rows // 32)
            block_of = (pos[:, None] * C + np.arange(C)[None, :]).ravel()
            mx_requant(qr, D[key], sf[blocks], D[key + "_sf"], block_of, fmts[name])
    assert row_rel(bf16_vals(bits(rows_of(b.H, rows))), bf16_vals(D["H"])) < 2e-3
    assert row_rel(bf16_vals(bits(rows_of(b.y, rows))), bf16_vals(D["y"])) < 2e-3
    assert row_rel(bf16_vals(bits(rows_of(b.dH, rows))), bf16_vals(D["dH"])) < 5e-3
    assert row_rel(rows_of(b.dN, rows).cpu().numpy().astype(np.float64), D["dN"].astype(np.float64)) < 5e-3
    assert row_rel(bf16_vals(bits(rows_of(b.dX, rows))), bf16_vals(D["dX"])) < 5e-3
    assert row_rel(rows_of(b.dW_d, D["rows_dWd"]).cpu().numpy().astype(np.float64),
                   D["dWd"].astype(np.float64)) < 5e-3
    assert row_rel(rows_of(b.dW_gu, D["rows_dWgu"]).cpu().numpy().astype(np.float64),
                   D["dWgu"].astype(np.float64)) < 5e-3
    assert row_rel(b.dg.cpu().numpy()[None, :].astype(np.float64), D["dg"][None, :].astype(np.float64)) < 5e-3
