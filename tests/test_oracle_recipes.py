"""Pins of the oracle's recipes against the pages' worked examples, closed
forms, invariants and reductions to already-pinned pieces.

Each test is chosen so that a plausible slip (a swapped Fmax, s = alpha
instead of 1/alpha, a wrong emax, a transposed index, a wrong block
boundary, a nibble order flip) fails it.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def f32(v):
    return np.asarray(v, np.float32)


def dec8(c, fmt=O.E4M3):
    """Decode via torch (library), not via the oracle."""
    dt = torch.float8_e4m3fn if fmt == O.E4M3 else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(dt).float().numpy()


E2M1_VALUES = np.array(gold("e2m1_values.json")["values"], np.float32)


def dec4(nibbles):
    return E2M1_VALUES[np.asarray(nibbles, np.int64)]


# ---------------------------------------------------------------------------
# per-tensor current scaling
# ---------------------------------------------------------------------------

def test_cs_worked_example():
    g = gold("cs_worked_example.json")
    x = f32([g["x"]])
    r = O.current_scaling(x, O.E4M3, rowwise=True, colwise=True)
    assert r.amax == g["amax"]
    alpha, s = O.cs_scale(r.amax, O.E4M3)
    assert alpha == np.float32(g["alpha"])                # 448 / 1000 in FP32
    assert np.array_equal(dec8(r.q_row)[0], f32(g["q"]))
    assert np.array_equal(r.q_colT[:, 0], r.q_row[0])
    assert abs(float(r.scale) - g["s_approx"]) < g["s_tol"]
    assert r.scale == np.float32(1) / np.float32(g["alpha"])
    xhat = O.dq_current_scaling(r.q_row, r.scale)[0]
    assert np.allclose(xhat, g["xhat_approx"], rtol=g["xhat_tol"], atol=0)
    # scaled values before the cast
    assert np.allclose(alpha * x[0], g["scaled"], rtol=1e-6)


def test_cs_error_example():
    g = gold("cs_error_example.json")
    w = gold("cs_worked_example.json")
    x = f32([w["x"]])
    r = O.current_scaling(x)
    alpha, _ = O.cs_scale(r.amax)
    q = dec8(r.q_row)[0, 1]
    assert abs((q - alpha * np.float32(g["x"])) - g["scaled_error"]) < g["tol"]
    xhat = O.dq_current_scaling(r.q_row, r.scale)[0, 1]
    assert abs((xhat - g["x"]) - g["restored_error_approx"]) < g["tol"]
    rel_scaled = abs(q - alpha * g["x"]) / abs(alpha * g["x"])
    rel_restored = abs(xhat - g["x"]) / g["x"]
    assert abs(rel_scaled - g["relative_error_approx"]) < g["tol"]
    assert abs(rel_restored - g["relative_error_approx"]) < g["tol"]


def test_cs_underflow_and_cancellation_examples():
    g = gold("cs_underflow_example.json")
    r = O.current_scaling(f32([g["x"]]))
    assert np.array_equal(dec8(r.q_row)[0], f32(g["q_expected"]))
    c = gold("cs_cancellation_example.json")
    # the two inputs sit in a tensor whose amax is 1000 (alpha = 0.448)
    r = O.current_scaling(f32([c["x"]]))
    xhat = O.dq_current_scaling(r.q_row, r.scale)[0]
    assert c["x"][1] - c["x"][0] == c["true_difference"]
    assert xhat[1] - xhat[0] == c["quantized_difference"]


def test_cs_multi_rank_amax_example():
    g = gold("multi_rank_amax.json")
    shards = [f32([s]) for s in g["shards"]]
    local = [O.amax(s) for s in shards]
    assert local == g["local_amax"]
    glob = max(local)
    assert glob == g["global_amax"]
    alpha, _ = O.cs_scale(glob)
    assert alpha == np.float32(448) / np.float32(100) and abs(alpha - g["alpha"]) < 1e-6
    # quantizing each shard with the global amax equals quantizing the whole tensor
    whole = O.current_scaling(np.concatenate(shards, axis=1))
    parts = [O.current_scaling(s, amax_in=glob) for s in shards]
    assert np.array_equal(np.concatenate([p.q_row for p in parts], axis=1), whole.q_row)
    assert all(p.scale == whole.scale for p in parts)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_cs_row_sharding_invariance(fmt):
    """The quantized tensor must not depend on how rows are split across ranks
    once the amax is MAX-reduced ("Mixed-precision training: fp16 to fp8",
    section "FP8 communication", TP all-gather)."""
    x = W.gen("grad" if fmt == O.E5M2 else "normal", (96, 64), 5, bf16=True)
    whole = O.current_scaling(x, fmt, rowwise=True, colwise=True)
    cuts = [0, 16, 48, 96]
    shards = [x[a:b] for a, b in zip(cuts[:-1], cuts[1:])]
    glob = max(O.amax(s) for s in shards)
    parts = [O.current_scaling(s, fmt, rowwise=True, colwise=True, amax_in=glob) for s in shards]
    assert np.array_equal(np.concatenate([p.q_row for p in parts], 0), whole.q_row)
    assert np.array_equal(np.concatenate([p.q_colT for p in parts], 1), whole.q_colT)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_cs_power_of_two_invariance(fmt):
    """Relative error is scale-invariant ("FP8 Current Scaling ...", section
    "Does scaling amplify the error"): x * 2^k gives the same codes and
    s * 2^k exactly."""
    x = W.gen("outliers", (64, 48), 9, bf16=False)
    base = O.current_scaling(x, fmt)
    for k in (-20, -3, 1, 7, 30):
        r = O.current_scaling((x * np.float32(2.0 ** k)).astype(np.float32), fmt)
        assert np.array_equal(r.q_row, base.q_row)
        assert r.scale == base.scale * np.float32(2.0 ** k)
        assert r.amax == base.amax * np.float32(2.0 ** k)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_cs_codes_are_nearest_of_scaled_values(fmt):
    """q_i is the saturated nearest code of the FP32 product alpha * x_i,
    alpha = Fmax / amax; the nearest code is found by search over
    torch-decoded codes."""
    x = W.gen("outliers", (32, 40), 3, bf16=True)
    r = O.current_scaling(x, fmt, colwise=True)
    xf = W.bf16_bits_to_f32(x)
    fmax = np.float32(448.0 if fmt == O.E4M3 else 57344.0)
    alpha = fmax / np.float32(np.abs(xf).max())
    y = (alpha * xf).astype(np.float32).ravel()
    table = dec8(np.arange(256, dtype=np.uint8), fmt).astype(np.float64)
    fin = np.isfinite(table)
    got = dec8(r.q_row, fmt).astype(np.float64).ravel()
    best = np.abs(table[fin][None, :] - y[:, None]).min(axis=1)
    assert np.all(np.abs(got - y) == best)
    assert np.array_equal(r.q_colT, r.q_row.T)
    assert r.scale == np.float32(1) / alpha
    assert np.abs(got).max() == fmax


def test_cs_zero_tensor_scale_one():
    r = O.current_scaling(np.zeros((4, 8), np.float32))
    assert r.amax == 0 and r.scale == 1
    assert not r.q_row.any()


@pytest.mark.parametrize("out", [O.F32, O.BF16])
def test_cs_dequant_closed_form(out):
    x = W.gen("normal", (16, 32), 1, bf16=True)
    r = O.current_scaling(x, O.E5M2)
    y = O.dq_current_scaling(r.q_row, r.scale, O.E5M2, out)
    want = (dec8(r.q_row, O.E5M2) * r.scale).astype(np.float32)
    if out == O.BF16:
        want = W.to_bf16_bits(want)
    assert np.array_equal(y, want)


# ---------------------------------------------------------------------------
# MXFP8
# ---------------------------------------------------------------------------

def _mx_closed_form_codes(blocks, emax):
    """Scale code per block from numpy's frexp: floor(log2 b) = exponent - 1."""
    b = np.abs(blocks.astype(np.float64)).max(axis=-1)
    _, e = np.frexp(b)
    code = np.clip(e - 1 - emax + 127, 0, 254)
    return np.where(b == 0, 127, code).astype(np.uint8)


@pytest.mark.parametrize("fmt,emax", [(O.E4M3, 8), (O.E5M2, 15)])
def test_mx_scale_closed_form_and_block_range(fmt, emax):
    x = W.gen("lognormal_rows", (64, 128), 1, bf16=True)
    xf = W.bf16_bits_to_f32(x)
    r = O.mxfp8(x, fmt)
    assert np.array_equal(r.e8m0_row, _mx_closed_form_codes(xf.reshape(64, 4, 32), emax))
    assert np.array_equal(r.e8m0_col, _mx_closed_form_codes(xf.reshape(2, 32, 128).transpose(0, 2, 1), emax))
    # the block maximum lands in [2^emax, 2^(emax+1)) before saturation, so its code
    # magnitude lies in [256, 448] for E4M3 and [32768, 57344] for E5M2
    q = np.abs(dec8(r.q_row, fmt).reshape(64, 4, 32)).max(axis=-1)
    assert np.all(q >= 2.0 ** emax) and np.all(q <= (448.0 if fmt == O.E4M3 else 57344.0))


def test_mx_power_of_two_invariance_and_symmetry():
    x = W.gen("normal", (64, 96), 2, bf16=False)
    r = O.mxfp8(x)
    for k in (-9, 5):
        r2 = O.mxfp8((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(r2.q_row, r.q_row) and np.array_equal(r2.q_col, r.q_col)
        assert np.array_equal(r2.e8m0_row.astype(int), r.e8m0_row.astype(int) + k)
        assert np.array_equal(r2.e8m0_col.astype(int), r.e8m0_col.astype(int) + k)
    # columnwise 32x1 of x equals rowwise 1x32 of x^T, transposed back
    rt = O.mxfp8(np.ascontiguousarray(x.T))
    assert np.array_equal(r.q_col, rt.q_row.T) and np.array_equal(r.e8m0_col, rt.e8m0_row.T)


@pytest.mark.parametrize("direction", [O.ROW, O.COL])
def test_mx_dequant_value_is_element_times_scale(direction):
    """value = element * block scale ("Mixed-precision training: fp16 to
    fp8", section "MXFP8"); relative error of a normal-range element <= 2^-4,
    or < 1/8 where the scaled value in [448, 512) saturated to 448."""
    x = W.gen("lognormal_rows", (64, 64), 4, bf16=True)
    r = O.mxfp8(x)
    q, e = (r.q_row, r.e8m0_row) if direction == O.ROW else (r.q_col, r.e8m0_col)
    y = O.dq_mxfp8(q, e, O.E4M3, direction)
    sc = torch.from_numpy(e).view(torch.float8_e8m0fnu).float().numpy()
    sc = np.repeat(sc, 32, axis=1) if direction == O.ROW else np.repeat(sc, 32, axis=0)
    assert np.array_equal(y, (dec8(q) * sc).astype(np.float32))
    xf = W.bf16_bits_to_f32(x)
    normal = np.abs(dec8(q)) >= 2.0 ** -6
    rel = np.where(np.abs(dec8(q)) == 448, 0.125, 2.0 ** -4)
    assert np.all((np.abs(y - xf) <= np.abs(xf) * rel)[normal])
    assert np.any(np.abs(dec8(q)) == 448)


def test_mx_zero_block():
    x = W.gen("normal", (32, 64), 7, bf16=False)
    x[:, :32] = 0
    r = O.mxfp8(x)
    assert np.all(r.e8m0_row[:, 0] == 127) and not r.q_row[:, :32].any()
    assert np.all(r.e8m0_col[0, :32] == 127)


def test_mx_row_to_col_requant_near_identity():
    """Power-of-two scales make dequantize -> requantize in the other direction
    nearly lossless ("Mixed-precision training: fp16 to fp8", section "FP8
    communication", EP): requantizing the rowwise dequantized tensor
    columnwise matches direct columnwise quantization almost everywhere."""
    x = W.gen("lognormal_rows", (128, 128), 8, bf16=True)
    r = O.mxfp8(x)
    y = O.dq_mxfp8(r.q_row, r.e8m0_row, O.E4M3, O.ROW)
    r2 = O.mxfp8(y)
    assert np.mean(r2.q_col == r.q_col) > 0.95
    assert np.mean(r2.e8m0_col == r.e8m0_col) > 0.95


# ---------------------------------------------------------------------------
# blockwise
# ---------------------------------------------------------------------------

def test_bw_1x128_reduces_to_current_scaling_per_tile():
    x = W.gen("normal", (8, 384), 2, bf16=True)
    r = O.blockwise(x, O.T1x128, rowwise=True, colwise=False)
    for m in range(8):
        for kb in range(3):
            t = O.current_scaling(np.ascontiguousarray(x[m:m + 1, kb * 128:(kb + 1) * 128]))
            assert np.array_equal(r.q_row[m, kb * 128:(kb + 1) * 128], t.q_row[0])
            assert r.s_row[m, kb] == t.scale


def test_bw_1x128_colwise_is_rowwise_of_transpose():
    x = W.gen("normal", (256, 256), 3, bf16=True)
    r = O.blockwise(x, O.T1x128, rowwise=True, colwise=True)
    rt = O.blockwise(np.ascontiguousarray(x.T), O.T1x128, rowwise=True)
    assert np.array_equal(r.q_colT, rt.q_row) and np.array_equal(r.s_colT, rt.s_row)
    assert r.s_colT.shape == (256, 2)


def test_bw_128x128_tile_and_transpose():
    x = W.gen("weight", (256, 384), 4, bf16=True)
    r = O.blockwise(x, O.T128x128, rowwise=True, colwise=True)
    assert np.array_equal(r.q_colT, r.q_row.T) and np.array_equal(r.s_colT, r.s_row.T)
    for mb in range(2):
        for kb in range(3):
            t = O.current_scaling(np.ascontiguousarray(x[mb * 128:(mb + 1) * 128, kb * 128:(kb + 1) * 128]))
            assert np.array_equal(r.q_row[mb * 128:(mb + 1) * 128, kb * 128:(kb + 1) * 128], t.q_row)
            assert r.s_row[mb, kb] == t.scale


@pytest.mark.parametrize("tile", [O.T1x128, O.T128x128])
def test_bw_dequant(tile):
    x = W.gen("normal", (128, 256), 5, bf16=True)
    r = O.blockwise(x, tile, rowwise=True, colwise=True)
    y = O.dq_blockwise(r.q_row, r.s_row, tile)
    s = np.repeat(r.s_row, 128, axis=1) if tile == O.T1x128 else np.repeat(np.repeat(r.s_row, 128, 0), 128, 1)
    assert np.array_equal(y, (dec8(r.q_row) * s).astype(np.float32))
    yt = O.dq_blockwise(r.q_colT, r.s_colT, tile)
    if tile == O.T128x128:
        assert np.array_equal(yt, y.T)


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------

def test_nv_global_scale_and_max_block():
    x = W.gen("normal", (32, 64), 6, bf16=False)
    r = O.nvfp4(x, O.B1x16, rowwise=True, colwise=True)
    A = np.float32(np.abs(x).max())
    assert r.amax == A
    assert r.s_global == np.float32(1) / (np.float32(2688) / A)
    # the block holding the tensor's amax gets the largest E4M3 scale and a +-6 code
    m, k = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert r.sb_row[m, k // 16] == 0x7E and r.sb_colT[k, m // 16] == 0x7E
    assert O.unpack_e2m1(r.q_row, 64)[m, k] & 7 == 7
    assert O.unpack_e2m1(r.q_colT, 32)[k, m] & 7 == 7


def test_nv_power_of_two_invariance():
    x = W.gen("t3", (32, 64), 6, bf16=False)
    base = O.nvfp4(x, O.B1x16, rowwise=True, colwise=True)
    for k in (-10, 4):
        r = O.nvfp4((x * np.float32(2.0 ** k)).astype(np.float32), O.B1x16, rowwise=True, colwise=True)
        assert np.array_equal(r.q_row, base.q_row) and np.array_equal(r.q_colT, base.q_colT)
        assert np.array_equal(r.sb_row, base.sb_row) and np.array_equal(r.sb_colT, base.sb_colT)
        assert r.s_global == base.s_global * np.float32(2.0 ** k)


def test_nv_1x16_colwise_is_rowwise_of_transpose_and_nibble_order():
    x = W.gen("normal", (48, 32), 2, bf16=True)
    r = O.nvfp4(x, O.B1x16, rowwise=True, colwise=True)
    rt = O.nvfp4(np.ascontiguousarray(x.T), O.B1x16, rowwise=True)
    assert np.array_equal(r.q_colT, rt.q_row) and np.array_equal(r.sb_colT, rt.sb_row)
    # even element in the low nibble: a tensor whose even columns are +max and odd columns 0
    z = np.zeros((1, 16), np.float32)
    z[0, 0::2] = 1.0
    q = O.nvfp4(z, O.B1x16).q_row
    assert np.all(q == 0x07)


def test_nv_16x16_transpose_identity():
    x = W.gen("weight", (64, 96), 3, bf16=True)
    r = O.nvfp4(x, O.B16x16, rowwise=True, colwise=True)
    codes = O.unpack_e2m1(r.q_row, 96)
    codes_t = O.unpack_e2m1(r.q_colT, 64)
    assert np.array_equal(codes_t, codes.T)
    assert np.array_equal(r.sb_colT, r.sb_row.T)
    # one scale per 16x16 tile: its value is the E4M3 cast of (tile max * alpha_g) / 6
    xf = W.bf16_bits_to_f32(x)
    alpha_g = np.float32(2688) / np.float32(np.abs(xf).max())
    tb = np.abs(xf).reshape(4, 16, 6, 16).max(axis=(1, 3)).astype(np.float32)
    sbf = ((tb * alpha_g).astype(np.float32) / np.float32(6)).astype(np.float32)
    want = torch.from_numpy(sbf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(r.sb_row, want)


@pytest.mark.parametrize("blk", [O.B1x16, O.B16x16])
def test_nv_dequant_identity_and_error_bound(blk):
    x = W.gen("normal", (64, 64), 11, bf16=True)
    r = O.nvfp4(x, blk, rowwise=True)
    y = O.dq_nvfp4(r.q_row, r.sb_row, r.s_global, blk)
    sb = dec8(r.sb_row)
    f = (sb * r.s_global).astype(np.float32)
    f = np.repeat(f, 16, axis=1) if blk == O.B1x16 else np.repeat(np.repeat(f, 16, 0), 16, 1)
    codes = O.unpack_e2m1(r.q_row, 64)
    assert np.array_equal(y, (dec4(codes) * f).astype(np.float32))
    # error bound: half an E2M1 spacing at the scaled value, plus any saturation overshoot
    xf = W.bf16_bits_to_f32(x)
    yscaled = np.abs(xf) / f
    spacing = np.where(yscaled < 2, 0.5, np.where(yscaled < 4, 1.0, 2.0))
    bound = (spacing / 2 + np.maximum(yscaled - 6, 0)) * f * (1 + 1e-5)
    assert np.all(np.abs(y - xf) <= bound)


def test_nv_encode_factor_is_one_division_per_block():
    """The encode factor is enc = fl(alpha_g / f(sb)), one FP32 division per
    block (R-NV; "Mixed-precision training: fp16 to fp8", recipe 6: E4M3
    block scale with an FP32 tensor scale).  A hand-derived case where the
    element lands exactly on an E2M1 tie under that reading and just past it
    under either plausible alternative:
      A = 39 (the row's other block holds 39), alpha_g = fl(2688 / 39)
        = 68.92308 (bits 0x4289D89E);
      block maximum b = 19.625: fl(fl(b * alpha_g) / 6) = 225.43591, E4M3
        RTNE -> 224 (code 0x76: 1.75 * 2^7);
      enc = fl(alpha_g / 224) = 0.30769232 (bits 0x3E9D89D9);
      x = 0.8125: fl(x * enc) = 0.25 exactly, the tie between 0 and 0.5 ->
        0 (even), code 0x0; b itself: fl(19.625 * enc) = 6.038 -> 6, code 0x7.
    The alternatives fl(alpha_g * fl(1 / 224)) = 0.30769235 and
    fl(fl(x * alpha_g) / 224) both give 0.25000003 -> 0.5, code 0x1."""
    row = np.zeros((1, 32), np.float32)
    row[0, 0], row[0, 1] = 19.625, 0.8125
    row[0, 16] = 39.0
    r = O.nvfp4(row, O.B1x16, O.RN, rowwise=True)
    assert np.float32(r.amax) == np.float32(39.0)
    assert int(r.sb_row[0, 0]) == 0x76
    codes = O.unpack_e2m1(r.q_row, 32)[0]
    assert int(codes[0]) == 0x7 and int(codes[1]) == 0x0
    # the arithmetic behind the literals, in numpy FP32
    f32 = np.float32
    alpha = f32(f32(2688.0) / f32(39.0))
    assert int(alpha.view(np.uint32)) == 0x4289D89E
    enc = f32(alpha / f32(224.0))
    assert int(enc.view(np.uint32)) == 0x3E9D89D9 and f32(f32(0.8125) * enc) == f32(0.25)
    for wrong in (f32(f32(0.8125) * f32(alpha * f32(f32(1.0) / f32(224.0)))), f32(f32(f32(0.8125) * alpha) / f32(224.0))):
        assert wrong > f32(0.25) and O.cast_e2m1(np.array([wrong], np.float32))[0] == 0x1


def test_nv_zero_block_scale_one():
    x = W.gen("normal", (16, 32), 1, bf16=False)
    x[:, 16:] = 0
    r = O.nvfp4(x, O.B1x16, rowwise=True)
    assert np.all(r.sb_row[:, 1] == 0x38)
    assert not O.unpack_e2m1(r.q_row, 32)[:, 16:].any()
    r = O.nvfp4(np.zeros((16, 16), np.float32), O.B16x16, rowwise=True)
    assert r.s_global == 1 and np.all(r.sb_row == 0x38)


def test_nv_sr_rounds_to_neighbours_and_matches_rn_on_grid():
    x = W.gen("t3", (32, 64), 12, bf16=True)
    rn = O.nvfp4(x, O.B1x16, O.RN, rowwise=True, colwise=True)
    sr = O.nvfp4(x, O.B1x16, O.SR, seed=4, offset=0, rowwise=True, colwise=True)
    assert np.array_equal(sr.sb_row, rn.sb_row) and np.array_equal(sr.sb_colT, rn.sb_colT)
    d_rn = dec4(O.unpack_e2m1(rn.q_row, 64))
    d_sr = dec4(O.unpack_e2m1(sr.q_row, 64))
    # SR lands on the other neighbour only; the RN code is always one of the two
    assert np.all(np.abs(d_sr - d_rn) <= 2)
    assert 0 < np.mean(d_sr != d_rn) < 0.6
    sr2 = O.nvfp4(x, O.B1x16, O.SR, seed=4, offset=0, rowwise=True, colwise=True)
    assert np.array_equal(sr.q_row, sr2.q_row) and np.array_equal(sr.q_colT, sr2.q_colT)
    sr3 = O.nvfp4(x, O.B1x16, O.SR, seed=5, offset=0, rowwise=True)
    assert not np.array_equal(sr.q_row, sr3.q_row)


def test_nv_sr_uses_row_and_column_indices():
    """Rowwise element (m, k) draws index m*K + k on stream 0; the columnwise
    copy of element (m, k) draws index ((m // 16)*K + k)*16 + m % 16 on stream 1
    (16-row groups of x, then columns, then rows), which does not depend on M."""
    x = W.gen("t3", (32, 32), 13, bf16=False)
    r = O.nvfp4(x, O.B1x16, O.SR, seed=99, offset=5, rowwise=True, colwise=True)
    alpha_g, _ = O.nvfp4_global(r.amax)
    sbv = dec8(r.sb_row)
    enc = (alpha_g / sbv).astype(np.float32)
    y = (x * np.repeat(enc, 16, axis=1)).astype(np.float32)
    want = O.sr_e2m1_batch(y.ravel(), seed=99, offset=5, stream=0).reshape(32, 32)
    assert np.array_equal(O.unpack_e2m1(r.q_row, 32), want)
    sbc = dec8(r.sb_colT)
    encc = (alpha_g / sbc).astype(np.float32)
    yt = (np.ascontiguousarray(x.T) * np.repeat(encc, 16, axis=1)).astype(np.float32)
    M, K = x.shape
    wantc = np.array([[O.sr_e2m1(yt[k, m], O.philox_bits16(99, 5, 1, ((m // 16) * K + k) * 16 + m % 16))
                       for m in range(M)] for k in range(K)], np.uint8)
    assert np.array_equal(O.unpack_e2m1(r.q_colT, M), wantc)
    # the transposed-layout numbering k*M + m, and 8-row groups, give other
    # codes here (so the test tells the numberings apart)
    old = O.sr_e2m1_batch(yt.ravel(), seed=99, offset=5, stream=1).reshape(32, 32)
    assert not np.array_equal(old, wantc)
    old8 = np.array([[O.sr_e2m1(yt[k, m], O.philox_bits16(99, 5, 1, ((m // 8) * K + k) * 8 + m % 8))
                      for m in range(M)] for k in range(K)], np.uint8)
    assert not np.array_equal(old8, wantc)


@pytest.mark.parametrize("blk", [O.B1x16, O.B16x16])
def test_nv_sr_row_shards_draw_what_the_whole_tensor_draws(blk):
    """A band of rows [r0, r0 + h) quantized alone with counter offset
    offset + r0*K/16 and the whole tensor's amax gives exactly that band of the
    unsharded stochastic quantization, rowwise and columnwise ("Mixed-precision
    training: fp16 to fp8", FP8 communication, TP: the FP8 tensor must not
    depend on the split)."""
    x = W.gen("t3", (96, 64), 14, bf16=True)
    M, K = x.shape
    A = O.amax(x)
    whole = O.nvfp4(x, blk, O.SR, seed=31, offset=1000, rowwise=True, colwise=True)
    for r0, h in ((0, 32), (32, 16), (48, 48)):
        band = O.nvfp4(np.ascontiguousarray(x[r0:r0 + h]), blk, O.SR, seed=31, offset=1000 + r0 * K // 16,
                       rowwise=True, colwise=True, amax_in=A)
        assert np.array_equal(band.q_row, whole.q_row[r0:r0 + h])
        assert np.array_equal(band.q_colT, whole.q_colT[:, r0 // 2:(r0 + h) // 2])
        if blk == O.B1x16:
            assert np.array_equal(band.sb_row, whole.sb_row[r0:r0 + h])
            assert np.array_equal(band.sb_colT, whole.sb_colT[:, r0 // 16:(r0 + h) // 16])
    # without the shifted offset the bands repeat the first band's draws
    b2 = O.nvfp4(np.ascontiguousarray(x[32:64]), blk, O.SR, seed=31, offset=1000, rowwise=True, amax_in=A)
    assert not np.array_equal(b2.q_row, whole.q_row[32:64])


# ---------------------------------------------------------------------------
# MXFP8 row -> col re-quantization
# ---------------------------------------------------------------------------

def test_mx_requant_exact_on_grid_inputs():
    """Inputs that both directions represent exactly (signed powers of two
    spanning 8 binades, every 32-element block and 32-row block holding a
    2^7) dequantize exactly, so re-quantizing the rowwise copy gives the
    direct columnwise quantization bit for bit."""
    rng = np.random.default_rng(21)
    k = rng.integers(0, 8, (64, 96))
    x = (np.where(rng.random((64, 96)) < 0.5, -1.0, 1.0) * 2.0 ** k).astype(np.float32)
    x[np.arange(64), (np.arange(64) * 7) % 96] = 128.0          # a 2^7 in every row block ...
    for mb in range(2):
        x[mb * 32 + (np.arange(96) % 32), np.arange(96)] = 128.0  # ... and in every column block
    for fmt in (O.E4M3, O.E5M2):
        r = O.mxfp8(x, fmt)
        assert np.array_equal(O.dq_mxfp8(r.q_row, r.e8m0_row, fmt, O.ROW), x)
        q_col, e_col = O.mxfp8_requant_col(r.q_row, r.e8m0_row, fmt)
        assert np.array_equal(q_col, r.q_col) and np.array_equal(e_col, r.e8m0_col)


def test_mx_requant_close_to_direct_columnwise():
    x = W.gen("lognormal_rows", (128, 128), 8, bf16=True)
    r = O.mxfp8(x)
    q_col, e_col = O.mxfp8_requant_col(r.q_row, r.e8m0_row)
    assert np.mean(q_col == r.q_col) > 0.95 and np.mean(e_col == r.e8m0_col) > 0.95
    # both decode to within the two quantizations' error of x: each step is off by at
    # most 1/16 (1/8 where a value in [448, 512) saturated) relative
    d1 = O.dq_mxfp8(q_col, e_col, O.E4M3, O.COL)
    xf = W.bf16_bits_to_f32(x)
    big = np.abs(dec8(r.q_col)) >= 2.0 ** -6
    assert np.all((np.abs(d1 - xf) <= np.abs(xf) * (1 / 8 + 1 / 8 * 9 / 8) + 1e-30)[big])


# ---------------------------------------------------------------------------
# per-tensor delayed scaling ("Mixed-precision training: fp16 to fp8",
# "Per-tensor delayed scaling")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_ds_cast_equals_current_scaling_at_the_same_alpha(fmt):
    x = W.gen("outliers", (96, 160), 31, bf16=True)
    A = O.amax(x)
    alpha, _ = O.cs_scale(A, fmt)
    q_row, q_colT, a = O.ds_cast(x, alpha, fmt, rowwise=True, colwise=True)
    cs = O.current_scaling(x, fmt, rowwise=True, colwise=True)
    assert np.array_equal(q_row, cs.q_row) and np.array_equal(q_colT, cs.q_colT)
    assert q_colT.shape == (160, 96) and np.array_equal(q_colT, q_row.T)
    assert a == A


def test_ds_cast_alpha_one_reproduces_grid_values():
    """Every finite E4M3 value cast with alpha = 1 returns its own code."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8).reshape(1, -1)
    x = dec8(codes).astype(np.float32)
    q_row, _, a = O.ds_cast(x, 1.0, O.E4M3)
    assert np.array_equal(q_row, codes)
    assert a == np.float32(448.0)


def test_ds_scale_update_closed_forms():
    z = np.zeros(16, np.float32)
    assert O.ds_scale_update(z, 0) == (1.0, 1.0)                        # empty window: alpha = s = 1
    h = z.copy()
    h[5] = 8.0
    al, s = O.ds_scale_update(h, 9)
    assert al == np.float32(56.0) and s == np.float32(1.0) / np.float32(56.0)   # 448 / 8
    al, s = O.ds_scale_update(h, 9, fmt=O.E5M2)
    assert al == np.float32(7168.0)                                      # 57344 / 8
    assert O.ds_scale_update(h, 9, O.HIST_MOST_RECENT) == (1.0, 1.0)    # slot 9 is empty
    assert O.ds_scale_update(h, 5, O.HIST_MOST_RECENT)[0] == np.float32(56.0)
    h[2] = 1e-45                                                         # 448 / 1e-45 overflows: FLT_MAX
    assert O.ds_scale_update(h, 2, O.HIST_MOST_RECENT)[0] == np.finfo(np.float32).max
    h[3] = np.nan
    assert np.isnan(O.ds_scale_update(h, 9)[0])                          # a NaN entry wins the max


@pytest.mark.parametrize("algo,N", [(O.HIST_MAX, 4), (O.HIST_MAX, 1), (O.HIST_MOST_RECENT, 4), (O.HIST_MAX, 1024)])
def test_ds_window_against_a_plain_list_model(algo, N):
    """A run of steps through the ring (slot = step % N) against a list of
    the last N amaxes: each step's alpha is 448 / max (or / latest) of the
    amaxes recorded before it, and 1 before any."""
    rng = np.random.default_rng(4)
    base = W.gen("normal", (16, 32), 9, bf16=False)
    base /= np.abs(base).max()                                           # amax of base = 1 exactly
    amaxes = [np.float32(2.0) ** int(e) for e in rng.integers(-6, 7, 3 * N + 5)]
    amaxes[1] = np.float32(4096.0)                                       # an outlier that must leave after N steps
    hist = np.zeros(N, np.float32)
    alpha = np.float32(1.0)
    window = []
    for t, a in enumerate(amaxes):
        if window:
            ref = max(window) if algo == O.HIST_MAX else window[-1]
            want = np.float32(448.0) / np.float32(ref)
        else:
            want = np.float32(1.0)
        assert alpha == want, (t, alpha, want)
        x = (base * a).astype(np.float32)
        q_row, _, got_a = O.ds_cast(x, alpha, O.E4M3)
        assert got_a == np.float32(a)
        assert np.array_equal(q_row, O.cast_fp8((alpha * x).astype(np.float32), O.E4M3))
        hist[t % N] = got_a
        alpha, s = O.ds_scale_update(hist, t % N, algo)
        assert s == np.float32(1.0) / alpha
        window = (window + [np.float32(a)])[-N:]


def test_ds_repeated_tensor_converges_to_current_scaling():
    """Quantizing the same tensor every step: from the second step on the
    window holds its amax, so the codes are the current-scaling codes."""
    x = W.gen("t3", (64, 48), 12, bf16=True)
    hist = np.zeros(8, np.float32)
    alpha = np.float32(1.0)
    cs = O.current_scaling(x, O.E4M3, rowwise=True, colwise=True)
    for t in range(3):
        q_row, q_colT, a = O.ds_cast(x, alpha, O.E4M3, rowwise=True, colwise=True)
        if t > 0:
            assert np.array_equal(q_row, cs.q_row) and np.array_equal(q_colT, cs.q_colT)
        hist[t % 8] = a
        alpha, _ = O.ds_scale_update(hist, t % 8)
    assert alpha == O.cs_scale(O.amax(x))[0]
