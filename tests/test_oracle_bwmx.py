"""Pins of the oracle's blockwise-as-MXFP8 quantizer (power-of-two tile
scales stored as E8M0, reading R-BWMX), against values computed by hand, the
pinned blockwise and MXFP8 oracles, and invariants:

* scale codes of hand-picked tile maxima (the rounding direction of the
  power of two and its clamps);
* with a tile maximum of 448 * 2^k the FP32 blockwise scale is itself a power
  of two, and the codes equal the blockwise codes;
* when every 32-element sub-block of a tile holds the tile maximum (with a
  significand of at most 1.75) the MXFP8 floor rule gives the same code, and
  the result equals MXFP8 quantization;
* the tile maximum never saturates and lands in (224, 448];
* the 128x128 transposed copy is the transposed row copy; every tile's code
  is repeated over its 32-element groups;
* dequantizing with the MXFP8 decoder recovers x within E4M3's error.
"""
import numpy as np
import pytest

import oracle as O


def _row(b, n=256):
    """One FP32 row whose every 1x128 tile has maximum |x| = b."""
    x = np.full((1, n), np.float32(b) / 4, np.float32)
    x[0, ::128] = np.float32(b)
    return x


@pytest.mark.parametrize("b,code", [
    (448.0, 127),                      # b / 448 = 1 = 2^0
    (449.0, 128),                      # just above: round up to 2^1
    (224.0, 126),                      # 2^-1 exactly
    (1.0, 119),                        # 1/448 = 2^-8.81 -> 2^-8
    (1.75, 119),                       # 1.75/448 = 2^-8 exactly
    (1.7578125, 120),                  # 1.75 + 2^-7: above 2^-8 -> 2^-7
    (0.0, 127),                        # zero tile: scale 1
    (2.0 ** -140, 0),                  # FP32 subnormal maximum: 2^-148 clamps to code 0
    (3.0e38, 247),                     # 448 * 2^119 < 3e38 <= 448 * 2^120
])
def test_scale_codes_by_hand(b, code):
    r = O.blockwise_mx(_row(b), O.T1x128)
    assert np.all(r.e8m0_row == code), (b, r.e8m0_row)


def test_nonfinite_tile_takes_the_mxfp8_code():
    x = _row(1.0)
    x[0, 5] = np.inf
    r = O.blockwise_mx(x, O.T1x128)
    mx = O.mxfp8(np.tile(x[:, :128], (32, 1)), O.E4M3)
    assert r.e8m0_row[0, 0] == mx.e8m0_row[0, 0] == 247
    assert r.e8m0_row[0, 4] == 119


@pytest.mark.parametrize("tile", [O.T1x128, O.T128x128])
def test_equals_blockwise_when_its_scale_is_a_power_of_two(tile):
    rng = np.random.default_rng(5)
    M, K = 256, 384
    x = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    ks = rng.integers(-12, 12, (M // 128, K // 128))
    for i in range(M // 128):
        for j in range(K // 128):
            t = x[128 * i:128 * i + 128, 128 * j:128 * j + 128]
            t *= np.float32(448.0 * 2.0 ** ks[i, j])
            if tile == O.T1x128:
                t[:, 0] = np.float32(448.0 * 2.0 ** ks[i, j])   # every 1x128 row of the tile
            t[0, :] = np.float32(-448.0 * 2.0 ** ks[i, j])      # every 128x1 column of the tile
    bw = O.blockwise(x, tile, rowwise=True, colwise=True)
    mx = O.blockwise_mx(x, tile, rowwise=True, colwise=True)
    assert np.array_equal(mx.q_row, bw.q_row)
    assert np.array_equal(mx.q_colT, bw.q_colT)
    # the power-of-two code is the FP32 blockwise scale
    if tile == O.T1x128:
        assert np.array_equal(np.ldexp(1.0, mx.e8m0_row[:, ::4].astype(int) - 127), bw.s_row)
        assert np.array_equal(np.ldexp(1.0, mx.e8m0_colT[:, ::4].astype(int) - 127), bw.s_colT)
    else:
        assert np.array_equal(np.ldexp(1.0, mx.e8m0_row[::128, ::4].astype(int) - 127), bw.s_row)
        assert np.array_equal(np.ldexp(1.0, mx.e8m0_colT[::128, ::4].astype(int) - 127), bw.s_colT)


def test_equals_mxfp8_when_every_subblock_holds_the_tile_maximum():
    """MXFP8 takes floor(log2 b) - 8; with a significand of b at most 1.75
    that is the same power of two, and the elements follow the same rule."""
    rng = np.random.default_rng(6)
    M, K = 128, 512
    x = rng.standard_normal((M, K)).astype(np.float32)
    x = np.clip(x, -1.0, 1.0) * np.float32(0.9)
    b = np.float32(1.5 * 2.0 ** 3)
    x[:, ::32] = b           # rowwise: every 1x32 block of every row holds b
    x[::32, :] = -b          # columnwise: every 32x1 block of every column holds |b|
    want = O.mxfp8(x, O.E4M3)
    got = O.blockwise_mx(x, O.T1x128, rowwise=True, colwise=True)
    assert np.array_equal(got.q_row, want.q_row)
    assert np.array_equal(got.e8m0_row, want.e8m0_row)
    assert np.array_equal(got.q_colT, want.q_col.T)
    assert np.array_equal(got.e8m0_colT, want.e8m0_col.T)


@pytest.mark.parametrize("tile", [O.T1x128, O.T128x128])
def test_tile_maximum_lands_in_the_top_binade_and_never_saturates(tile):
    rng = np.random.default_rng(7)
    M, K = 256, 256
    x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-20, 20, (M, 1)))).astype(np.float32)
    r = O.blockwise_mx(x, tile, rowwise=True, colwise=False)
    scaled = np.abs(x.astype(np.float64)) * np.ldexp(1.0, 127 - np.repeat(r.e8m0_row.astype(int), 32, axis=1))
    assert np.all(scaled <= 448.0)
    if tile == O.T1x128:
        tmax = scaled.reshape(M, K // 128, 128).max(axis=2)
    else:
        tmax = scaled.reshape(M // 128, 128, K // 128, 128).max(axis=(1, 3))
    assert np.all((tmax > 224.0) & (tmax <= 448.0))
    assert np.all(r.q_row & 0x7F != 0x7F)       # no NaN code from finite input


def test_128x128_copies_and_code_repetition():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((256, 384)).astype(np.float32)
    r = O.blockwise_mx(x, O.T128x128, rowwise=True, colwise=True)
    assert np.array_equal(r.q_colT, r.q_row.T)
    assert np.array_equal(r.e8m0_colT.reshape(384, 2, 4)[:, :, 0],
                          r.e8m0_row.reshape(2, 128, 3, 4)[:, 0, :, 0].T.repeat(128, axis=0))
    for e in (r.e8m0_row, r.e8m0_colT):
        assert np.all(e.reshape(e.shape[0], -1, 4) == e.reshape(e.shape[0], -1, 4)[:, :, :1])
    assert np.all(r.e8m0_row.reshape(2, 128, -1) == r.e8m0_row.reshape(2, 128, -1)[:, :1, :])


@pytest.mark.parametrize("tile", [O.T1x128, O.T128x128])
def test_mxfp8_decode_recovers_x(tile):
    rng = np.random.default_rng(9)
    x = O.bf16_round(rng.standard_normal((128, 256)).astype(np.float32))    # BF16 bit patterns
    r = O.blockwise_mx(x, tile, rowwise=True, colwise=True)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for q, e, ref in ((r.q_row, r.e8m0_row, xf), (r.q_colT, r.e8m0_colT, xf.T)):
        y = O.dq_mxfp8(q, e, O.E4M3, O.ROW, O.F32).astype(np.float64)
        step = np.ldexp(1.0, np.repeat(e.astype(int), 32, axis=1) - 127)     # the scale 2^(code - 127)
        # E4M3: relative half-step 2^-4 for normal codes, absolute 2^-10 * scale below 2^-6
        assert np.all(np.abs(y - ref) <= np.maximum(np.abs(ref) * 2.0 ** -4, step * 2.0 ** -10) * (1 + 1e-12))
