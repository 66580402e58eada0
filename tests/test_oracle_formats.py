"""Pins of the oracle's element casts against things other than itself.

* brute-force nearest-value search over every code (values decoded by
  ml_dtypes / torch, not by the oracle), ties to the even code, over all 65536
  BF16 bit patterns;
* the library casts of ml_dtypes and torch where they agree with a
  saturating cast (magnitudes up to Fmax plus half an ulp);
* the values the pages print: E4M3 grid in [32, 64), the maxima 448 / 57344,
  the 16 E2M1 values in code order.
"""
import json
import os


import numpy as np
import pytest

ml_dtypes = pytest.importorskip("ml_dtypes")
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


ALL_BF16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)

FP8 = {
    O.E4M3: dict(mld=ml_dtypes.float8_e4m3fn, torch=torch.float8_e4m3fn, max=448.0, nan=0x7F, maxcode=0x7E),
    O.E5M2: dict(mld=ml_dtypes.float8_e5m2, torch=torch.float8_e5m2, max=57344.0, nan=0x7F, maxcode=0x7B),
}


def lib_decode_fp8(fmt):
    """Decoded value of every byte, by ml_dtypes (independent of the oracle)."""
    return np.arange(256, dtype=np.uint8).view(FP8[fmt]["mld"]).astype(np.float64)


def brute_force_fp8(v, fmt):
    """Nearest finite code by exhaustive search, ties to the even code,
    saturating, NaN -> 0x7F, sign from the input's sign bit."""
    table = lib_decode_fp8(fmt)
    pos = np.arange(0, FP8[fmt]["maxcode"] + 1)          # positive finite codes, ascending value
    mags = table[pos]
    assert np.all(np.diff(mags) > 0)
    v = np.asarray(v, np.float32)
    a = np.abs(np.nan_to_num(v, nan=0.0).astype(np.float64))
    out = np.empty(v.shape, np.uint8)
    d = np.abs(mags[None, :] - a[:, None])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    # among equally near codes take the even one (the two candidates of a tie are adjacent codes)
    even = cand & ((pos[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    code = pos[pick]
    code = np.where(a >= FP8[fmt]["max"], FP8[fmt]["maxcode"], code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    out[:] = code
    out[np.isnan(v)] = FP8[fmt]["nan"]
    return out


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_cast_exhaustive_bf16_brute_force(fmt):
    got = O.cast_fp8(ALL_BF16, fmt)
    want = brute_force_fp8(ALL_BF16, fmt)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"first mismatches: {[(hex(int(i)), got[i], want[i]) for i in bad[:5]]}"


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_cast_random_fp32_brute_force(fmt):
    rng = np.random.default_rng(11)
    mx = FP8[fmt]["max"]
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(mx / 4),
        (rng.standard_normal(20000) * 1e-3).astype(np.float32),
        np.float32(mx) * rng.uniform(0.9, 1.2, 2000).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 3.4e38], np.float32),
    ])
    assert np.array_equal(O.cast_fp8(v, fmt), brute_force_fp8(v, fmt))


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_cast_matches_libraries_in_range(fmt):
    """ml_dtypes and torch cast with RTNE but without saturation; they must
    agree with the oracle wherever no saturation decision is involved."""
    mx = FP8[fmt]["max"]
    v = ALL_BF16[np.isfinite(ALL_BF16) & (np.abs(ALL_BF16) <= mx)]
    got = O.cast_fp8(v, fmt)
    lib = v.astype(FP8[fmt]["mld"]).view(np.uint8)
    assert np.array_equal(got, lib)
    tt = torch.from_numpy(v).to(FP8[fmt]["torch"]).view(torch.uint8).numpy()
    assert np.array_equal(got, tt)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_decode_matches_library_all_codes(fmt):
    codes = np.arange(256, dtype=np.uint8)
    got = O.decode_fp8(codes, fmt).astype(np.float64)
    want = lib_decode_fp8(fmt)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_encode_decode_round_trip(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = O.decode_fp8(codes, fmt)
    finite = np.isfinite(vals)
    assert np.array_equal(O.cast_fp8(vals[finite], fmt), codes[finite])


def test_page_e4m3_grid_and_maxima():
    g = gold("e4m3_grid.json")
    for v in g["representable_in_32_64"]:
        c = O.cast_fp8(np.array([v], np.float32), O.E4M3)
        assert O.decode_fp8(c, O.E4M3)[0] == np.float32(v)
    # everything the format holds in [32, 64) is spaced by 4
    table = lib_decode_fp8(O.E4M3)
    inside = np.sort(table[(table >= 32) & (table < 64)])
    assert np.array_equal(inside, np.arange(32, 64, 4))
    for v in g["not_representable"]:
        assert float(O.decode_fp8(O.cast_fp8(np.array([v], np.float32), O.E4M3), O.E4M3)[0]) != v
    m = gold("format_maxima.json")
    assert O.decode_fp8(np.array([0x7E], np.uint8), O.E4M3)[0] == m["E4M3"]["max"]
    assert O.decode_fp8(np.array([0x7B], np.uint8), O.E5M2)[0] == m["E5M2"]["max"]
    assert np.nanmax(np.where(np.isfinite(lib_decode_fp8(O.E4M3)), lib_decode_fp8(O.E4M3), np.nan)) == 448.0
    assert np.isinf(O.decode_fp8(np.array([0x7C], np.uint8), O.E5M2)[0])                # E5M2 has inf
    assert not np.isinf(O.decode_fp8(np.arange(256, dtype=np.uint8), O.E4M3)).any()   # E4M3 has none
    # saturation: anything beyond the maximum, infinities included, clamps
    for fmt, mx in ((O.E4M3, 448.0), (O.E5M2, 57344.0)):
        big = np.array([mx * 1.01, mx * 4, np.inf, -np.inf, 3e38], np.float32)
        assert np.array_equal(np.abs(O.decode_fp8(O.cast_fp8(big, fmt), fmt)), np.full(5, mx, np.float32))


def test_page_e2m1_values_in_code_order():
    g = gold("e2m1_values.json")
    vals = O.decode_e2m1(np.arange(16, dtype=np.uint8))
    assert np.array_equal(vals, np.array(g["values"], np.float32))
    assert np.array_equal(np.signbit(vals), np.signbit(np.array(g["values"], np.float32)))
    # the library's decode of the same nibbles
    lib = np.arange(16, dtype=np.uint8).view(ml_dtypes.float4_e2m1fn).astype(np.float32)
    assert np.array_equal(vals, lib)


def brute_force_e2m1(v):
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    codes = np.arange(8)
    v = np.asarray(v, np.float32)
    a = np.abs(np.nan_to_num(v, nan=0.0).astype(np.float64))
    d = np.abs(mags[None, :] - a[:, None])
    cand = d == d.min(axis=1, keepdims=True)
    even = cand & ((codes[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    out = (codes[pick] | np.where(np.signbit(v), 8, 0)).astype(np.uint8)
    out[a >= 6] = (7 | np.where(np.signbit(v), 8, 0))[a >= 6]
    out[np.isnan(v)] = 7
    return out


def test_e2m1_cast_exhaustive_bf16_brute_force():
    assert np.array_equal(O.cast_e2m1(ALL_BF16), brute_force_e2m1(ALL_BF16))


def test_e2m1_cast_matches_ml_dtypes():
    """ml_dtypes' E2M1 cast saturates and rounds to nearest even, like the
    oracle, for every finite input."""
    v = ALL_BF16[np.isfinite(ALL_BF16)]
    lib = v.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(O.cast_e2m1(v), lib)


def test_e2m1_ties():
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0], np.float32)
    want = np.array([0, 1, 1, 2, 2, 4, 4, -0.0, -4], np.float32)
    got = O.decode_e2m1(O.cast_e2m1(v))
    assert np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))


def test_e8m0_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = O.decode_e8m0(codes)
    tt = torch.from_numpy(codes).view(torch.float8_e8m0fnu).float().numpy()
    assert np.isnan(got[255]) and np.isnan(tt[255])
    assert np.array_equal(got[:255], tt[:255])
    # the code is the FP32 exponent field: 2^(c-127) has biased exponent c
    normal = got[1:255].view(np.uint32)
    assert np.array_equal((normal >> 23) & 0xFF, codes[1:255].astype(np.uint32))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(10000) * 1e-38).astype(np.float32),
        np.array([3.3895e38, 3.39e38, 3.4e38, -3.4e38, np.inf, -np.inf, 0.0, -0.0, 1e-45], np.float32),
        # exact ties between two BF16 values
        ((np.arange(1000, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
    ])
    v = v[np.isfinite(v) | np.isinf(v)]
    got = O.bf16_round(v)
    tt = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, tt)
