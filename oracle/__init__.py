"""CPU oracle for the tensor quantizers (numpy front end over ``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package; the library
(``nvfp4_quantization_current_gb300``) never does, and shares no code with it.

Every function takes and returns numpy arrays in the same layouts as the
library's C ABI:

* inputs ``x``: 2-D ``uint16`` holding BF16 bit patterns, or ``float32``;
* FP8 codes ``uint8`` [M, K] (rowwise) or [K, M] (columnwise, transposed);
* NVFP4 codes ``uint8`` [M, K/2] / [K, M/2], two E2M1 codes per byte, even
  element in the low nibble;
* scales: FP32 (current scaling, blockwise), E8M0 bytes (MXFP8, and
  blockwise tiles held as MXFP8), E4M3 bytes (NVFP4 block scales) + one FP32
  tensor scale.

The arithmetic lives in ``oracle.c`` (plain loops, FP32 steps as single
IEEE operations, no FMA contraction); its header lists the pages followed and
every reading taken where they are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

BF16, F32 = 0, 1
E4M3, E5M2 = 0, 1
T1x128, T128x128 = 0, 1
B1x16, B16x16 = 0, 1
RN, SR = 0, 1
ROW, COL = 0, 1

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I64, I, F, U64, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32
        sig = {
            "or_enc_e4m3": (ctypes.c_uint8, [F]),
            "or_enc_e5m2": (ctypes.c_uint8, [F]),
            "or_enc_e2m1": (ctypes.c_uint8, [F]),
            "or_dec_e4m3": (F, [ctypes.c_uint8]),
            "or_dec_e5m2": (F, [ctypes.c_uint8]),
            "or_dec_e2m1": (F, [ctypes.c_uint8]),
            "or_dec_e8m0": (F, [ctypes.c_uint8]),
            "or_cast_fp8": (None, [P, I64, I, P]),
            "or_cast_e2m1": (None, [P, I64, P]),
            "or_decode_fp8": (None, [P, I64, I, P]),
            "or_decode_e2m1": (None, [P, I64, P]),
            "or_bf16_round": (None, [P, I64, P]),
            "or_philox4_generic": (None, [I, I, P, P, P, P, P]),
            "or_philox4x32_10": (None, [P, P, P]),
            "or_philox_bits16": (U32, [U64, U64, U32, U64]),
            "or_sr_e2m1": (ctypes.c_uint8, [F, U32]),
            "or_sr_e2m1_batch": (None, [P, I64, U64, U64, U32, P]),
            "or_amax": (F, [P, I, I64]),
            "or_cs_scale": (None, [F, I, P, P]),
            "or_current_scaling": (None, [P, I, I64, I64, I, P, P, P, P, P]),
            "or_dq_current_scaling": (None, [P, F, I64, I64, I, I, P]),
            "or_mxfp8": (None, [P, I, I64, I64, I, P, P, P, P]),
            "or_dq_mxfp8": (None, [P, P, I64, I64, I, I, I, P]),
            "or_mxfp8_requant_col": (None, [P, P, I64, I64, I, P, P]),
            "or_rht16": (None, [P, U32]),
            "or_rht_cols": (None, [P, I, I64, I64, U32, P]),
            "or_nvfp4_rht_colT": (None, [P, I, I64, I64, U32, I, U64, U64, P, P, P, P, P]),
            "or_ds_cast": (None, [P, I, I64, I64, I, F, P, P, P]),
            "or_ds_scale_update": (None, [P, I64, I64, I, I, P, P]),
            "or_blockwise": (None, [P, I, I64, I64, I, P, P, P, P]),
            "or_blockwise_mx": (None, [P, I, I64, I64, I, P, P, P, P]),
            "or_dq_blockwise": (None, [P, P, I64, I64, I, I, P]),
            "or_nvfp4_global": (None, [F, P, P]),
            "or_nvfp4": (None, [P, I, I64, I64, I, I, U64, U64, P, P, P, P, P, P, P]),
            "or_dq_nvfp4": (None, [P, P, F, I64, I64, I, I, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _x(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.float32:
        return x, F32
    raise TypeError(f"oracle input must be uint16 (BF16 bits) or float32, got {x.dtype}")


def _fbuf(v=0.0):
    return np.array([v], dtype=np.float32)


# --------------------------------------------------------------------------
# element casts
# --------------------------------------------------------------------------

def cast_fp8(v, fmt=E4M3):
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _L().or_cast_fp8(_p(v), v.size, fmt, _p(out))
    return out


def cast_e2m1(v):
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _L().or_cast_e2m1(_p(v), v.size, _p(out))
    return out


def decode_fp8(c, fmt=E4M3):
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float32)
    _L().or_decode_fp8(_p(c), c.size, fmt, _p(out))
    return out


def decode_e2m1(c):
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float32)
    _L().or_decode_e2m1(_p(c), c.size, _p(out))
    return out


def decode_e8m0(c):
    return np.array([_L().or_dec_e8m0(int(v)) for v in np.ravel(c)], np.float32).reshape(np.shape(c))


def bf16_round(v):
    """FP32 -> BF16 bits, round to nearest even."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    _L().or_bf16_round(_p(v), v.size, _p(out))
    return out


def unpack_e2m1(packed, n_cols):
    """[R, C/2] packed bytes -> [R, C] 4-bit codes (even element low nibble)."""
    packed = np.asarray(packed, np.uint8)
    out = np.empty(packed.shape[:-1] + (n_cols,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


# --------------------------------------------------------------------------
# Philox / stochastic rounding
# --------------------------------------------------------------------------

def philox4_generic(width, rounds, ctr, key, mult, weyl):
    arr = lambda a, n: np.ascontiguousarray(np.array(a, dtype=np.uint64).reshape(n))
    c, k, m, w = arr(ctr, 4), arr(key, 2), arr(mult, 2), arr(weyl, 2)
    out = np.zeros(4, np.uint64)
    _L().or_philox4_generic(width, rounds, _p(c), _p(k), _p(m), _p(w), _p(out))
    return out


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(np.array(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.array(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, np.uint32)
    _L().or_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def philox_bits16(seed, offset, stream, i):
    return int(_L().or_philox_bits16(seed, offset, stream, i))


def sr_e2m1(y, r16):
    return int(_L().or_sr_e2m1(float(y), int(r16)))


def sr_e2m1_batch(y, seed, offset=0, stream=0):
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, np.uint8)
    _L().or_sr_e2m1_batch(_p(y), y.size, seed, offset, stream, _p(out))
    return out


# --------------------------------------------------------------------------
# recipes
# --------------------------------------------------------------------------

def amax(x):
    x, dt = _x(x)
    return float(np.float32(_L().or_amax(_p(x), dt, x.size)))


def cs_scale(a, fmt=E4M3):
    al, s = _fbuf(), _fbuf()
    _L().or_cs_scale(float(a), fmt, _p(al), _p(s))
    return al[0], s[0]


@dataclass
class CS:
    q_row: np.ndarray | None
    q_colT: np.ndarray | None
    amax: np.float32
    scale: np.float32


def current_scaling(x, fmt=E4M3, rowwise=True, colwise=False, amax_in=None):
    x, dt = _x(x)
    M, K = x.shape
    q_row = np.empty((M, K), np.uint8) if rowwise else None
    q_colT = np.empty((K, M), np.uint8) if colwise else None
    a_out, s_out = _fbuf(), _fbuf()
    a_in = None if amax_in is None else _fbuf(amax_in)
    _L().or_current_scaling(_p(x), dt, M, K, fmt, _p(a_in), _p(q_row), _p(q_colT), _p(a_out), _p(s_out))
    return CS(q_row, q_colT, a_out[0], s_out[0])


HIST_MAX, HIST_MOST_RECENT = 0, 1


def ds_cast(x, alpha, fmt=E4M3, rowwise=True, colwise=False):
    """Delayed scaling, one step's cast: codes of Q(alpha x) with the given
    alpha, and the step's amax (to be recorded in the history)."""
    x, dt = _x(x)
    M, K = x.shape
    q_row = np.empty((M, K), np.uint8) if rowwise else None
    q_colT = np.empty((K, M), np.uint8) if colwise else None
    a_out = _fbuf()
    _L().or_ds_cast(_p(x), dt, M, K, fmt, float(np.float32(alpha)), _p(q_row), _p(q_colT), _p(a_out))
    return q_row, q_colT, a_out[0]


def ds_scale_update(hist, pos, algo=HIST_MAX, fmt=E4M3):
    """(alpha, s) for the next step from the amax window ``hist`` (float32
    ring, slot ``pos`` holds the latest amax)."""
    h = np.ascontiguousarray(hist, np.float32)
    al, s = _fbuf(), _fbuf()
    _L().or_ds_scale_update(_p(h), h.size, int(pos), algo, fmt, _p(al), _p(s))
    return al[0], s[0]


def dq_current_scaling(q, s, fmt=E4M3, out=F32):
    q = np.ascontiguousarray(q, np.uint8)
    R, C = q.shape
    y = np.empty((R, C), np.float32 if out == F32 else np.uint16)
    _L().or_dq_current_scaling(_p(q), float(s), R, C, fmt, out, _p(y))
    return y


@dataclass
class MX:
    q_row: np.ndarray | None
    e8m0_row: np.ndarray | None
    q_col: np.ndarray | None
    e8m0_col: np.ndarray | None


def mxfp8(x, fmt=E4M3, rowwise=True, colwise=True):
    x, dt = _x(x)
    M, K = x.shape
    q_row = np.empty((M, K), np.uint8) if rowwise else None
    e_row = np.empty((M, K // 32), np.uint8) if rowwise else None
    q_col = np.empty((M, K), np.uint8) if colwise else None
    e_col = np.empty((M // 32, K), np.uint8) if colwise else None
    _L().or_mxfp8(_p(x), dt, M, K, fmt, _p(q_row), _p(e_row), _p(q_col), _p(e_col))
    return MX(q_row, e_row, q_col, e_col)


def dq_mxfp8(q, e8m0, fmt=E4M3, direction=ROW, out=F32):
    q = np.ascontiguousarray(q, np.uint8)
    e8m0 = np.ascontiguousarray(e8m0, np.uint8)
    R, C = q.shape
    y = np.empty((R, C), np.float32 if out == F32 else np.uint16)
    _L().or_dq_mxfp8(_p(q), _p(e8m0), R, C, fmt, direction, out, _p(y))
    return y


def mxfp8_requant_col(q_row, e8m0_row, fmt=E4M3):
    """Columnwise MXFP8 of the rowwise dequantization (the re-quantize step)."""
    q_row = np.ascontiguousarray(q_row, np.uint8)
    e8m0_row = np.ascontiguousarray(e8m0_row, np.uint8)
    M, K = q_row.shape
    q_col = np.empty((M, K), np.uint8)
    e_col = np.empty((M // 32, K), np.uint8)
    _L().or_mxfp8_requant_col(_p(q_row), _p(e8m0_row), M, K, fmt, _p(q_col), _p(e_col))
    return q_col, e_col


@dataclass
class BW:
    q_row: np.ndarray | None
    s_row: np.ndarray | None
    q_colT: np.ndarray | None
    s_colT: np.ndarray | None


def blockwise(x, tile=T1x128, rowwise=True, colwise=False):
    x, dt = _x(x)
    M, K = x.shape
    q_row = np.empty((M, K), np.uint8) if rowwise else None
    q_colT = np.empty((K, M), np.uint8) if colwise else None
    if tile == T1x128:
        s_row = np.empty((M, K // 128), np.float32) if rowwise else None
        s_colT = np.empty((K, M // 128), np.float32) if colwise else None
    else:
        s_row = np.empty((M // 128, K // 128), np.float32) if rowwise else None
        s_colT = np.empty((K // 128, M // 128), np.float32) if colwise else None
    _L().or_blockwise(_p(x), dt, M, K, tile, _p(q_row), _p(s_row), _p(q_colT), _p(s_colT))
    return BW(q_row, s_row, q_colT, s_colT)


@dataclass
class BWMX:
    q_row: np.ndarray | None       # [M, K] E4M3 codes
    e8m0_row: np.ndarray | None    # [M, K/32], the tile's code repeated
    q_colT: np.ndarray | None      # [K, M]
    e8m0_colT: np.ndarray | None   # [K, M/32]


def blockwise_mx(x, tile=T1x128, rowwise=True, colwise=False):
    """Blockwise tiles with power-of-two scales stored as MXFP8 (R-BWMX):
    both copies dequantize with dq_mxfp8(..., direction=ROW)."""
    x, dt = _x(x)
    M, K = x.shape
    q_row = np.empty((M, K), np.uint8) if rowwise else None
    e_row = np.empty((M, K // 32), np.uint8) if rowwise else None
    q_colT = np.empty((K, M), np.uint8) if colwise else None
    e_colT = np.empty((K, M // 32), np.uint8) if colwise else None
    _L().or_blockwise_mx(_p(x), dt, M, K, tile, _p(q_row), _p(e_row), _p(q_colT), _p(e_colT))
    return BWMX(q_row, e_row, q_colT, e_colT)


def dq_blockwise(q, s, tile=T1x128, out=F32):
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.float32)
    R, C = q.shape
    y = np.empty((R, C), np.float32 if out == F32 else np.uint16)
    _L().or_dq_blockwise(_p(q), _p(s), R, C, tile, out, _p(y))
    return y


@dataclass
class NV:
    q_row: np.ndarray | None
    sb_row: np.ndarray | None
    q_colT: np.ndarray | None
    sb_colT: np.ndarray | None
    amax: np.float32
    s_global: np.float32


def nvfp4_global(a):
    al, s = _fbuf(), _fbuf()
    _L().or_nvfp4_global(float(a), _p(al), _p(s))
    return al[0], s[0]


def nvfp4(x, blk=B1x16, rnd=RN, seed=0, offset=0, rowwise=True, colwise=False, amax_in=None):
    x, dt = _x(x)
    M, K = x.shape
    q_row = np.zeros((M, K // 2), np.uint8) if rowwise else None
    q_colT = np.zeros((K, M // 2), np.uint8) if colwise else None
    if blk == B1x16:
        sb_row = np.empty((M, K // 16), np.uint8) if rowwise else None
        sb_colT = np.empty((K, M // 16), np.uint8) if colwise else None
    else:
        sb_row = np.empty((M // 16, K // 16), np.uint8) if rowwise else None
        sb_colT = np.empty((K // 16, M // 16), np.uint8) if colwise else None
    a_out, s_out = _fbuf(), _fbuf()
    a_in = None if amax_in is None else _fbuf(amax_in)
    _L().or_nvfp4(_p(x), dt, M, K, blk, rnd, seed, offset, _p(a_in),
                  _p(q_row), _p(sb_row), _p(q_colT), _p(sb_colT), _p(a_out), _p(s_out))
    return NV(q_row, sb_row, q_colT, sb_colT, a_out[0], s_out[0])


def rht16(v, sign_mask):
    """The 16-point random Hadamard transform of one group (float32[16])."""
    v = np.array(v, np.float32).copy()
    assert v.size == 16
    _L().or_rht16(_p(v), int(sign_mask) & 0xFFFF)
    return v


def rht_cols(x, sign_mask):
    """FP32 [M, K]: the transform along M of every column's 16-row groups."""
    x, dt = _x(x)
    M, K = x.shape
    xr = np.empty((M, K), np.float32)
    _L().or_rht_cols(_p(x), dt, M, K, int(sign_mask) & 0xFFFF, _p(xr))
    return xr


def nvfp4_rht_colT(x, sign_mask, rnd=RN, seed=0, offset=0, amax_in=None):
    """Columnwise NVFP4 copy of the transformed tensor: (q_colT [K, M/2],
    sb_colT [K, M/16], amax of the transformed tensor, s_global)."""
    x, dt = _x(x)
    M, K = x.shape
    q_colT = np.zeros((K, M // 2), np.uint8)
    sb_colT = np.empty((K, M // 16), np.uint8)
    a_out, s_out = _fbuf(), _fbuf()
    a_in = None if amax_in is None else _fbuf(amax_in)
    _L().or_nvfp4_rht_colT(_p(x), dt, M, K, int(sign_mask) & 0xFFFF, rnd, seed, offset, _p(a_in), _p(q_colT),
                           _p(sb_colT), _p(a_out), _p(s_out))
    return q_colT, sb_colT, a_out[0], s_out[0]


def dq_nvfp4(q, sb, s_global, blk=B1x16, out=F32):
    q = np.ascontiguousarray(q, np.uint8)
    sb = np.ascontiguousarray(sb, np.uint8)
    R, C = q.shape[0], q.shape[1] * 2
    y = np.empty((R, C), np.float32 if out == F32 else np.uint16)
    _L().or_dq_nvfp4(_p(q), _p(sb), float(s_global), R, C, blk, out, _p(y))
    return y
