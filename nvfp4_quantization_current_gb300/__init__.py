"""GB300 (sm_103a) tensor quantizers for FP8 / FP4 mixed-precision training.

A thin Python binding over the C ABI of ``libq.so`` (declared in
``include/q.h``).  This module only marshals arguments: it allocates output
tensors with torch (device memory), passes raw pointers and the current CUDA
stream, and raises on any non-zero status.  Every step of the computation
runs in the library's CUDA kernels; there is no CPU path.  If ``libq.so`` is
missing (build it with ``python -m nvfp4_quantization_current_gb300.build``
or ``__graft_entry__.build()``) every call raises.

Recipes (each with its dequantizer, rowwise and columnwise outputs):

* :func:`q_current_scaling` -- per-tensor current scaling to E4M3 / E5M2
  ("FP8 Current Scaling: quantization, scaling and precision bounds",
  section "Current Scaling");
* :func:`q_delayed_scaling` / :class:`DelayedScaling` -- per-tensor delayed
  scaling: the scale comes from a window of earlier amaxes and the step's
  amax is recorded in the same read ("Mixed-precision training: fp16 to
  fp8", "Per-tensor delayed scaling");
* :func:`q_mxfp8` -- 1x32 blocks with E8M0 scales ("Mixed-precision
  training: fp16 to fp8", section "MXFP8");
* :func:`q_mxfp8_requant_col` -- MXFP8 rowwise codes to columnwise codes
  (dequantize + re-quantize, same page, "FP8 communication");
* :func:`q_blockwise` -- DeepSeek-V3-like 1x128 / 128x128 FP32-scaled E4M3
  (same page, recipe 4);
* :func:`q_nvfp4` -- E2M1 with E4M3 1x16 / 16x16 block scales and an FP32
  tensor scale, RTNE or stochastic rounding (same page, "NVFP4"; "From BF16
  to FP8/FP4 ...", section 2.4);
* :func:`q_nvfp4_rht_colT` -- the columnwise NVFP4 copy of the random
  Hadamard transform of x, for the weight-gradient GEMM inputs ("From BF16
  to FP8/FP4 ...", sections 2.4 and 5.6).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq.so")

# enums of include/q.h
Q_OK, Q_ERR_ARG, Q_ERR_SHAPE, Q_ERR_ALIGN, Q_ERR_DTYPE, Q_ERR_CUDA = range(6)
Q_BF16, Q_F32 = 0, 1
Q_E4M3, Q_E5M2 = 0, 1
Q_T1x128, Q_T128x128 = 0, 1
Q_B1x16, Q_B16x16 = 0, 1
Q_RN, Q_SR = 0, 1
Q_ROW, Q_COL = 0, 1
Q_AMAX_COMPUTE, Q_AMAX_GIVEN = 0, 1
Q_ST_NONFINITE, Q_ST_TIMEOUT = 1, 2

STATUS_NAMES = {Q_OK: "Q_OK", Q_ERR_ARG: "Q_ERR_ARG", Q_ERR_SHAPE: "Q_ERR_SHAPE", Q_ERR_ALIGN: "Q_ERR_ALIGN",
                Q_ERR_DTYPE: "Q_ERR_DTYPE", Q_ERR_CUDA: "Q_ERR_CUDA"}

# every exported entry point: name -> (restype, argtypes)
_P, _I64, _I, _U64, _U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32
SIGNATURES = {
    "q_last_error": (ctypes.c_char_p, []),
    "q_abi_version": (_I, []),
    "q_amax": (_I, [_P, _I, _I64, _P, _P, _P]),
    "q_current_scaling": (_I, [_P, _I, _I64, _I64, _I, _P, _P, _P, _I, _P, _P, _P]),
    "q_mxfp8": (_I, [_P, _I, _I64, _I64, _I, _P, _P, _P, _P, _P, _P]),
    "q_delayed_scaling": (_I, [_P, _I, _I64, _I64, _I, _P, _P, _P, _P, _P, _P, _P]),
    "q_delayed_scale_update": (_I, [_P, _I64, _I64, _I, _I, _P, _P]),
    "q_selftest_wait_timeout": (_I, [_P, _U64, _P]),
    "q_selftest_inject_launch_error": (_I, [_I]),
    "q_mxfp8_requant_col": (_I, [_P, _P, _I64, _I64, _I, _P, _P, _P, _P]),
    "q_blockwise": (_I, [_P, _I, _I64, _I64, _I, _P, _P, _P, _P, _P, _P]),
    "q_blockwise_mx": (_I, [_P, _I, _I64, _I64, _I, _P, _P, _P, _P, _P, _P]),
    "q_nvfp4_recipe": (_I, [_P, _I, _I64, _I64, _U32, _I, _U64, _U64, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "q_nvfp4_rht_amax2": (_I, [_P, _I, _I64, _I64, _U32, _P, _P, _P, _P]),
    "q_nvfp4": (_I, [_P, _I, _I64, _I64, _I, _I, _U64, _U64, _P, _P, _P, _P, _P, _I, _P, _P, _P]),
    "q_nvfp4_rht_amax": (_I, [_P, _I, _I64, _I64, _U32, _P, _P, _P]),
    "q_nvfp4_rht_colT": (_I, [_P, _I, _I64, _I64, _U32, _I, _U64, _U64, _P, _P, _P, _I, _P, _P, _P]),
    "dq_current_scaling": (_I, [_P, _P, _I64, _I64, _I, _I, _P, _P]),
    "dq_mxfp8": (_I, [_P, _P, _I64, _I64, _I, _I, _I, _P, _P]),
    "dq_blockwise": (_I, [_P, _P, _I64, _I64, _I, _I, _P, _P]),
    "dq_nvfp4": (_I, [_P, _P, _P, _I64, _I64, _I, _I, _P, _P]),
}

_lib = None


class QuantError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def lib():
    """The loaded ``libq.so`` (ctypes), with every signature declared.
    Raises if the library has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -m nvfp4_quantization_current_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != Q_OK:
        raise QuantError(name, st, lib().q_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _in(x: torch.Tensor):
    if not x.is_cuda:
        raise ValueError("input must be a CUDA tensor (the library has no CPU path)")
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("input must be a contiguous 2-D tensor")
    if x.dtype == torch.bfloat16:
        return Q_BF16
    if x.dtype == torch.float32:
        return Q_F32
    raise ValueError(f"input dtype {x.dtype} is not bfloat16 or float32")


def _fmt(fmt):
    return {"e4m3": Q_E4M3, "e5m2": Q_E5M2, Q_E4M3: Q_E4M3, Q_E5M2: Q_E5M2}[fmt]


def _out(dtype):
    return {torch.float32: Q_F32, torch.bfloat16: Q_BF16}[dtype]


def _u8(shape, dev):
    return torch.empty(shape, dtype=torch.uint8, device=dev)


def _f32(shape, dev):
    return torch.empty(shape, dtype=torch.float32, device=dev)


# ---------------------------------------------------------------------------
# a1: amax
# ---------------------------------------------------------------------------

def q_amax(x: torch.Tensor, out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """max|x| as a one-element FP32 device tensor."""
    dt = _in(x)
    out = _f32((1,), x.device) if out is None else out
    _call("q_amax", _ptr(x), dt, x.numel(), _ptr(out), _ptr(status), _stream(x.device))
    return out


# ---------------------------------------------------------------------------
# a1-a3: current scaling
# ---------------------------------------------------------------------------

@dataclass
class CurrentScalingTensor:
    q_row: Optional[torch.Tensor]     # [M, K] uint8 FP8 codes
    q_colT: Optional[torch.Tensor]    # [K, M] uint8 FP8 codes (transposed copy)
    amax: torch.Tensor                # (1,) FP32
    scale: torch.Tensor               # (1,) FP32, s = 1 / alpha
    fmt: int

    def dequantize(self, direction=Q_ROW, dtype=torch.float32):
        q = self.q_row if direction == Q_ROW else self.q_colT
        return dq_current_scaling(q, self.scale, self.fmt, dtype)


def alloc_current_scaling(M, K, device, fmt="e4m3", rowwise=True, colwise=False) -> CurrentScalingTensor:
    return CurrentScalingTensor(_u8((M, K), device) if rowwise else None, _u8((K, M), device) if colwise else None,
                                _f32((1,), device), _f32((1,), device), _fmt(fmt))


def q_current_scaling(x: torch.Tensor, fmt="e4m3", rowwise=True, colwise=False, amax: Optional[torch.Tensor] = None,
                      out: Optional[CurrentScalingTensor] = None, status: Optional[torch.Tensor] = None):
    """Per-tensor current scaling.  ``amax`` (a one-element device tensor)
    skips the amax pass and uses the given value (e.g. after a MAX
    all-reduce over shards)."""
    dt = _in(x)
    M, K = x.shape
    if out is None:
        out = alloc_current_scaling(M, K, x.device, fmt, rowwise, colwise)
    mode = Q_AMAX_COMPUTE
    if amax is not None:
        out.amax = amax
        mode = Q_AMAX_GIVEN
    _call("q_current_scaling", _ptr(x), dt, M, K, out.fmt, _ptr(out.q_row), _ptr(out.q_colT), _ptr(out.amax), mode,
          _ptr(out.scale), _ptr(status), _stream(x.device))
    return out


def dq_current_scaling(q: torch.Tensor, scale: torch.Tensor, fmt="e4m3", dtype=torch.float32, out=None):
    R, C = q.shape
    y = torch.empty((R, C), dtype=dtype, device=q.device) if out is None else out
    _call("dq_current_scaling", _ptr(q), _ptr(scale), R, C, _fmt(fmt), _out(dtype), _ptr(y), _stream(q.device))
    return y


# ---------------------------------------------------------------------------
# per-tensor delayed scaling
# ---------------------------------------------------------------------------

Q_HIST_MAX, Q_HIST_MOST_RECENT = 0, 1


def _algo(algo):
    return {"max": Q_HIST_MAX, "most_recent": Q_HIST_MOST_RECENT, Q_HIST_MAX: Q_HIST_MAX,
            Q_HIST_MOST_RECENT: Q_HIST_MOST_RECENT}[algo]


def q_delayed_scaling(x: torch.Tensor, ds: torch.Tensor, amax_out: torch.Tensor, fmt="e4m3", rowwise=True,
                      colwise=False, out: Optional[CurrentScalingTensor] = None,
                      status: Optional[torch.Tensor] = None) -> CurrentScalingTensor:
    """One delayed-scaling cast: codes of x with alpha = ds[0] (the pair
    [alpha, s] from the previous :func:`q_delayed_scale_update`), max|x|
    written to ``amax_out`` (this step's window slot) and s = ds[1] to the
    result's ``scale``.  Reads x once."""
    dt = _in(x)
    M, K = x.shape
    if out is None:
        out = alloc_current_scaling(M, K, x.device, fmt, rowwise, colwise)
    out.amax = amax_out
    _call("q_delayed_scaling", _ptr(x), dt, M, K, out.fmt, _ptr(out.q_row), _ptr(out.q_colT), _ptr(ds),
          _ptr(amax_out), _ptr(out.scale), _ptr(status), _stream(x.device))
    return out


def q_delayed_scale_update(hist: torch.Tensor, pos: int, ds: torch.Tensor, fmt="e4m3", algo="max") -> torch.Tensor:
    """ds = [alpha, s] for the next step from the amax window ``hist`` (FP32,
    slot ``pos`` the latest)."""
    _call("q_delayed_scale_update", _ptr(hist), hist.numel(), int(pos), _algo(algo), _fmt(fmt), _ptr(ds),
          _stream(hist.device))
    return ds


class DelayedScaling:
    """Delayed-scaling state of one tensor: a window of ``history_len`` amaxes
    (a ring, zero-initialized), the pair [alpha, s] (initially [1, 1]) and
    the step counter.  ``quantize`` runs one step: the cast with the current
    pair (recording the step's amax in slot ``step % history_len``), an
    optional MAX all-reduce of that slot over ``group`` (so that every shard
    of a distributed tensor keeps the same window), and the update of the
    pair from the window (``algo`` "max" or "most_recent").  The result's
    ``amax`` is a view of the window slot, overwritten ``history_len`` steps
    later."""

    def __init__(self, fmt="e4m3", history_len=1024, algo="max", device="cuda"):
        if history_len < 1:
            raise ValueError("history_len must be >= 1")
        self.fmt, self.algo = _fmt(fmt), _algo(algo)
        self.hist = torch.zeros(history_len, dtype=torch.float32, device=device)
        self.ds = torch.ones(2, dtype=torch.float32, device=device)
        self.step = 0

    def quantize(self, x: torch.Tensor, rowwise=True, colwise=False, out: Optional[CurrentScalingTensor] = None,
                 status: Optional[torch.Tensor] = None, group=None) -> CurrentScalingTensor:
        pos = self.step % self.hist.numel()
        slot = self.hist[pos:pos + 1]
        res = q_delayed_scaling(x, self.ds, slot, self.fmt, rowwise, colwise, out, status)
        if group is not None:
            from .distributed import allreduce_amax_
            allreduce_amax_(slot, group)
        q_delayed_scale_update(self.hist, pos, self.ds, self.fmt, self.algo)
        self.step += 1
        return res


# ---------------------------------------------------------------------------
# a4/a5: MXFP8
# ---------------------------------------------------------------------------

@dataclass
class MXFP8Tensor:
    q_row: Optional[torch.Tensor]      # [M, K] codes, 1x32 blocks
    e8m0_row: Optional[torch.Tensor]   # [M, K/32]
    q_col: Optional[torch.Tensor]      # [M, K] codes, 32x1 blocks
    e8m0_col: Optional[torch.Tensor]   # [M/32, K]
    fmt: int

    def dequantize(self, direction=Q_ROW, dtype=torch.float32):
        if direction == Q_ROW:
            return dq_mxfp8(self.q_row, self.e8m0_row, self.fmt, Q_ROW, dtype)
        return dq_mxfp8(self.q_col, self.e8m0_col, self.fmt, Q_COL, dtype)


def alloc_mxfp8(M, K, device, fmt="e4m3", rowwise=True, colwise=True) -> MXFP8Tensor:
    return MXFP8Tensor(_u8((M, K), device) if rowwise else None, _u8((M, K // 32), device) if rowwise else None,
                       _u8((M, K), device) if colwise else None, _u8((M // 32, K), device) if colwise else None,
                       _fmt(fmt))


def q_mxfp8(x: torch.Tensor, fmt="e4m3", rowwise=True, colwise=True, out: Optional[MXFP8Tensor] = None,
            status: Optional[torch.Tensor] = None):
    dt = _in(x)
    M, K = x.shape
    out = alloc_mxfp8(M, K, x.device, fmt, rowwise, colwise) if out is None else out
    _call("q_mxfp8", _ptr(x), dt, M, K, out.fmt, _ptr(out.q_row), _ptr(out.e8m0_row), _ptr(out.q_col),
          _ptr(out.e8m0_col), _ptr(status), _stream(x.device))
    return out


def q_mxfp8_requant_col(q_row: torch.Tensor, e8m0_row: torch.Tensor, fmt="e4m3", out: Optional[MXFP8Tensor] = None,
                        status: Optional[torch.Tensor] = None) -> MXFP8Tensor:
    """Columnwise MXFP8 codes and scales from the rowwise ones: each element is
    dequantized with its 1x32 row-block scale and re-quantized in 32x1 column
    blocks.  Returns an MXFP8Tensor with only the columnwise half set (or
    fills ``out.q_col`` / ``out.e8m0_col``)."""
    M, K = q_row.shape
    if out is None:
        out = alloc_mxfp8(M, K, q_row.device, fmt, rowwise=False, colwise=True)
    _call("q_mxfp8_requant_col", _ptr(q_row), _ptr(e8m0_row), M, K, _fmt(fmt), _ptr(out.q_col), _ptr(out.e8m0_col),
          _ptr(status), _stream(q_row.device))
    return out


def dq_mxfp8(q, e8m0, fmt="e4m3", direction=Q_ROW, dtype=torch.float32, out=None):
    R, C = q.shape
    y = torch.empty((R, C), dtype=dtype, device=q.device) if out is None else out
    _call("dq_mxfp8", _ptr(q), _ptr(e8m0), R, C, _fmt(fmt), direction, _out(dtype), _ptr(y), _stream(q.device))
    return y


# ---------------------------------------------------------------------------
# a6/a7: blockwise
# ---------------------------------------------------------------------------

@dataclass
class BlockwiseTensor:
    q_row: Optional[torch.Tensor]
    s_row: Optional[torch.Tensor]
    q_colT: Optional[torch.Tensor]
    s_colT: Optional[torch.Tensor]
    tile: int

    def dequantize(self, direction=Q_ROW, dtype=torch.float32):
        if direction == Q_ROW:
            return dq_blockwise(self.q_row, self.s_row, self.tile, dtype)
        return dq_blockwise(self.q_colT, self.s_colT, self.tile, dtype)


def _tile(tile):
    return {"1x128": Q_T1x128, "128x128": Q_T128x128, Q_T1x128: Q_T1x128, Q_T128x128: Q_T128x128}[tile]


def alloc_blockwise(M, K, device, tile="1x128", rowwise=True, colwise=False) -> BlockwiseTensor:
    t = _tile(tile)
    if t == Q_T1x128:
        sr, sc = (M, K // 128), (K, M // 128)
    else:
        sr, sc = (M // 128, K // 128), (K // 128, M // 128)
    return BlockwiseTensor(_u8((M, K), device) if rowwise else None, _f32(sr, device) if rowwise else None,
                           _u8((K, M), device) if colwise else None, _f32(sc, device) if colwise else None, t)


def q_blockwise(x: torch.Tensor, tile="1x128", rowwise=True, colwise=False, out: Optional[BlockwiseTensor] = None,
                status: Optional[torch.Tensor] = None):
    dt = _in(x)
    M, K = x.shape
    out = alloc_blockwise(M, K, x.device, tile, rowwise, colwise) if out is None else out
    _call("q_blockwise", _ptr(x), dt, M, K, out.tile, _ptr(out.q_row), _ptr(out.s_row), _ptr(out.q_colT),
          _ptr(out.s_colT), _ptr(status), _stream(x.device))
    return out


def dq_blockwise(q, s, tile="1x128", dtype=torch.float32, out=None):
    R, C = q.shape
    y = torch.empty((R, C), dtype=dtype, device=q.device) if out is None else out
    _call("dq_blockwise", _ptr(q), _ptr(s), R, C, _tile(tile), _out(dtype), _ptr(y), _stream(q.device))
    return y


@dataclass
class BlockwiseMXTensor:
    """Blockwise tiles held as MXFP8: E4M3 codes with the tile's power-of-two
    scale as an E8M0 code once per 32 elements (MXFP8 row layout for both
    copies, so an MXFP8 GEMM consumes them)."""
    q_row: Optional[torch.Tensor]       # [M, K] E4M3 codes
    e8m0_row: Optional[torch.Tensor]    # [M, K/32], the tile's code repeated
    q_colT: Optional[torch.Tensor]      # [K, M] (128x1 blocks along M, or the 2D codes transposed)
    e8m0_colT: Optional[torch.Tensor]   # [K, M/32]
    tile: int

    def dequantize(self, direction=Q_ROW, dtype=torch.float32):
        if direction == Q_ROW:
            return dq_mxfp8(self.q_row, self.e8m0_row, Q_E4M3, Q_ROW, dtype)
        return dq_mxfp8(self.q_colT, self.e8m0_colT, Q_E4M3, Q_ROW, dtype)


def alloc_blockwise_mx(M, K, device, tile="1x128", rowwise=True, colwise=False) -> BlockwiseMXTensor:
    return BlockwiseMXTensor(_u8((M, K), device) if rowwise else None, _u8((M, K // 32), device) if rowwise else None,
                             _u8((K, M), device) if colwise else None, _u8((K, M // 32), device) if colwise else None,
                             _tile(tile))


def q_blockwise_mx(x: torch.Tensor, tile="1x128", rowwise=True, colwise=False,
                   out: Optional[BlockwiseMXTensor] = None, status: Optional[torch.Tensor] = None):
    """Blockwise 1x128 / 128x128 quantization with power-of-two tile scales
    stored as MXFP8 E8M0 codes (the blockwise recipe emulated on MXFP8)."""
    dt = _in(x)
    M, K = x.shape
    out = alloc_blockwise_mx(M, K, x.device, tile, rowwise, colwise) if out is None else out
    _call("q_blockwise_mx", _ptr(x), dt, M, K, out.tile, _ptr(out.q_row), _ptr(out.e8m0_row), _ptr(out.q_colT),
          _ptr(out.e8m0_colT), _ptr(status), _stream(x.device))
    return out


# ---------------------------------------------------------------------------
# a8-a11: NVFP4
# ---------------------------------------------------------------------------

@dataclass
class NVFP4Tensor:
    q_row: Optional[torch.Tensor]     # [M, K/2] packed E2M1
    sb_row: Optional[torch.Tensor]    # [M, K/16] (1x16) or [M/16, K/16] (16x16), E4M3 codes
    q_colT: Optional[torch.Tensor]    # [K, M/2]
    sb_colT: Optional[torch.Tensor]   # [K, M/16] or [K/16, M/16]
    amax: torch.Tensor
    s_global: torch.Tensor
    blk: int

    def dequantize(self, direction=Q_ROW, dtype=torch.float32):
        if direction == Q_ROW:
            return dq_nvfp4(self.q_row, self.sb_row, self.s_global, self.blk, dtype)
        return dq_nvfp4(self.q_colT, self.sb_colT, self.s_global, self.blk, dtype)


def _blk(blk):
    return {"1x16": Q_B1x16, "16x16": Q_B16x16, Q_B1x16: Q_B1x16, Q_B16x16: Q_B16x16}[blk]


def alloc_nvfp4(M, K, device, blk="1x16", rowwise=True, colwise=False) -> NVFP4Tensor:
    b = _blk(blk)
    if b == Q_B1x16:
        sr, sc = (M, K // 16), (K, M // 16)
    else:
        sr, sc = (M // 16, K // 16), (K // 16, M // 16)
    return NVFP4Tensor(_u8((M, K // 2), device) if rowwise else None, _u8(sr, device) if rowwise else None,
                       _u8((K, M // 2), device) if colwise else None, _u8(sc, device) if colwise else None,
                       _f32((1,), device), _f32((1,), device), b)


def q_nvfp4(x: torch.Tensor, blk="1x16", rounding="rn", seed=0, offset=0, rowwise=True, colwise=False,
            amax: Optional[torch.Tensor] = None, out: Optional[NVFP4Tensor] = None,
            status: Optional[torch.Tensor] = None):
    """NVFP4.  rounding "rn" (round to nearest even) or "sr" (stochastic,
    Philox4x32-10 keyed by ``seed``, counter offset ``offset``)."""
    dt = _in(x)
    M, K = x.shape
    out = alloc_nvfp4(M, K, x.device, blk, rowwise, colwise) if out is None else out
    rnd = {"rn": Q_RN, "sr": Q_SR, Q_RN: Q_RN, Q_SR: Q_SR}[rounding]
    mode = Q_AMAX_COMPUTE
    if amax is not None:
        out.amax = amax
        mode = Q_AMAX_GIVEN
    _call("q_nvfp4", _ptr(x), dt, M, K, out.blk, rnd, int(seed), int(offset), _ptr(out.q_row), _ptr(out.sb_row),
          _ptr(out.q_colT), _ptr(out.sb_colT), _ptr(out.amax), mode, _ptr(out.s_global), _ptr(status),
          _stream(x.device))
    return out


def q_nvfp4_rht_amax(x: torch.Tensor, sign_mask: int, out: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """max|x'| of the random Hadamard transform that :func:`q_nvfp4_rht_colT`
    applies (one-element FP32 device tensor), e.g. to all-reduce over shards
    and pass back as its ``amax``."""
    dt = _in(x)
    M, K = x.shape
    out = _f32((1,), x.device) if out is None else out
    _call("q_nvfp4_rht_amax", _ptr(x), dt, M, K, int(sign_mask), _ptr(out), _ptr(status), _stream(x.device))
    return out


def q_nvfp4_rht_amax2(x: torch.Tensor, sign_mask: int, out: Optional[tuple] = None,
                      status: Optional[torch.Tensor] = None):
    """(max|x'|, max|x|) in one read of x, x' the random Hadamard transform
    of q_nvfp4_rht_amax: the two maxima of q_nvfp4_recipe, for callers that
    reduce them across shards before the casts."""
    dt = _in(x)
    M, K = x.shape
    a_rht, a_x = (_f32((1,), x.device), _f32((1,), x.device)) if out is None else out
    _call("q_nvfp4_rht_amax2", _ptr(x), dt, M, K, sign_mask, _ptr(a_rht), _ptr(a_x), _ptr(status), _stream(x.device))
    return a_rht, a_x


def q_nvfp4_recipe(x: torch.Tensor, sign_mask: int, rounding="rn", seed=0, offset=0,
                   amax_row: Optional[torch.Tensor] = None, amax_col: Optional[torch.Tensor] = None,
                   out: Optional[tuple] = None, status: Optional[torch.Tensor] = None):
    """Both NVFP4 copies of x as the training recipe uses them: the rowwise
    1x16 copy of x and the columnwise copy of its random Hadamard transform,
    with one amax pass for both maxima (or both given as one-element device
    tensors: max|x| as ``amax_row``, max|x'| as ``amax_col``), then one pass
    for both copies of a BF16 x.  Returns (row, colT), two NVFP4Tensor whose
    outputs equal q_nvfp4(x, rowwise only) and q_nvfp4_rht_colT(x, sign_mask)
    with the same seed and offset."""
    dt = _in(x)
    M, K = x.shape
    if (amax_row is None) != (amax_col is None):
        raise ValueError("give both maxima or neither")
    if out is None:
        out = (alloc_nvfp4(M, K, x.device, "1x16", rowwise=True, colwise=False),
               alloc_nvfp4(M, K, x.device, "1x16", rowwise=False, colwise=True))
    row, col = out
    mode = Q_AMAX_COMPUTE
    if amax_row is not None:
        row.amax, col.amax = amax_row, amax_col
        mode = Q_AMAX_GIVEN
    rnd = {"rn": Q_RN, "sr": Q_SR, Q_RN: Q_RN, Q_SR: Q_SR}[rounding]
    _call("q_nvfp4_recipe", _ptr(x), dt, M, K, sign_mask, rnd, seed, offset, _ptr(row.q_row),
          _ptr(row.sb_row), _ptr(row.amax), _ptr(row.s_global), _ptr(col.q_colT), _ptr(col.sb_colT), _ptr(col.amax),
          _ptr(col.s_global), mode, _ptr(status), _stream(x.device))
    return row, col


def q_nvfp4_rht_colT(x: torch.Tensor, sign_mask: int, rounding="rn", seed=0, offset=0,
                     amax: Optional[torch.Tensor] = None, out: Optional[NVFP4Tensor] = None,
                     status: Optional[torch.Tensor] = None) -> NVFP4Tensor:
    """Columnwise NVFP4 copy (1x16 blocks along M, stored [K, M/2]) of the
    random Hadamard transform of x: (1/4) H D on each 16-row group of every
    column, D the signs of the 16-bit ``sign_mask``.  For the inputs of the
    weight-gradient GEMM; use the same mask for both of its operands.
    ``amax`` (one-element device tensor) gives the transformed tensor's
    amax instead of computing it.  Returns an NVFP4Tensor with only the
    columnwise half set."""
    dt = _in(x)
    M, K = x.shape
    out = alloc_nvfp4(M, K, x.device, "1x16", rowwise=False, colwise=True) if out is None else out
    rnd = {"rn": Q_RN, "sr": Q_SR, Q_RN: Q_RN, Q_SR: Q_SR}[rounding]
    mode = Q_AMAX_COMPUTE
    if amax is not None:
        out.amax = amax
        mode = Q_AMAX_GIVEN
    _call("q_nvfp4_rht_colT", _ptr(x), dt, M, K, int(sign_mask), rnd, int(seed), int(offset), _ptr(out.q_colT),
          _ptr(out.sb_colT), _ptr(out.amax), mode, _ptr(out.s_global), _ptr(status), _stream(x.device))
    return out


def selftest_wait_timeout(status: torch.Tensor, wait_ns: int = 50_000_000) -> torch.Tensor:
    """Diagnostic: one warp waits ``wait_ns`` on a barrier nothing completes and
    reports Q_ST_TIMEOUT in ``status`` (a one-element int32 device tensor),
    exercising the bounded-wait path every kernel uses."""
    _call("q_selftest_wait_timeout", _ptr(status), int(wait_ns), _stream(status.device))
    return status


def dq_nvfp4(q, sb, s_global, blk="1x16", dtype=torch.float32, out=None):
    R, C = q.shape[0], q.shape[1] * 2
    y = torch.empty((R, C), dtype=dtype, device=q.device) if out is None else out
    _call("dq_nvfp4", _ptr(q), _ptr(sb), _ptr(s_global), R, C, _blk(blk), _out(dtype), _ptr(y), _stream(q.device))
    return y


__all__ = [n for n in dir() if n.startswith(("q_", "dq_", "alloc_", "Q_"))] + [
    "CurrentScalingTensor", "DelayedScaling", "MXFP8Tensor", "BlockwiseTensor", "BlockwiseMXTensor", "NVFP4Tensor",
    "QuantError", "lib", "SIGNATURES"]
