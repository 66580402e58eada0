"""Seeded synthetic inputs shared by the tests and the benchmark.

This module only draws random numbers and rounds them to BF16 (through
torch's own RTNE conversion).  It holds none of the quantizers' arithmetic,
and imports neither the library nor the oracle.

The full-size workloads follow the shapes of the pages' training setups:
hidden 4096 / FFN 14336 / sequence 8192 (the Megatron Llama-like baseline of
"From BF16 to FP8/FP4 ...", section 4.2) and a 7168 / 18432 DeepSeek-V3-like
layer, each drawn from a stated distribution:

=====  ====  =========================================================
name   seed  tensors (numpy default_rng(seed), FP32, then BF16 RTNE)
=====  ====  =========================================================
cs1    0     x 1024x1024 FP32 N(0,1) with 16 outliers of +-1000
mx2    1     act 8192x4096 N(0,1) * per-row lognormal(0,1)
bw3    2     act 16384x7168 N(0,1); w 7168x18432 N(0,0.02)
hy4    3     grad 8192x14336 Student-t(3) * 1e-3; w 14336x4096 N(0,0.02)
nv5    4     act 8192x4096 N(0,1); grad same shape Student-t(3);
             w 4096x4096 N(0,0.02)
=====  ====  =========================================================
"""
from __future__ import annotations

import numpy as np
import torch


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 array -> uint16 array of BF16 bit patterns (torch RTNE)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# distributions (one rng per call; the draw order is part of the recipe)
# ---------------------------------------------------------------------------

def normal(rng, shape, std=1.0):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def lognormal_rows(rng, shape):
    z = rng.standard_normal(shape, dtype=np.float32)
    m = rng.lognormal(0.0, 1.0, (shape[0], 1)).astype(np.float32)
    return (z * m).astype(np.float32)


def student_t(rng, shape, df=3.0, scale=1.0):
    return (rng.standard_t(df, shape).astype(np.float32) * np.float32(scale)).astype(np.float32)


def with_outliers(rng, x, count=16, value=1000.0):
    flat = x.reshape(-1)
    pos = rng.choice(flat.size, count, replace=False)
    signs = rng.choice(np.array([-1.0, 1.0], np.float32), count)
    flat[pos] = signs * np.float32(value)
    return x


def gen(kind: str, shape, seed: int, bf16: bool = True) -> np.ndarray:
    """One tensor of a named distribution.  kind: normal | lognormal_rows |
    t3 (Student-t(3)) | grad (Student-t(3) * 1e-3) | weight (N(0, 0.02)) |
    outliers (N(0,1) with 16 entries of +-1000).  Returns BF16 bits (uint16)
    or FP32."""
    rng = np.random.default_rng(seed)
    if kind == "normal":
        a = normal(rng, shape)
    elif kind == "lognormal_rows":
        a = lognormal_rows(rng, shape)
    elif kind == "t3":
        a = student_t(rng, shape)
    elif kind == "grad":
        a = student_t(rng, shape, scale=1e-3)
    elif kind == "weight":
        a = normal(rng, shape, std=0.02)
    elif kind == "outliers":
        a = with_outliers(rng, normal(rng, shape), count=min(16, int(np.prod(shape))))
    else:
        raise ValueError(kind)
    return to_bf16_bits(a) if bf16 else a


# ---------------------------------------------------------------------------
# the five full-size workloads
# ---------------------------------------------------------------------------

WORKLOADS = {
    "cs1": dict(seed=0, tensors={"x": ((1024, 1024), "outliers", False)}),
    "mx2": dict(seed=1, tensors={"act": ((8192, 4096), "lognormal_rows", True)}),
    "bw3": dict(seed=2, tensors={"act": ((16384, 7168), "normal", True),
                                 "w": ((7168, 18432), "weight", True)}),
    "hy4": dict(seed=3, tensors={"grad": ((8192, 14336), "grad", True),
                                 "w": ((14336, 4096), "weight", True)}),
    "nv5": dict(seed=4, tensors={"act": ((8192, 4096), "normal", True),
                                 "grad": ((8192, 4096), "t3", True),
                                 "w": ((4096, 4096), "weight", True)}),
}

# The worked example of "FP8 Current Scaling ..." section "Current Scaling".
EXAMPLE_X = np.array([[-1000.0, 100.0, 1000.0]], np.float32)


def workload(name: str, scale_rows: float = 1.0) -> dict:
    """Tensors of one workload.  Tensor j of workload `name` draws from
    default_rng(seed + 1000 * j) so that each tensor can be regenerated alone.
    scale_rows < 1 shrinks M (kept a multiple of 256) for quick runs."""
    spec = WORKLOADS[name]
    out = {}
    for j, (tname, (shape, kind, bf16)) in enumerate(spec["tensors"].items()):
        M, K = shape
        if scale_rows != 1.0:
            M = max(256, int(M * scale_rows) // 256 * 256)
        out[tname] = gen(kind, (M, K), spec["seed"] + 1000 * j, bf16=bf16)
    return out


def sample_rows(n_rows: int, k: int, seed: int) -> np.ndarray:
    """Sorted distinct row indices for sampled full-size parity checks."""
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n_rows, size=min(k, n_rows), replace=False))
