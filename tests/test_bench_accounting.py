"""The benchmark's algorithmic bytes (the numerator of every GB/s figure and
of the roofline) against formulas written independently of the bench code:
input bytes times the reads the recipe needs, plus every output.  The step
is built on small CPU tensors (building allocates outputs only; nothing
runs), so this needs no GPU."""
import importlib.util
import os

import pytest
import torch

import nvfp4_quantization_current_gb300 as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


SHAPES = {"cs1": {"x": ((64, 80), torch.float32)},
          "mx2": {"act": ((64, 128), torch.bfloat16)},
          "bw3": {"act": ((256, 384), torch.bfloat16), "w": ((256, 256), torch.bfloat16)},
          "hy4": {"grad": ((64, 96), torch.bfloat16), "w": ((96, 64), torch.bfloat16)},
          "nv5": {"act": ((64, 128), torch.bfloat16), "grad": ((64, 128), torch.bfloat16),
                  "w": ((128, 64), torch.bfloat16)}}


def expected(name, M, K, b):
    """Bytes of one call on an [M, K] input of b-byte elements."""
    E = M * K
    table = {
        "cs_e4m3 row+colT": 2 * E * b + 2 * E + 4 + 4,          # amax pass + cast; codes both ways, s, amax read
        "cs_e5m2 row+colT": 2 * E * b + 2 * E + 4 + 4,
        "ds_e5m2 row+colT": E * b + 2 * E + 4 + 4 + 8 + 1024 * 4 + 8,   # one read; s, slot, [alpha, s]; window update
        "mxfp8_e4m3 row+col": E * b + 2 * E + 2 * (E // 32),
        "mxfp8_requant row->col": 2 * E + 2 * (E // 32),
        "dq_mxfp8 row->bf16": E + E // 32 + 2 * E,
        "dq_mxfp8 col->bf16": E + E // 32 + 2 * E,
        "blockwise_1x128 row+colT": E * b + 2 * E + 2 * 4 * (E // 128),
        "blockwise_128x128 row+colT": E * b + 2 * E + 2 * 4 * (E // 16384),
        "dq_blockwise_1x128 row->bf16": E + 4 * (E // 128) + 2 * E,
        "dq_blockwise_128x128 row->bf16": E + 4 * (E // 16384) + 2 * E,
        "blockwise_mx_1x128 row+colT": E * b + 2 * E + 2 * (E // 32),
        "blockwise_mx_128x128 row+colT": E * b + 2 * E + 2 * (E // 32),
        "nvfp4_1x16_rn row+colT": 2 * E * b + E + 2 * (E // 16) + 4 + 4,   # amax pass; packed codes both ways
        "nvfp4_1x16_sr row+colT": 2 * E * b + E + 2 * (E // 16) + 4 + 4,
        "nvfp4_16x16_rn row+colT": 2 * E * b + E + 2 * (E // 256) + 4 + 4,
        "dq_nvfp4_1x16 row->bf16": E // 2 + E // 16 + 4 + 2 * E,
        "dq_nvfp4_16x16 row->bf16": E // 2 + E // 256 + 4 + 2 * E,
        "nvfp4_rht_rn colT": 2 * E * b + E // 2 + E // 16 + 4 + 4,
        "nvfp4_rht_sr colT": 2 * E * b + E // 2 + E // 16 + 4 + 4,
        # BF16: one read for both maxima, one for both copies; FP32 reads x once per copy
        "nvfp4_recipe_sr row + RHT colT": (2 if b == 2 else 3) * E * b + E + 2 * (E // 16) + 2 * (4 + 4),
    }
    if name.startswith("dq_cs row->"):
        ob = 4 if name.endswith("float32") else 2
        return E + 4 + E * ob
    return table[name]


def test_every_call_counts_its_algorithmic_bytes(bench):
    dev = {wl: {tn: torch.zeros(shape, dtype=dt) for tn, (shape, dt) in t.items()} for wl, t in SHAPES.items()}
    calls = bench.build_step(dev, torch, Q)
    assert len(calls) == 26
    seen = set()
    for c in calls:
        tag, name = c.name.split(" ", 1)
        wl, tn = tag.split(".")
        x = dev[wl][tn]
        M, K = x.shape
        assert c.alg_bytes == expected(name, M, K, x.element_size()), c.name
        seen.add(name)
    assert "nvfp4_recipe_sr row + RHT colT" in seen and "blockwise_mx_128x128 row+colT" in seen


def test_each_piece_has_a_source_file_and_positive_bytes(bench):
    dev = {wl: {tn: torch.zeros(shape, dtype=dt) for tn, (shape, dt) in t.items()} for wl, t in SHAPES.items()}
    for c in bench.build_step(dev, torch, Q):
        for kernel, src, b, _ in c.pieces:
            assert b > 0 and os.path.exists(os.path.join(ROOT, "nvfp4_quantization_current_gb300", "csrc", src)), \
                (c.name, kernel)
