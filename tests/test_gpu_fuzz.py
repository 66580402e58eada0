"""GPU parity over seeded random shapes: for every entry point, cases drawn
from a fixed seed with random sizes (multiples of each recipe's block only
where the ABI requires them, ragged tiles otherwise), input dtype,
distribution, planted zero blocks and tiny / huge magnitudes, SR seeds and
counter offsets, compared bit for bit with the CPU oracle, dequantizers
included.  Sizes stay below ~0.4M elements so the oracle keeps up."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

Q = pytest.importorskip("nvfp4_quantization_current_gb300")

KINDS = ["normal", "lognormal_rows", "t3", "grad", "weight", "outliers"]
N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    Q.lib()


def dev(x):
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(x.copy()).cuda()


def host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def same(a, b, what):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.argwhere(a != b)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:3].tolist()}"


def dim(rng, mult, lo, hi):
    """A size in [lo, hi] that is a multiple of mult."""
    return int(rng.integers(max(1, lo // mult), hi // mult + 1)) * mult


def tensor(rng, M, K):
    """A seeded input of a random kind and dtype, with a planted zero block
    and a scaled band (tiny or huge magnitudes) at random places."""
    bf16 = bool(rng.integers(0, 2))
    x = W.gen(KINDS[int(rng.integers(0, len(KINDS)))], (M, K), int(rng.integers(0, 2 ** 31)), bf16=False)
    if M >= 16 and K >= 16 and rng.integers(0, 2):
        m0, k0 = int(rng.integers(0, M - 15)), int(rng.integers(0, K - 15))
        x[m0:m0 + 16, k0:k0 + 16] = 0
    if rng.integers(0, 3) == 0:
        r0 = int(rng.integers(0, M))
        x[r0:r0 + 8] *= np.float32(10.0 ** float(rng.choice([-30, -12, 12, 30])))
    return (W.to_bf16_bits(x) if bf16 else x.astype(np.float32)), bf16


def cases(recipe):
    return [(recipe, i) for i in range(N_CASES)]


def rng_of(recipe, i):
    return np.random.default_rng(sum(map(ord, recipe)) * 1000 + i)


OUTS = [torch.float32, torch.bfloat16]


def o_out(dt):
    return O.F32 if dt == torch.float32 else O.BF16


@pytest.mark.parametrize("recipe,i", cases("cs"))
def test_fuzz_current_scaling(recipe, i):
    rng = rng_of(recipe, i)
    colwise = bool(rng.integers(0, 2))
    M = dim(rng, 16 if colwise else 1, 1, 400)
    K = dim(rng, 16 if colwise else 1, 16, 900)
    fmt = int(rng.integers(0, 2))
    x, _ = tensor(rng, M, K)
    want = O.current_scaling(x, fmt, rowwise=True, colwise=colwise)
    got = Q.q_current_scaling(dev(x), "e4m3" if fmt == O.E4M3 else "e5m2", rowwise=True, colwise=colwise)
    same(host(got.amax), np.float32(want.amax).reshape(1), "amax")
    same(host(got.scale), np.float32(want.scale).reshape(1), "scale")
    same(host(got.q_row), want.q_row, "q_row")
    if colwise:
        same(host(got.q_colT), want.q_colT, "q_colT")
    dt = OUTS[int(rng.integers(0, 2))]
    same(host(got.dequantize(Q.Q_ROW, dt)), O.dq_current_scaling(want.q_row, want.scale, fmt, o_out(dt)), "dq")


@pytest.mark.parametrize("recipe,i", cases("ds"))
def test_fuzz_delayed_scaling_cast(recipe, i):
    rng = rng_of(recipe, i)
    colwise = bool(rng.integers(0, 2))
    M = dim(rng, 16 if colwise else 1, 1, 400)
    K = dim(rng, 16 if colwise else 1, 16, 900)
    fmt = int(rng.integers(0, 2))
    x, _ = tensor(rng, M, K)
    alpha = np.float32(2.0 ** float(rng.uniform(-20, 20)))
    q_row, q_colT, a = O.ds_cast(x, alpha, fmt, rowwise=True, colwise=colwise)
    ds = torch.tensor([alpha, np.float32(1.0) / alpha], dtype=torch.float32, device="cuda")
    slot = torch.full((1,), 123.0, device="cuda")
    got = Q.q_delayed_scaling(dev(x), ds, slot, "e4m3" if fmt == O.E4M3 else "e5m2", True, colwise)
    same(host(got.q_row), q_row, "q_row")
    if colwise:
        same(host(got.q_colT), q_colT, "q_colT")
    same(host(slot), np.float32(a).reshape(1), "recorded amax")


@pytest.mark.parametrize("recipe,i", cases("mx"))
def test_fuzz_mxfp8_and_requant(recipe, i):
    rng = rng_of(recipe, i)
    M = dim(rng, 32, 32, 384)
    K = dim(rng, 32, 32, 1100)
    fmt = int(rng.integers(0, 2))
    f = "e4m3" if fmt == O.E4M3 else "e5m2"
    x, _ = tensor(rng, M, K)
    want = O.mxfp8(x, fmt)
    got = Q.q_mxfp8(dev(x), f)
    for name in ("q_row", "e8m0_row", "q_col", "e8m0_col"):
        same(host(getattr(got, name)), getattr(want, name), name)
    wq, we = O.mxfp8_requant_col(want.q_row, want.e8m0_row, fmt)
    rq = Q.q_mxfp8_requant_col(got.q_row, got.e8m0_row, f)
    same(host(rq.q_col), wq, "requant q_col")
    same(host(rq.e8m0_col), we, "requant e8m0_col")
    dt = OUTS[int(rng.integers(0, 2))]
    same(host(got.dequantize(Q.Q_COL, dt)), O.dq_mxfp8(want.q_col, want.e8m0_col, fmt, O.COL, o_out(dt)), "dq col")


@pytest.mark.parametrize("recipe,i", cases("bw"))
def test_fuzz_blockwise_both_scale_kinds(recipe, i):
    rng = rng_of(recipe, i)
    tile = int(rng.integers(0, 2))
    colwise = tile == O.T128x128 or bool(rng.integers(0, 2))
    M = dim(rng, 128 if colwise else 1, 1, 400)
    K = dim(rng, 128, 128, 1024)
    x, _ = tensor(rng, M, K)
    t = "1x128" if tile == O.T1x128 else "128x128"
    want = O.blockwise(x, tile, rowwise=True, colwise=colwise)
    got = Q.q_blockwise(dev(x), t, rowwise=True, colwise=colwise)
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.s_row), want.s_row, "s_row")
    if colwise:
        same(host(got.q_colT), want.q_colT, "q_colT")
        same(host(got.s_colT), want.s_colT, "s_colT")
    dt = OUTS[int(rng.integers(0, 2))]
    same(host(got.dequantize(Q.Q_ROW, dt)), O.dq_blockwise(want.q_row, want.s_row, tile, o_out(dt)), "dq")
    wm = O.blockwise_mx(x, tile, rowwise=True, colwise=colwise)
    gm = Q.q_blockwise_mx(dev(x), t, rowwise=True, colwise=colwise)
    same(host(gm.q_row), wm.q_row, "mx q_row")
    same(host(gm.e8m0_row), wm.e8m0_row, "mx e8m0_row")
    if colwise:
        same(host(gm.q_colT), wm.q_colT, "mx q_colT")
        same(host(gm.e8m0_colT), wm.e8m0_colT, "mx e8m0_colT")


@pytest.mark.parametrize("recipe,i", cases("nv"))
def test_fuzz_nvfp4(recipe, i):
    rng = rng_of(recipe, i)
    blk = int(rng.integers(0, 2))
    rnd = int(rng.integers(0, 2))
    M = dim(rng, 16, 16, 400)
    K = dim(rng, 16, 16, 900)
    seed, offset = int(rng.integers(0, 2 ** 62)), int(rng.integers(0, 2 ** 20))
    x, _ = tensor(rng, M, K)
    want = O.nvfp4(x, blk, rnd, seed=seed, offset=offset, rowwise=True, colwise=True)
    got = Q.q_nvfp4(dev(x), "1x16" if blk == O.B1x16 else "16x16", "rn" if rnd == O.RN else "sr", seed, offset,
                    True, True)
    same(host(got.amax), np.float32(want.amax).reshape(1), "amax")
    same(host(got.s_global), np.float32(want.s_global).reshape(1), "s_global")
    for name in ("q_row", "sb_row", "q_colT", "sb_colT"):
        same(host(getattr(got, name)), getattr(want, name), name)
    dt = OUTS[int(rng.integers(0, 2))]
    same(host(got.dequantize(Q.Q_COL, dt)), O.dq_nvfp4(want.q_colT, want.sb_colT, want.s_global, blk, o_out(dt)),
         "dq colT")


@pytest.mark.parametrize("recipe,i", cases("rht"))
def test_fuzz_rht_colT(recipe, i):
    rng = rng_of(recipe, i)
    rnd = int(rng.integers(0, 2))
    M = dim(rng, 16, 16, 400)
    K = dim(rng, 16, 16, 900)
    mask = int(rng.integers(0, 1 << 16))
    seed, offset = int(rng.integers(0, 2 ** 62)), int(rng.integers(0, 2 ** 20))
    x, _ = tensor(rng, M, K)
    q, sb, a, sg = O.nvfp4_rht_colT(x, mask, rnd, seed=seed, offset=offset)
    got = Q.q_nvfp4_rht_colT(dev(x), mask, "rn" if rnd == O.RN else "sr", seed, offset)
    same(host(got.amax), np.float32(a).reshape(1), "amax of the transform")
    same(host(got.s_global), np.float32(sg).reshape(1), "s_global")
    same(host(got.q_colT), q, "q_colT")
    same(host(got.sb_colT), sb, "sb_colT")
    # the fused recipe: the same transposed copy, plus the rowwise copy of x
    row, col = Q.q_nvfp4_recipe(dev(x), mask, "rn" if rnd == O.RN else "sr", seed, offset)
    same(host(col.q_colT), q, "recipe q_colT")
    same(host(col.sb_colT), sb, "recipe sb_colT")
    w = O.nvfp4(x, O.B1x16, rnd, seed=seed, offset=offset, rowwise=True, colwise=False)
    same(host(row.q_row), w.q_row, "recipe q_row")
    same(host(row.sb_row), w.sb_row, "recipe sb_row")
    same(host(row.s_global), np.float32(w.s_global).reshape(1), "recipe s_global_row")
