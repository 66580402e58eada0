"""GPU parity: every recipe through the C ABI against the CPU oracle on the
same seeded inputs, element by element, 0 ULP (codes and scale bytes
bit-identical; FP32 / BF16 values bit-identical).

Sizes span several 128 x 256 CTA tiles with ragged tails in both
dimensions; edge cases: the pages' worked example, empty tensors, zero
tensors and zero blocks, FP32 inputs, tiny values (subnormal scaled
values), non-zero SR offsets.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

Q = pytest.importorskip("nvfp4_quantization_current_gb300")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    Q.lib()


def dev(x):
    """numpy BF16 bits (uint16) or FP32 -> CUDA tensor of the same values."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(x.copy()).cuda()


def host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def same(a, b, what=""):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.argwhere(a != b)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: gpu {a[tuple(bad[0])]} oracle {b[tuple(bad[0])]}"


def f32eq(a, b, what=""):
    assert np.float32(a).view(np.uint32) == np.float32(b).view(np.uint32), (what, a, b)


OUTS = [torch.float32, torch.bfloat16]


def o_out(dtype):
    return O.F32 if dtype == torch.float32 else O.BF16


# ---------------------------------------------------------------------------
# amax + current scaling
# ---------------------------------------------------------------------------

CS_CASES = [
    # (kind, shape, bf16, fmt, colwise)
    ("outliers", (1024, 1024), False, O.E4M3, True),      # the small FP32 workload
    ("outliers", (272, 528), True, O.E4M3, True),         # ragged in both tile dimensions
    ("grad", (384, 640), True, O.E5M2, True),
    ("weight", (256, 256), True, O.E4M3, False),
    ("normal", (1000, 784), True, O.E4M3, False),         # rowwise only: any shape
    ("t3", (37, 61), False, O.E5M2, False),               # odd sizes: vector tail + scalar tail
    ("normal", (16, 16), False, O.E4M3, True),
]


@pytest.mark.parametrize("kind,shape,bf16,fmt,colwise", CS_CASES)
def test_current_scaling_parity(kind, shape, bf16, fmt, colwise):
    x = W.gen(kind, shape, 101, bf16=bf16)
    want = O.current_scaling(x, fmt, rowwise=True, colwise=colwise)
    got = Q.q_current_scaling(dev(x), "e4m3" if fmt == O.E4M3 else "e5m2", rowwise=True, colwise=colwise)
    torch.cuda.synchronize()
    f32eq(got.amax.item(), want.amax, "amax")
    f32eq(got.scale.item(), want.scale, "scale")
    same(host(got.q_row), want.q_row, "q_row")
    if colwise:
        same(host(got.q_colT), want.q_colT, "q_colT")
    for dt in OUTS:
        y = got.dequantize(Q.Q_ROW, dt)
        same(host(y), O.dq_current_scaling(want.q_row, want.scale, fmt, o_out(dt)), f"dq {dt}")


def test_current_scaling_worked_example():
    x = W.EXAMPLE_X
    want = O.current_scaling(x)
    got = Q.q_current_scaling(dev(x))
    same(host(got.q_row), want.q_row)
    f32eq(got.scale.item(), want.scale)
    y = host(got.dequantize())
    same(y, O.dq_current_scaling(want.q_row, want.scale))
    assert host(got.q_row).tolist() == [[0xFE, 0x63, 0x7E]]     # -448, 44, 448


def test_amax_alone_and_given_amax_sharding():
    x = W.gen("outliers", (512, 384), 7, bf16=True)
    a = Q.q_amax(dev(x))
    f32eq(a.item(), O.amax(x))
    # two row shards quantized with the MAX of their local amaxes equal the whole tensor
    xs = [x[:128], x[128:]]
    loc = [Q.q_amax(dev(s)) for s in xs]
    g = torch.maximum(loc[0], loc[1])
    parts = [Q.q_current_scaling(dev(s), colwise=True, amax=g.clone()) for s in xs]
    whole = Q.q_current_scaling(dev(x), colwise=True)
    same(np.concatenate([host(p.q_row) for p in parts]), host(whole.q_row))
    same(np.concatenate([host(p.q_colT) for p in parts], axis=1), host(whole.q_colT))


def test_current_scaling_zero_and_empty():
    z = np.zeros((64, 64), np.uint16)
    got = Q.q_current_scaling(dev(z), colwise=True)
    assert got.amax.item() == 0 and got.scale.item() == 1
    assert not host(got.q_row).any() and not host(got.q_colT).any()
    e = torch.empty((0, 16), dtype=torch.bfloat16, device="cuda")
    got = Q.q_current_scaling(e)
    assert got.amax.item() == 0 and got.scale.item() == 1
    assert Q.q_amax(torch.empty((0,), dtype=torch.float32, device="cuda").view(0, 1)).item() == 0


def test_tiny_values_scale_to_fp32_subnormals():
    x = (W.gen("normal", (64, 64), 3, bf16=False) * np.float32(1e-38)).astype(np.float32)
    x[0, 0] = np.float32(1e-30)
    want = O.current_scaling(x, O.E4M3, colwise=True)
    got = Q.q_current_scaling(dev(x), colwise=True)
    same(host(got.q_row), want.q_row)
    same(host(got.q_colT), want.q_colT)
    f32eq(got.scale.item(), want.scale)


def test_bounded_wait_times_out_and_context_stays_usable():
    """A wait on a barrier that nothing completes gives up after its limit,
    reports Q_ST_TIMEOUT, and the next calls work normally."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    Q.selftest_wait_timeout(st, 50_000_000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 >= 0.045
    assert st.item() & Q.Q_ST_TIMEOUT
    x = W.gen("outliers", (64, 48), 5, bf16=True)
    got = Q.q_current_scaling(dev(x), "e4m3", colwise=True)
    want = O.current_scaling(x, O.E4M3, colwise=True)
    same(host(got.q_row), want.q_row)
    same(host(got.q_colT), want.q_colT)


def test_nonfinite_sets_status():
    x = W.gen("normal", (32, 32), 3, bf16=False)
    x[3, 4] = np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.q_current_scaling(dev(x), status=st)
    assert st.item() & Q.Q_ST_NONFINITE
    st.zero_()
    Q.q_mxfp8(dev(x), status=st)
    assert st.item() & Q.Q_ST_NONFINITE
    st.zero_()
    Q.q_nvfp4(dev(x), status=st)
    assert st.item() & Q.Q_ST_NONFINITE
    st.zero_()
    Q.q_current_scaling(dev(W.gen("normal", (32, 32), 3, bf16=False)), status=st)
    assert st.item() == 0


# ---------------------------------------------------------------------------
# random Hadamard transform + columnwise NVFP4 (weight-gradient inputs)
# ---------------------------------------------------------------------------

RHT_CASES = [
    ("outliers", (256, 512), True, O.RN, 0xA5C3),
    ("grad", (96, 800), True, O.SR, 0x0F0F),       # 96 rows < one tile; 800 = 3 x 256 + 32 columns
    ("normal", (64, 416), False, O.RN, 0xFFFF),    # FP32: 128-column tiles
    ("outliers", (384, 144), False, O.SR, 0x1234),  # FP32, 3 tile rows, ragged columns
    ("lognormal_rows", (16, 16), True, O.RN, 0x0000),
]


@pytest.mark.parametrize("kind,shape,bf16,rnd,mask", RHT_CASES)
def test_nvfp4_rht_colT_parity(kind, shape, bf16, rnd, mask):
    x = W.gen(kind, shape, 515, bf16=bf16)
    q, sb, a, sg = O.nvfp4_rht_colT(x, mask, rnd, seed=21, offset=5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = Q.q_nvfp4_rht_colT(dev(x), mask, "rn" if rnd == O.RN else "sr", seed=21, offset=5, status=st)
    torch.cuda.synchronize()
    f32eq(got.amax.item(), a, "amax of the transform")
    f32eq(Q.q_nvfp4_rht_amax(dev(x), mask).item(), a, "q_nvfp4_rht_amax")
    f32eq(got.s_global.item(), sg, "s_global")
    same(host(got.q_colT), q, "q_colT")
    same(host(got.sb_colT), sb, "sb_colT")
    assert st.item() == 0
    # a given amax (the sharded case) sets the tensor scale
    A = torch.tensor([np.float32(a) * 4], device="cuda")
    q2, sb2, _, sg2 = O.nvfp4_rht_colT(x, mask, rnd, seed=21, offset=5, amax_in=np.float32(a) * 4)
    got2 = Q.q_nvfp4_rht_colT(dev(x), mask, "rn" if rnd == O.RN else "sr", seed=21, offset=5, amax=A)
    same(host(got2.q_colT), q2, "q_colT, given amax")
    same(host(got2.sb_colT), sb2, "sb_colT, given amax")
    f32eq(got2.s_global.item(), sg2, "s_global, given amax")


RECIPE_CASES = [
    ("t3", (256, 512), True, O.SR, 0xB4E1, 9, 3),
    ("outliers", (272, 528), True, O.RN, 0x5A5A, 0, 0),      # ragged tiles both ways
    ("normal", (96, 160), False, O.SR, 0x0F0F, 77, 1000),    # FP32 input
    ("lognormal_rows", (16, 16), True, O.RN, 0xFFFF, 0, 0),
]


@pytest.mark.parametrize("kind,shape,bf16,rnd,mask,seed,offset", RECIPE_CASES)
def test_nvfp4_recipe_equals_its_two_calls(kind, shape, bf16, rnd, mask, seed, offset):
    """The fused recipe (one amax pass for max|x| and max|x'|, the rowwise
    copy of x, the columnwise copy of x') gives what q_nvfp4 (rowwise) and
    q_nvfp4_rht_colT give, both checked against the oracle."""
    x = W.gen(kind, shape, 616, bf16=bf16)
    x[:16, :16] = 0
    r = "rn" if rnd == O.RN else "sr"
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    row, col = Q.q_nvfp4_recipe(dev(x), mask, r, seed, offset, status=st)
    torch.cuda.synchronize()
    w = O.nvfp4(x, O.B1x16, rnd, seed=seed, offset=offset, rowwise=True, colwise=False)
    f32eq(row.amax.item(), w.amax, "amax_row")
    f32eq(row.s_global.item(), w.s_global, "s_global_row")
    same(host(row.q_row), w.q_row, "q_row")
    same(host(row.sb_row), w.sb_row, "sb_row")
    q, sb, a, sg = O.nvfp4_rht_colT(x, mask, rnd, seed=seed, offset=offset)
    f32eq(col.amax.item(), a, "amax_colT")
    f32eq(col.s_global.item(), sg, "s_global_colT")
    same(host(col.q_colT), q, "q_colT")
    same(host(col.sb_colT), sb, "sb_colT")
    assert st.item() == 0
    a_rht, a_x = Q.q_nvfp4_rht_amax2(dev(x), mask)
    f32eq(a_rht.item(), a, "amax2 rht")
    f32eq(a_x.item(), O.amax(x), "amax2 x")
    # the same casts with both maxima given (the path a sharded caller takes)
    ar = torch.tensor([w.amax], dtype=torch.float32, device="cuda")
    ac = torch.tensor([a], dtype=torch.float32, device="cuda")
    row2, col2 = Q.q_nvfp4_recipe(dev(x), mask, r, seed, offset, amax_row=ar, amax_col=ac, status=st)
    torch.cuda.synchronize()
    f32eq(ar.item(), w.amax, "given amax_row untouched")
    f32eq(ac.item(), a, "given amax_colT untouched")
    f32eq(row2.s_global.item(), w.s_global, "s_global_row, given")
    f32eq(col2.s_global.item(), sg, "s_global_colT, given")
    same(host(row2.q_row), w.q_row, "q_row, given")
    same(host(row2.sb_row), w.sb_row, "sb_row, given")
    same(host(col2.q_colT), q, "q_colT, given")
    same(host(col2.sb_colT), sb, "sb_colT, given")
    assert st.item() == 0


def test_nvfp4_recipe_empty_and_nonfinite():
    row, col = Q.q_nvfp4_recipe(torch.empty((0, 32), dtype=torch.bfloat16, device="cuda"), 0x1234)
    assert row.amax.item() == 0 and col.amax.item() == 0
    assert row.s_global.item() == 1 and col.s_global.item() == 1
    x = W.gen("normal", (32, 48), 3, bf16=False)
    x[5, 7] = np.nan
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a_rht, a_x = Q.q_nvfp4_rht_amax2(dev(x), 0x1234, status=st)
    assert st.item() & Q.Q_ST_NONFINITE
    # non-finite inputs are outside the amax contract: a NaN, and the same word q_amax gives
    assert np.isnan(a_x.item())
    f32eq(a_x.item(), Q.q_amax(dev(x)).item(), "amax2 x vs q_amax")


def test_nvfp4_rht_colT_row_shards_with_the_global_amax():
    """Row shards on 16-row boundaries, each encoded with the maximum of the
    shards' transform amaxes, concatenate to the unsharded copy (RTNE)."""
    x = W.gen("outliers", (256, 512), 77, bf16=True)
    xd = dev(x)
    mask = 0x6B1D
    cuts = [0, 64, 80, 256]
    amaxes = [Q.q_nvfp4_rht_amax(xd[a:b].contiguous(), mask) for a, b in zip(cuts, cuts[1:])]
    A = torch.stack(amaxes).max().reshape(1)
    parts = [Q.q_nvfp4_rht_colT(xd[a:b].contiguous(), mask, "rn", amax=A) for a, b in zip(cuts, cuts[1:])]
    whole = Q.q_nvfp4_rht_colT(xd, mask, "rn")
    f32eq(A.item(), whole.amax.item(), "global amax")
    same(np.concatenate([host(p.q_colT) for p in parts], axis=1), host(whole.q_colT), "q_colT")
    same(np.concatenate([host(p.sb_colT) for p in parts], axis=1), host(whole.sb_colT), "sb_colT")


def test_nvfp4_rht_colT_empty_and_nonfinite():
    e = Q.q_nvfp4_rht_colT(torch.empty((0, 32), dtype=torch.bfloat16, device="cuda"), 0x1)
    assert e.amax.item() == 0.0 and e.s_global.item() == 1.0
    x = W.gen("normal", (32, 32), 3, bf16=False)
    x[5, 6] = np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.q_nvfp4_rht_colT(dev(x), 0x1, status=st)
    assert st.item() & Q.Q_ST_NONFINITE


# ---------------------------------------------------------------------------
# per-tensor delayed scaling
# ---------------------------------------------------------------------------

DS_CASES = [
    ((256, 512), True, O.E4M3, True, "max", 4),        # tiled row + colT, 2 x 2 tiles
    ((96, 800), True, O.E5M2, True, "max", 3),         # ragged tiles
    ((64, 416), False, O.E4M3, True, "most_recent", 2),  # FP32 input
    ((100, 300), True, O.E4M3, False, "max", 4),       # rowwise only: flat path with a ragged tail (30000 % 16 = 0)
    ((37, 53), False, O.E5M2, False, "max", 5),        # flat path, 1961 elements (tail of 9)
]


@pytest.mark.parametrize("shape,bf16,fmt,colwise,algo,N", DS_CASES)
def test_delayed_scaling_steps_parity(shape, bf16, fmt, colwise, algo, N):
    """Seven steps with tensors of changing range (an outlier step that must
    leave the window after N steps): codes, s, the recorded amax and the
    next [alpha, s] all bit-identical to the oracle's run."""
    f = "e4m3" if fmt == O.E4M3 else "e5m2"
    oalgo = O.HIST_MAX if algo == "max" else O.HIST_MOST_RECENT
    state = Q.DelayedScaling(f, history_len=N, algo=algo)
    hist = np.zeros(N, np.float32)
    alpha, s = np.float32(1.0), np.float32(1.0)
    for t, scale in enumerate([1.0, 300.0, 0.5, 2.0, 1e-3, 7.0, 1.0]):
        x = W.gen("outliers", shape, 400 + t, bf16=False) * np.float32(scale)
        x = O.bf16_round(x.astype(np.float32)) if bf16 else x.astype(np.float32)
        q_row, q_colT, a = O.ds_cast(x, alpha, fmt, rowwise=True, colwise=colwise)
        got = state.quantize(dev(x), rowwise=True, colwise=colwise)
        torch.cuda.synchronize()
        same(host(got.q_row), q_row, f"step {t} q_row")
        if colwise:
            same(host(got.q_colT), q_colT, f"step {t} q_colT")
        f32eq(got.scale.item(), s, f"step {t} scale")
        f32eq(got.amax.item(), a, f"step {t} amax")
        hist[t % N] = a
        alpha, s = O.ds_scale_update(hist, t % N, oalgo, fmt)
        d = host(state.ds)
        f32eq(d[0], alpha, f"step {t} next alpha")
        f32eq(d[1], s, f"step {t} next s")
    same(host(state.hist), hist, "window")


@pytest.mark.parametrize("N", [1, 255, 1024, 1500])
def test_delayed_scale_update_parity(N):
    rng = np.random.default_rng(N)
    h = (rng.lognormal(0, 6, N) * (rng.random(N) < 0.9)).astype(np.float32)   # zeros among them
    hd = dev(h)
    ds = torch.empty(2, dtype=torch.float32, device="cuda")
    for fmt in (O.E4M3, O.E5M2):
        for algo in (O.HIST_MAX, O.HIST_MOST_RECENT):
            pos = int(rng.integers(0, N))
            Q.q_delayed_scale_update(hd, pos, ds, "e4m3" if fmt == O.E4M3 else "e5m2", algo)
            al, s = O.ds_scale_update(h, pos, algo, fmt)
            d = host(ds)
            f32eq(d[0], al, (N, fmt, algo))
            f32eq(d[1], s, (N, fmt, algo))
    h[N // 2] = 1e-45                                      # most recent: alpha overflows -> FLT_MAX
    Q.q_delayed_scale_update(dev(h), N // 2, ds, "e4m3", "most_recent")
    assert host(ds)[0] == np.finfo(np.float32).max
    h[N // 3] = np.nan                                     # a NaN entry wins the max
    Q.q_delayed_scale_update(dev(h), 0, ds, "e4m3", "max")
    assert np.isnan(host(ds)[0])


def test_delayed_scaling_empty_and_nonfinite():
    ds = torch.tensor([2.0, 0.5], device="cuda")
    a = torch.full((1,), 7.0, device="cuda")
    got = Q.q_delayed_scaling(torch.empty((0, 16), dtype=torch.bfloat16, device="cuda"), ds, a)
    assert got.amax.item() == 0.0 and got.scale.item() == 0.5
    x = W.gen("normal", (32, 48), 3, bf16=False)
    x[7, 9] = np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.q_delayed_scaling(dev(x), ds, a, colwise=True, status=st)
    assert st.item() & Q.Q_ST_NONFINITE and a.item() == np.inf
    st.zero_()
    Q.q_delayed_scaling(dev(W.gen("normal", (32, 48), 3, bf16=False)), ds, a, status=st)
    assert st.item() == 0


# ---------------------------------------------------------------------------
# MXFP8
# ---------------------------------------------------------------------------

MX_CASES = [
    ("lognormal_rows", (256, 512), True, O.E4M3),
    ("lognormal_rows", (96, 800), True, O.E4M3),     # ragged: 800 = 3 * 256 + 32
    ("t3", (160, 288), True, O.E5M2),
    ("normal", (64, 416), False, O.E4M3),             # FP32 input, 128-column CTA tiles
    ("grad", (32, 32), True, O.E5M2),
    ("normal", (96, 256), True, O.E4M3),              # dequant: a thread's 4 rows fill a 32-row block exactly
    ("t3", (128, 128), True, O.E4M3),                 # dequant: a thread's rows span 32-row blocks
]


@pytest.mark.parametrize("kind,shape,bf16,fmt", MX_CASES)
def test_mxfp8_parity(kind, shape, bf16, fmt):
    x = W.gen(kind, shape, 202, bf16=bf16)
    x_t = x.copy()
    if bf16:
        x_t[:, :32] = 0          # an all-zero row block in every row and a zero column block
    want = O.mxfp8(x_t, fmt)
    got = Q.q_mxfp8(dev(x_t), "e4m3" if fmt == O.E4M3 else "e5m2")
    torch.cuda.synchronize()
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.e8m0_row), want.e8m0_row, "e8m0_row")
    same(host(got.q_col), want.q_col, "q_col")
    same(host(got.e8m0_col), want.e8m0_col, "e8m0_col")
    for dt in OUTS:
        same(host(got.dequantize(Q.Q_ROW, dt)), O.dq_mxfp8(want.q_row, want.e8m0_row, fmt, O.ROW, o_out(dt)), "dq row")
        same(host(got.dequantize(Q.Q_COL, dt)), O.dq_mxfp8(want.q_col, want.e8m0_col, fmt, O.COL, o_out(dt)), "dq col")


def test_mxfp8_rowwise_only_ragged_rows():
    x = W.gen("lognormal_rows", (100, 288), 5, bf16=True)
    want = O.mxfp8(x, O.E4M3, rowwise=True, colwise=False)
    got = Q.q_mxfp8(dev(x), colwise=False)
    same(host(got.q_row), want.q_row)
    same(host(got.e8m0_row), want.e8m0_row)


def test_mxfp8_extreme_exponents():
    """Block maxima at FP32 subnormal / huge magnitudes exercise the clamps
    of the E8M0 code and the 2^-127 factor."""
    x = W.gen("normal", (64, 64), 6, bf16=False)
    x[:32, :32] *= np.float32(1e-42)          # subnormal inputs
    x[32:, 32:] *= np.float32(1e36)
    x = x.astype(np.float32)
    want = O.mxfp8(x, O.E4M3)
    got = Q.q_mxfp8(dev(x))
    same(host(got.q_row), want.q_row)
    same(host(got.e8m0_row), want.e8m0_row)
    same(host(got.q_col), want.q_col)
    same(host(got.e8m0_col), want.e8m0_col)
    same(host(got.dequantize(Q.Q_ROW)), O.dq_mxfp8(want.q_row, want.e8m0_row, O.E4M3, O.ROW, O.F32))


RQ_CASES = [
    ("lognormal_rows", (256, 512), True, O.E4M3),
    ("lognormal_rows", (96, 800), True, O.E4M3),      # 96 rows < one 128-row tile; 800 = 512 + 288 columns
    ("t3", (160, 288), True, O.E5M2),
    ("outliers", (384, 1056), False, O.E4M3),          # FP32 input, 3 x 3 tiles with ragged tails
    ("grad", (32, 32), True, O.E5M2),
]


@pytest.mark.parametrize("kind,shape,bf16,fmt", RQ_CASES)
def test_mxfp8_requant_col_parity(kind, shape, bf16, fmt):
    """Rowwise MXFP8 output -> columnwise codes: GPU requant vs the oracle's
    dequantize + re-quantize, bit for bit."""
    x = W.gen(kind, shape, 303, bf16=bf16)
    x[:32, :64] = 0                                   # zero blocks in both directions
    f = "e4m3" if fmt == O.E4M3 else "e5m2"
    rw = O.mxfp8(x, fmt, rowwise=True, colwise=False)
    want_q, want_e = O.mxfp8_requant_col(rw.q_row, rw.e8m0_row, fmt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = Q.q_mxfp8_requant_col(dev(rw.q_row), dev(rw.e8m0_row), f, status=st)
    torch.cuda.synchronize()
    same(host(got.q_col), want_q, "q_col")
    same(host(got.e8m0_col), want_e, "e8m0_col")
    assert st.item() == 0
    # the chain through the library's own rowwise quantizer gives the same result
    gr = Q.q_mxfp8(dev(x), f, colwise=False)
    got2 = Q.q_mxfp8_requant_col(gr.q_row, gr.e8m0_row, f)
    same(host(got2.q_col), want_q, "q_col via q_mxfp8")


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_mxfp8_requant_col_random_codes(fmt):
    """Every finite code with block scales over the whole range that does not
    overflow FP32 on dequantization (x_hat down to 2^-143, FP32 subnormal)."""
    rng = np.random.default_rng(7)
    M, K = 224, 640
    q = rng.integers(0, 256, (M, K), dtype=np.uint8)
    if fmt == O.E4M3:
        q[(q & 0x7F) == 0x7F] ^= 0x01                 # no NaN codes
        top = 246                                     # 448 * 2^(246-127) < FLT_MAX
    else:
        q[(q & 0x7C) == 0x7C] &= 0xFB                 # no inf / NaN codes
        top = 239
    e = rng.integers(0, top + 1, (M, K // 32), dtype=np.uint8)
    e[: M // 2, 0] = 0                                # smallest scale in whole column blocks
    e[M // 2:, 1] = top
    want_q, want_e = O.mxfp8_requant_col(q, e, fmt)
    got = Q.q_mxfp8_requant_col(dev(q), dev(e), "e4m3" if fmt == O.E4M3 else "e5m2")
    same(host(got.q_col), want_q, "q_col")
    same(host(got.e8m0_col), want_e, "e8m0_col")


def test_mxfp8_requant_col_nan_scale_and_args():
    q = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    e = torch.full((64, 2), 127, dtype=torch.uint8, device="cuda")
    e[5, 1] = 255
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.q_mxfp8_requant_col(q, e, status=st)
    torch.cuda.synchronize()
    assert st.item() & Q.Q_ST_NONFINITE
    empty = Q.q_mxfp8_requant_col(q[:0], e[:0])
    assert empty.q_col.shape == (0, 64)
    with pytest.raises(Q.QuantError):
        Q.q_mxfp8_requant_col(q[:48], e[:48])         # M % 32 != 0


# ---------------------------------------------------------------------------
# blockwise
# ---------------------------------------------------------------------------

BW_CASES = [
    ("normal", (256, 640), True, O.T1x128, True),
    ("normal", (384, 384), False, O.T1x128, True),
    ("t3", (300, 384), True, O.T1x128, False),          # ragged rows, rowwise only
    ("weight", (384, 640), True, O.T128x128, True),
    ("weight", (128, 128), False, O.T128x128, True),
]


@pytest.mark.parametrize("kind,shape,bf16,tile,colwise", BW_CASES)
def test_blockwise_parity(kind, shape, bf16, tile, colwise):
    x = W.gen(kind, shape, 303, bf16=bf16)
    if shape[0] >= 256:
        x[128:256, 128:256] = 0      # an all-zero tile
    want = O.blockwise(x, tile, rowwise=True, colwise=colwise)
    got = Q.q_blockwise(dev(x), "1x128" if tile == O.T1x128 else "128x128", rowwise=True, colwise=colwise)
    torch.cuda.synchronize()
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.s_row), want.s_row, "s_row")
    if colwise:
        same(host(got.q_colT), want.q_colT, "q_colT")
        same(host(got.s_colT), want.s_colT, "s_colT")
    for dt in OUTS:
        same(host(got.dequantize(Q.Q_ROW, dt)), O.dq_blockwise(want.q_row, want.s_row, tile, o_out(dt)), "dq row")
        if colwise:
            same(host(got.dequantize(Q.Q_COL, dt)), O.dq_blockwise(want.q_colT, want.s_colT, tile, o_out(dt)), "dq colT")


BWMX_CASES = [
    ("normal", (256, 640), True, O.T1x128, True),
    ("outliers", (384, 384), False, O.T1x128, True),     # FP32 input, 128-column CTA tiles
    ("t3", (300, 384), True, O.T1x128, False),           # ragged rows, rowwise only
    ("weight", (384, 640), True, O.T128x128, True),      # ragged last tile: one 128-column block
    ("weight", (256, 512), True, O.T128x128, True),
    ("lognormal_rows", (128, 128), False, O.T128x128, True),
]


@pytest.mark.parametrize("kind,shape,bf16,tile,colwise", BWMX_CASES)
def test_blockwise_mx_parity(kind, shape, bf16, tile, colwise):
    """Blockwise tiles with power-of-two scales held as MXFP8 E8M0 codes."""
    x = W.gen(kind, shape, 313, bf16=bf16)
    if shape[0] >= 256:
        x[128:256, 128:256] = 0      # an all-zero tile
    if not bf16:
        x[:128, :128] *= np.float32(1e-39)   # FP32 subnormal tile maxima: code clamps to 0
    want = O.blockwise_mx(x, tile, rowwise=True, colwise=colwise)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = Q.q_blockwise_mx(dev(x), "1x128" if tile == O.T1x128 else "128x128", rowwise=True, colwise=colwise,
                           status=st)
    torch.cuda.synchronize()
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.e8m0_row), want.e8m0_row, "e8m0_row")
    if colwise:
        same(host(got.q_colT), want.q_colT, "q_colT")
        same(host(got.e8m0_colT), want.e8m0_colT, "e8m0_colT")
    assert st.item() == 0
    for dt in OUTS:
        same(host(got.dequantize(Q.Q_ROW, dt)), O.dq_mxfp8(want.q_row, want.e8m0_row, O.E4M3, O.ROW, o_out(dt)), "dq row")
        if colwise:
            same(host(got.dequantize(Q.Q_COL, dt)), O.dq_mxfp8(want.q_colT, want.e8m0_colT, O.E4M3, O.ROW, o_out(dt)),
                 "dq colT")


def test_blockwise_mx_nonfinite_and_empty():
    x = W.gen("normal", (128, 256), 5, bf16=False)
    x[3, 200] = np.inf
    x[70, 10] = np.nan
    want = O.blockwise_mx(x, O.T1x128, rowwise=True, colwise=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = Q.q_blockwise_mx(dev(x), "1x128", rowwise=True, colwise=True, status=st)
    torch.cuda.synchronize()
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.e8m0_row), want.e8m0_row, "e8m0_row")
    same(host(got.q_colT), want.q_colT, "q_colT")
    same(host(got.e8m0_colT), want.e8m0_colT, "e8m0_colT")
    assert st.item() & Q.Q_ST_NONFINITE
    empty = Q.q_blockwise_mx(torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"))
    assert empty.q_row.shape == (0, 128)


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------

NV_CASES = [
    # kind, shape, bf16, blk, rnd, seed, offset
    ("normal", (256, 512), True, O.B1x16, O.RN, 0, 0),
    ("normal", (272, 528), True, O.B1x16, O.RN, 0, 0),      # ragged both ways
    ("t3", (272, 528), True, O.B1x16, O.SR, 4, 0),
    ("t3", (128, 256), True, O.B1x16, O.SR, 0xDEADBEEFCAFE, 12345),
    ("normal", (48, 160), False, O.B1x16, O.RN, 0, 0),      # FP32 input
    ("t3", (48, 160), False, O.B1x16, O.SR, 9, 3),
    ("weight", (256, 512), True, O.B16x16, O.RN, 0, 0),
    ("weight", (144, 272), True, O.B16x16, O.RN, 0, 0),
    ("weight", (144, 272), True, O.B16x16, O.SR, 77, 5),
    ("weight", (64, 96), False, O.B16x16, O.RN, 0, 0),
    ("t3", (96, 160), False, O.B16x16, O.SR, 21, 7),        # FP32 16x16 SR: four-element words
]


@pytest.mark.parametrize("kind,shape,bf16,blk,rnd,seed,offset", NV_CASES)
def test_nvfp4_parity(kind, shape, bf16, blk, rnd, seed, offset):
    x = W.gen(kind, shape, 404, bf16=bf16)
    x[:16, :16] = 0                                   # an all-zero block
    want = O.nvfp4(x, blk, rnd, seed=seed, offset=offset, rowwise=True, colwise=True)
    got = Q.q_nvfp4(dev(x), "1x16" if blk == O.B1x16 else "16x16", "rn" if rnd == O.RN else "sr",
                    seed=seed, offset=offset, rowwise=True, colwise=True)
    torch.cuda.synchronize()
    f32eq(got.amax.item(), want.amax, "amax")
    f32eq(got.s_global.item(), want.s_global, "s_global")
    same(host(got.sb_row), want.sb_row, "sb_row")
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.sb_colT), want.sb_colT, "sb_colT")
    same(host(got.q_colT), want.q_colT, "q_colT")
    for dt in OUTS:
        same(host(got.dequantize(Q.Q_ROW, dt)), O.dq_nvfp4(want.q_row, want.sb_row, want.s_global, blk, o_out(dt)), "dq row")
        same(host(got.dequantize(Q.Q_COL, dt)), O.dq_nvfp4(want.q_colT, want.sb_colT, want.s_global, blk, o_out(dt)), "dq colT")


@pytest.mark.parametrize("blk", [O.B1x16, O.B16x16])
def test_dq_nvfp4_into_outputs_off_a_32_byte_boundary(blk):
    """The dequantizer writes 32 bytes per store only into 32-byte aligned
    outputs; an output 16 bytes past such a boundary (what the C ABI still
    accepts) takes 16-byte stores and must hold the same values."""
    x = W.gen("normal", (96, 160), 405, bf16=True)
    want = O.nvfp4(x, blk, O.RN, rowwise=True, colwise=False)
    b = "1x16" if blk == O.B1x16 else "16x16"
    got = Q.q_nvfp4(dev(x), b, "rn", rowwise=True, colwise=False)
    for dt in OUTS:
        esz = torch.empty((), dtype=dt).element_size()
        buf = torch.empty(96 * 160 + 64 // esz, dtype=dt, device="cuda")
        base = buf.data_ptr() % 32
        shift = ((16 - base) % 32) // esz   # elements to a 16 (mod 32) address
        y = buf[shift:shift + 96 * 160].view(96, 160)
        assert y.data_ptr() % 32 == 16
        Q.dq_nvfp4(got.q_row, got.sb_row, got.s_global, b, dt, out=y)
        same(host(y), O.dq_nvfp4(want.q_row, want.sb_row, want.s_global, blk, o_out(dt)), f"dq {dt}")


def test_nvfp4_sr_unbiased_on_the_gpu_over_1e7_draws():
    """Stochastic rounding through the GPU path is unbiased: E[dq(q(x))] = x
    within 1e-3 relative over ~10^7 draws, in both copies.  x tiles a 16x16
    BF16 pattern P whose first row and first column hold the tensor's amax
    A = 1, so every 1x16 and 16x1 block has maximum A, its scale code is 448
    exactly (amax * alpha_g / 6 = 2688 / 6) and enc = 6: y = 6x is exact, never
    above 6, and each entry of P is drawn 40960 times per copy."""
    rng = np.random.default_rng(11)
    P = rng.uniform(-1, 1, (16, 16)).astype(np.float32)
    P = (P.view(np.uint32) & 0xFFFF0000).view(np.float32)   # BF16-exact
    P[0, :] = 1.0
    P[:, 0] = 1.0
    M, K = 4096, 2560
    x = (np.tile(P, (M // 16, K // 16)).view(np.uint32) >> 16).astype(np.uint16)   # BF16 bits
    got = Q.q_nvfp4(dev(x), "1x16", "sr", seed=2024, offset=7, rowwise=True, colwise=True)
    assert got.amax.item() == 1.0
    assert np.all(host(got.sb_row) == 0x7E) and np.all(host(got.sb_colT) == 0x7E)   # E4M3 448
    means = {
        "row": host(got.dequantize(Q.Q_ROW)).astype(np.float64),
        "col": host(got.dequantize(Q.Q_COL)).astype(np.float64).T,
    }
    y = 6.0 * np.abs(P.astype(np.float64))
    ulp = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
    frac = (y - np.floor(y / ulp) * ulp) / ulp
    n = (M // 16) * (K // 16)
    sigma = ulp / 6 * np.sqrt(frac * (1 - frac) / n)
    for name, d in means.items():
        mean = d.reshape(M // 16, 16, K // 16, 16).mean(axis=(0, 2))
        agg = abs((mean - P).sum()) / np.abs(P).sum()
        assert agg < 1e-3, (name, agg)
        assert np.all(np.abs(mean - P) <= 5 * sigma + 1e-6), name


def _f32_same_or_both_nan(a, b, what):
    a, b = np.float32(a), np.float32(b)
    if np.isnan(a) or np.isnan(b):
        assert np.isnan(a) and np.isnan(b), (what, a, b)
    else:
        f32eq(a, b, what)


@pytest.mark.parametrize("blk", [O.B1x16, O.B16x16])
@pytest.mark.parametrize("rnd", [O.RN, O.SR])
@pytest.mark.parametrize("case", ["inf", "nan", "given_amax_below_block_max"])
def test_nvfp4_bf16_nonfinite_and_overflowing_scales_match_the_oracle(case, rnd, blk):
    """BF16 inputs whose tensor amax is inf or NaN (the FP32 tensor scale is
    then 0 or NaN), and a caller-given amax far below a block's maximum (the
    block scale's product overflows FP32): every code and scale byte still
    follows the oracle's IEEE rules, and Q_ST_NONFINITE is reported."""
    x = W.gen("normal", (64, 96), 808, bf16=True)
    xf = W.bf16_bits_to_f32(x)
    big = np.float32(3.0e38)
    xf[5, 7] = big                                   # huge finite values in other blocks
    xf[40, 70] = -big
    amax_in = None
    if case == "inf":
        xf[20, 33] = np.inf
    elif case == "nan":
        xf[20, 33] = np.nan
    else:
        amax_in = 1.0e-30                            # b * alpha_g overflows for every block
    x = O.bf16_round(xf)
    want = O.nvfp4(x, blk, rnd, seed=3, offset=11, rowwise=True, colwise=True, amax_in=amax_in)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = None if amax_in is None else torch.tensor([amax_in], dtype=torch.float32, device="cuda")
    got = Q.q_nvfp4(dev(x), "1x16" if blk == O.B1x16 else "16x16", "rn" if rnd == O.RN else "sr", seed=3,
                    offset=11, rowwise=True, colwise=True, amax=a, status=st)
    torch.cuda.synchronize()
    _f32_same_or_both_nan(got.amax.item(), want.amax, "amax")
    _f32_same_or_both_nan(got.s_global.item(), want.s_global, "s_global")
    same(host(got.sb_row), want.sb_row, "sb_row")
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.sb_colT), want.sb_colT, "sb_colT")
    same(host(got.q_colT), want.q_colT, "q_colT")
    if case != "given_amax_below_block_max":
        assert st.item() & Q.Q_ST_NONFINITE


@pytest.mark.parametrize("rnd", [O.RN, O.SR])
@pytest.mark.parametrize("case", ["inf", "nan", "given_maxima_below_block_max"])
def test_nvfp4_recipe_bf16_nonfinite_and_overflowing_scales_match_the_oracle(case, rnd):
    """The one-pass recipe kernel on BF16 inputs with an inf or NaN element
    (the transform spreads it over its 16-row group; the tensor scales become
    0 or NaN) and with caller-given maxima far below the blocks' maxima: both
    copies follow the oracle's IEEE rules byte for byte."""
    x = W.gen("normal", (64, 96), 809, bf16=True)
    xf = W.bf16_bits_to_f32(x)
    big = np.float32(3.0e38)
    xf[5, 7] = big
    xf[40, 70] = -big
    given = None
    if case == "inf":
        xf[20, 33] = np.inf
    elif case == "nan":
        xf[20, 33] = np.nan
    else:
        given = 1.0e-30
    x = O.bf16_round(xf)
    mask, r = 0x5A3C, "rn" if rnd == O.RN else "sr"
    w = O.nvfp4(x, O.B1x16, rnd, seed=3, offset=11, rowwise=True, colwise=False, amax_in=given)
    q, sb, a, sg = O.nvfp4_rht_colT(x, mask, rnd, seed=3, offset=11, amax_in=given)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = {}
    if given is not None:
        kw = dict(amax_row=torch.tensor([given], dtype=torch.float32, device="cuda"),
                  amax_col=torch.tensor([given], dtype=torch.float32, device="cuda"))
    row, col = Q.q_nvfp4_recipe(dev(x), mask, r, 3, 11, status=st, **kw)
    torch.cuda.synchronize()
    _f32_same_or_both_nan(row.amax.item(), w.amax, "amax_row")
    _f32_same_or_both_nan(row.s_global.item(), w.s_global, "s_global_row")
    _f32_same_or_both_nan(col.amax.item(), a, "amax_colT")
    _f32_same_or_both_nan(col.s_global.item(), sg, "s_global_colT")
    same(host(row.sb_row), w.sb_row, "sb_row")
    same(host(row.q_row), w.q_row, "q_row")
    same(host(col.sb_colT), sb, "sb_colT")
    same(host(col.q_colT), q, "q_colT")
    if given is None:
        assert st.item() & Q.Q_ST_NONFINITE


@pytest.mark.parametrize("bf16", [True, False])
def test_nvfp4_encode_factor_case_through_the_kernel(bf16):
    """The hand-derived case of the oracle pin (A = 39, block maximum 19.625
    -> block scale 224, x = 0.8125 -> fl(x * fl(alpha_g / 224)) = 0.25, a tie
    that rounds to 0): the kernels' block scale table (BF16) and two-operation
    path (FP32) give block code 0x76 and element codes 0x7, 0x0."""
    x = np.zeros((16, 32), np.float32)
    x[0, 0], x[0, 1], x[0, 16] = 19.625, 0.8125, 39.0
    if bf16:
        x = O.bf16_round(x)
    got = Q.q_nvfp4(dev(x), rowwise=True, colwise=True)
    want = O.nvfp4(x, O.B1x16, O.RN, rowwise=True, colwise=True)
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.sb_row), want.sb_row, "sb_row")
    same(host(got.q_colT), want.q_colT, "q_colT")
    assert int(host(got.sb_row)[0, 0]) == 0x76
    assert int(host(got.q_row)[0, 0]) == 0x07   # element 0 -> 6 (low nibble), element 1 -> 0 (high nibble)


def test_nvfp4_single_direction_and_given_amax():
    x = W.gen("t3", (128, 256), 5, bf16=True)
    a = Q.q_amax(dev(x)) * 2          # a larger (e.g. all-reduced) amax
    want = O.nvfp4(x, O.B1x16, O.SR, seed=1, offset=0, rowwise=False, colwise=True, amax_in=float(a.item()))
    got = Q.q_nvfp4(dev(x), rounding="sr", seed=1, rowwise=False, colwise=True, amax=a)
    same(host(got.q_colT), want.q_colT)
    same(host(got.sb_colT), want.sb_colT)
    f32eq(got.s_global.item(), want.s_global)


@pytest.mark.parametrize("rows", [48, 272, 288])
@pytest.mark.parametrize("direction", ["row", "col"])
@pytest.mark.parametrize("rnd", [O.RN, O.SR])
def test_nvfp4_1x16_one_direction_ragged(rows, direction, rnd):
    """One copy only (all warps of the 1x16 kernel on it): row counts that
    are not multiples of 32 (48, 272) take the columnwise path's 8-byte
    stores, 288 its bulk tensor store with a half-filled last row tile;
    528 columns leave a partial column tile."""
    x = W.gen("t3", (rows, 528), 406, bf16=True)
    rw, cw = direction == "row", direction == "col"
    want = O.nvfp4(x, O.B1x16, rnd, seed=3, offset=11, rowwise=rw, colwise=cw)
    got = Q.q_nvfp4(dev(x), "1x16", "rn" if rnd == O.RN else "sr", seed=3, offset=11, rowwise=rw, colwise=cw)
    f32eq(got.s_global.item(), want.s_global, "s_global")
    if rw:
        same(host(got.q_row), want.q_row, "q_row")
        same(host(got.sb_row), want.sb_row, "sb_row")
    else:
        same(host(got.q_colT), want.q_colT, "q_colT")
        same(host(got.sb_colT), want.sb_colT, "sb_colT")


def test_nvfp4_empty():
    got = Q.q_nvfp4(torch.empty((0, 32), dtype=torch.bfloat16, device="cuda"))
    assert got.amax.item() == 0 and got.s_global.item() == 1


def test_e2m1_cast_exhaustive_through_nvfp4():
    """Every BF16 magnitude below 6 reaches the E2M1 conversion unscaled:
    with a given amax of 2688 (alpha_g = 1), a 16-element block whose
    largest entry is 6 has block scale 1 and enc = 1."""
    vals = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 6)]
    n = (len(vals) + 14) // 15 * 15
    vals = np.concatenate([vals, np.zeros(n - len(vals), np.float32)]).reshape(-1, 15)
    blocks = np.concatenate([np.full((vals.shape[0], 1), 6.0, np.float32), vals], axis=1)
    rows = (blocks.shape[0] + 15) // 16 * 16
    x = np.zeros((rows, 16), np.float32)
    x[: blocks.shape[0]] = blocks
    amax = torch.tensor([2688.0], device="cuda")
    want = O.nvfp4(x, O.B1x16, O.RN, rowwise=True, amax_in=2688.0)
    got = Q.q_nvfp4(dev(x), rowwise=True, amax=amax)
    same(host(got.sb_row), want.sb_row)
    same(host(got.q_row), want.q_row)
    assert np.all(want.sb_row[: blocks.shape[0]] == 0x38)


@pytest.mark.parametrize("fmt,fmax", [(O.E4M3, 448.0), (O.E5M2, 57344.0)])
def test_fp8_cast_exhaustive_bf16(fmt, fmax):
    """Every BF16 bit pattern (NaN and inf included) through the cast with
    alpha = Fmax / Fmax = 1: the codes are the plain saturating RTNE cast."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(4096, 16)
    amax = torch.tensor([fmax], device="cuda")
    want = O.current_scaling(x, fmt, rowwise=True, colwise=True, amax_in=fmax)
    got = Q.q_current_scaling(dev(x), "e4m3" if fmt == O.E4M3 else "e5m2", colwise=True, amax=amax)
    f32eq(got.scale.item(), 1.0)
    same(host(got.q_row), want.q_row, "q_row")
    same(host(got.q_colT), want.q_colT, "q_colT")


def test_calls_on_two_streams_run_concurrently_and_match_the_oracle():
    """The calls share no device state: NVFP4 SR and current scaling on one
    stream, blockwise and MXFP8 on another, enqueued back to back without
    synchronizing, give the oracle's results."""
    x1 = W.gen("t3", (1024, 2048), 61, bf16=True)
    x2 = W.gen("normal", (1024, 2048), 62, bf16=True)
    d1, d2 = dev(x1), dev(x2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        nv = Q.q_nvfp4(d1, "1x16", "sr", seed=3, offset=1, colwise=True)
        cs = Q.q_current_scaling(d1, "e5m2", colwise=True)
    with torch.cuda.stream(s2):
        bw = Q.q_blockwise(d2, "1x128", colwise=True)
        mx = Q.q_mxfp8(d2)
    torch.cuda.synchronize()
    w = O.nvfp4(x1, O.B1x16, O.SR, seed=3, offset=1, rowwise=True, colwise=True)
    same(host(nv.q_row), w.q_row, "nv q_row")
    same(host(nv.q_colT), w.q_colT, "nv q_colT")
    w = O.current_scaling(x1, O.E5M2, rowwise=True, colwise=True)
    same(host(cs.q_row), w.q_row, "cs q_row")
    same(host(cs.q_colT), w.q_colT, "cs q_colT")
    w = O.blockwise(x2, O.T1x128, rowwise=True, colwise=True)
    same(host(bw.q_colT), w.q_colT, "bw q_colT")
    same(host(bw.s_colT), w.s_colT, "bw s_colT")
    w = O.mxfp8(x2)
    same(host(mx.q_col), w.q_col, "mx q_col")
    same(host(mx.e8m0_row), w.e8m0_row, "mx e8m0_row")


def test_nvfp4_recipe_row_shards_with_the_global_maxima():
    """Two row shards (16-row boundaries) that take their local maxima from
    q_nvfp4_rht_amax2, reduce them with MAX and cast with the global values
    give the unsharded recipe's outputs (RTNE; the shard helper itself runs
    as one rank)."""
    from nvfp4_quantization_current_gb300.distributed import quantize_shard_nvfp4_recipe
    x = W.gen("outliers", (384, 256), 71, bf16=True)
    whole_row, whole_col = Q.q_nvfp4_recipe(dev(x), 0x2D4B)
    parts = [x[:144], x[144:]]
    maxima = [Q.q_nvfp4_rht_amax2(dev(p), 0x2D4B) for p in parts]
    a_rht = torch.maximum(maxima[0][0], maxima[1][0])
    a_x = torch.maximum(maxima[0][1], maxima[1][1])
    got = [Q.q_nvfp4_recipe(dev(p), 0x2D4B, amax_row=a_x.clone(), amax_col=a_rht.clone()) for p in parts]
    rows, cols = [g[0] for g in got], [g[1] for g in got]
    same(np.concatenate([host(r.q_row) for r in rows]), host(whole_row.q_row), "q_row")
    same(np.concatenate([host(r.sb_row) for r in rows]), host(whole_row.sb_row), "sb_row")
    same(np.concatenate([host(c.q_colT) for c in cols], axis=1), host(whole_col.q_colT), "q_colT")
    same(np.concatenate([host(c.sb_colT) for c in cols], axis=1), host(whole_col.sb_colT), "sb_colT")
    r1, c1 = quantize_shard_nvfp4_recipe(dev(x), 0x2D4B)
    same(host(r1.q_row), host(whole_row.q_row), "helper q_row")
    same(host(c1.q_colT), host(whole_col.q_colT), "helper q_colT")
    # stochastic rounding: each shard moves the Philox offset by its first row
    from nvfp4_quantization_current_gb300.distributed import sr_offset
    sw_row, sw_col = Q.q_nvfp4_recipe(dev(x), 0x2D4B, "sr", 12, 40)
    got = [Q.q_nvfp4_recipe(dev(p), 0x2D4B, "sr", 12, sr_offset(40, r0, x.shape[1]), amax_row=a_x.clone(),
                            amax_col=a_rht.clone()) for p, r0 in zip(parts, (0, 144))]
    same(np.concatenate([host(g[0].q_row) for g in got]), host(sw_row.q_row), "SR q_row")
    same(np.concatenate([host(g[1].q_colT) for g in got], axis=1), host(sw_col.q_colT), "SR q_colT")
    same(np.concatenate([host(g[1].sb_colT) for g in got], axis=1), host(sw_col.sb_colT), "SR sb_colT")


def test_shard_helpers_on_one_rank_equal_the_plain_calls():
    """Without torch.distributed the all-reduce is the identity, so each shard
    helper must give exactly the unsharded call's outputs through the
    library."""
    from nvfp4_quantization_current_gb300 import distributed as D
    x = dev(W.gen("outliers", (256, 384), 91, bf16=True))
    a = D.quantize_shard_current_scaling(x, "e4m3", True, True)
    b = Q.q_current_scaling(x, "e4m3", True, True)
    same(host(a.q_row), host(b.q_row), "cs q_row")
    same(host(a.q_colT), host(b.q_colT), "cs q_colT")
    a = D.quantize_shard_nvfp4(x, "1x16", "sr", 5, 0, True, True)
    b = Q.q_nvfp4(x, "1x16", "sr", 5, 0, True, True)
    same(host(a.q_row), host(b.q_row), "nv q_row")
    same(host(a.q_colT), host(b.q_colT), "nv q_colT")
    a = D.quantize_shard_nvfp4_rht_colT(x, 0x1357, "rn")
    b = Q.q_nvfp4_rht_colT(x, 0x1357, "rn")
    same(host(a.q_colT), host(b.q_colT), "rht q_colT")
    g = D.all_gather_quantized(b)
    assert g.q_colT is b.q_colT
