"""Tensors past 2^31 elements: every element index, row and column offset,
transposed address and SR counter of the kernels is 64-bit.  A 65792 x 32768
BF16 tensor (2.16e9 elements, 4.3 GB) is drawn on the device from a seeded
generator in (-1, 1); the last 16 rows of its last column are set to 3.5
times the signs of the random-Hadamard mask, so the tensor's amax is 3.5
and the amax of its transform is 14 (that group becomes (14, 0, ..., 0);
every other group stays below 16 / 4), both by construction and at the
highest indices.  The oracle recomputes the last 256-row band (with the
tensor-wide maxima where the recipe needs one, and the band's counter
offset for stochastic rounding), and every output that band determines is
compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

Q = pytest.importorskip("nvfp4_quantization_current_gb300")

M, K = 65536 + 256, 32768          # M * K = 2,155,872,256 > 2^31
BAND = 256
A = np.float32(3.5)
MASK = 0x6B1D
A_RHT = np.float32(14.0)


@pytest.fixture(scope="module")
def big():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    Q.lib()
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    x.uniform_(-0.999, 0.999, generator=g)
    signs = torch.tensor([-1.0 if (MASK >> i) & 1 else 1.0 for i in range(16)], device="cuda")
    x[M - 16:, K - 1] = (float(A) * signs).to(torch.bfloat16)
    band = x[M - BAND:].view(torch.int16).cpu().numpy().view(np.uint16)
    yield x, band
    del x
    torch.cuda.empty_cache()


def host(t):
    return t.cpu().numpy()


def same(a, b, what):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.argwhere(a != b)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:3].tolist()}"


def test_current_scaling_past_2_31_elements(big):
    x, band = big
    got = Q.q_current_scaling(x, "e4m3", rowwise=True, colwise=True)
    assert got.amax.item() == A
    want = O.current_scaling(band, O.E4M3, rowwise=True, colwise=True, amax_in=float(A))
    same(np.float32(got.scale.item()), np.float32(want.scale), "scale")
    same(host(got.q_row[M - BAND:]), want.q_row, "q_row band")
    same(host(got.q_colT[:, M - BAND:]), want.q_colT, "q_colT band")
    y = Q.dq_current_scaling(got.q_row, got.scale, "e4m3", torch.bfloat16)
    same(y[M - BAND:].view(torch.int16).cpu().numpy().view(np.uint16),
         O.dq_current_scaling(want.q_row, want.scale, O.E4M3, O.BF16), "dq band")
    del got, y
    # rowwise only: the flat cast kernel
    got = Q.q_current_scaling(x, "e5m2", rowwise=True, colwise=False)
    want = O.current_scaling(band, O.E5M2, rowwise=True, colwise=False, amax_in=float(A))
    same(host(got.q_row[M - BAND:]), want.q_row, "flat q_row band")


def test_nvfp4_past_2_31_elements(big):
    x, band = big
    got = Q.q_nvfp4(x, "1x16", "rn", rowwise=True, colwise=True)
    assert got.amax.item() == A
    want = O.nvfp4(band, O.B1x16, O.RN, rowwise=True, colwise=True, amax_in=float(A))
    same(np.float32(got.s_global.item()), np.float32(want.s_global), "s_global")
    same(host(got.q_row[M - BAND:]), want.q_row, "q_row band")
    same(host(got.sb_row[M - BAND:]), want.sb_row, "sb_row band")
    same(host(got.q_colT[:, (M - BAND) // 2:]), want.q_colT, "q_colT band")
    same(host(got.sb_colT[:, (M - BAND) // 16:]), want.sb_colT, "sb_colT band")
    del got
    # stochastic rounding: the band draws what the whole tensor draws there with counter offset
    # offset + (M - BAND) * K / 16, in both copies
    got = Q.q_nvfp4(x, "1x16", "sr", seed=77, offset=5, rowwise=True, colwise=True)
    want = O.nvfp4(band, O.B1x16, O.SR, seed=77, offset=5 + (M - BAND) * K // 16, rowwise=True, colwise=True,
                   amax_in=float(A))
    same(host(got.q_row[M - BAND:]), want.q_row, "SR q_row band")
    same(host(got.q_colT[:, (M - BAND) // 2:]), want.q_colT, "SR q_colT band")
    same(host(got.sb_colT[:, (M - BAND) // 16:]), want.sb_colT, "SR sb_colT band")
    del got
    for rnd, orn in (("rn", O.RN), ("sr", O.SR)):
        got = Q.q_nvfp4(x, "16x16", rnd, seed=9, offset=3, rowwise=True, colwise=True)
        want = O.nvfp4(band, O.B16x16, orn, seed=9, offset=3 + (M - BAND) * K // 16, rowwise=True, colwise=True,
                       amax_in=float(A))
        same(host(got.q_row[M - BAND:]), want.q_row, f"16x16 {rnd} q_row band")
        same(host(got.sb_row[(M - BAND) // 16:]), want.sb_row, f"16x16 {rnd} sb_row band")
        same(host(got.q_colT[:, (M - BAND) // 2:]), want.q_colT, f"16x16 {rnd} q_colT band")
        same(host(got.sb_colT[:, (M - BAND) // 16:]), want.sb_colT, f"16x16 {rnd} sb_colT band")
        del got


def test_nvfp4_rht_and_recipe_past_2_31_elements(big):
    x, band = big
    for rnd, orn in (("rn", O.RN), ("sr", O.SR)):
        got = Q.q_nvfp4_rht_colT(x, MASK, rnd, seed=21, offset=8)
        assert got.amax.item() == A_RHT
        q, sb, _, sg = O.nvfp4_rht_colT(band, MASK, orn, seed=21, offset=8 + (M - BAND) * K // 16,
                                        amax_in=float(A_RHT))
        same(np.float32(got.s_global.item()), np.float32(sg), f"rht {rnd} s_global")
        same(host(got.q_colT[:, (M - BAND) // 2:]), q, f"rht {rnd} q_colT band")
        same(host(got.sb_colT[:, (M - BAND) // 16:]), sb, f"rht {rnd} sb_colT band")
        del got
    row, col = Q.q_nvfp4_recipe(x, MASK, "sr", seed=21, offset=8)
    assert row.amax.item() == A and col.amax.item() == A_RHT
    w = O.nvfp4(band, O.B1x16, O.SR, seed=21, offset=8 + (M - BAND) * K // 16, rowwise=True, colwise=False,
                amax_in=float(A))
    q, sb, _, _ = O.nvfp4_rht_colT(band, MASK, O.SR, seed=21, offset=8 + (M - BAND) * K // 16, amax_in=float(A_RHT))
    same(host(row.q_row[M - BAND:]), w.q_row, "recipe q_row band")
    same(host(row.sb_row[M - BAND:]), w.sb_row, "recipe sb_row band")
    same(host(col.q_colT[:, (M - BAND) // 2:]), q, "recipe q_colT band")
    same(host(col.sb_colT[:, (M - BAND) // 16:]), sb, "recipe sb_colT band")


def test_block_recipes_past_2_31_elements(big):
    x, band = big
    got = Q.q_blockwise(x, "1x128", rowwise=True, colwise=True)
    want = O.blockwise(band, O.T1x128, rowwise=True, colwise=True)
    same(host(got.q_row[M - BAND:]), want.q_row, "blockwise q_row band")
    same(host(got.s_row[M - BAND:]), want.s_row, "blockwise s_row band")
    same(host(got.q_colT[:, M - BAND:]), want.q_colT, "blockwise q_colT band")
    same(host(got.s_colT[:, (M - BAND) // 128:]), want.s_colT, "blockwise s_colT band")
    del got
    got = Q.q_blockwise(x, "128x128", rowwise=True, colwise=True)
    want = O.blockwise(band, O.T128x128, rowwise=True, colwise=True)
    same(host(got.q_row[M - BAND:]), want.q_row, "blockwise 128x128 q_row band")
    same(host(got.s_row[(M - BAND) // 128:]), want.s_row, "blockwise 128x128 s_row band")
    same(host(got.q_colT[:, M - BAND:]), want.q_colT, "blockwise 128x128 q_colT band")
    same(host(got.s_colT[:, (M - BAND) // 128:]), want.s_colT, "blockwise 128x128 s_colT band")
    del got
    got = Q.q_mxfp8(x, "e4m3")
    want = O.mxfp8(band, O.E4M3)
    same(host(got.q_row[M - BAND:]), want.q_row, "mxfp8 q_row band")
    same(host(got.e8m0_row[M - BAND:]), want.e8m0_row, "mxfp8 e8m0_row band")
    same(host(got.q_col[M - BAND:]), want.q_col, "mxfp8 q_col band")
    same(host(got.e8m0_col[(M - BAND) // 32:]), want.e8m0_col, "mxfp8 e8m0_col band")
