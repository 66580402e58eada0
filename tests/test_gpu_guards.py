"""Out-of-bounds write check: every output of every entry point is placed
inside a larger buffer filled with 0xA5, with 256 bytes of guard band on each
side, and the bands must be intact after the call.  Shapes are ragged where
the entry point allows it, so that edge tiles, partial row groups and both
copy-out paths run."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

Q = pytest.importorskip("nvfp4_quantization_current_gb300")
G = 256


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    Q.lib()


def dev(x):
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(x.copy()).cuda()


class Guards:
    def __init__(self):
        self.bufs = []

    def like(self, t):
        if t is None:
            return None
        nb = t.numel() * t.element_size()
        buf = torch.full((nb + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
        self.bufs.append((buf, nb))
        return buf[G:G + nb].view(t.dtype).view(t.shape)

    def wrap(self, obj):
        for f in dataclasses.fields(obj):
            v = getattr(obj, f.name)
            if isinstance(v, torch.Tensor):
                setattr(obj, f.name, self.like(v))
        return obj

    def check(self, what):
        torch.cuda.synchronize()
        for i, (buf, nb) in enumerate(self.bufs):
            h = buf.cpu().numpy()
            assert (h[:G] == 0xA5).all(), f"{what}: guard before buffer {i} overwritten"
            assert (h[G + nb:] == 0xA5).all(), f"{what}: guard after buffer {i} overwritten"


@pytest.mark.parametrize("shape,bf16,colwise", [((37, 61), False, False), ((272, 528), True, True), ((16, 16), True, True)])
def test_current_and_delayed_scaling_stay_in_bounds(shape, bf16, colwise):
    x = W.gen("outliers", shape, 1, bf16=bf16)
    g = Guards()
    amax = g.like(torch.empty(1, device="cuda"))
    Q.q_amax(dev(x), out=amax)
    out = g.wrap(Q.alloc_current_scaling(*shape, "cuda", "e4m3", True, colwise))
    Q.q_current_scaling(dev(x), "e4m3", True, colwise, out=out)
    ref = O.current_scaling(x, O.E4M3, True, colwise)
    assert np.array_equal(out.q_row.cpu().numpy(), ref.q_row)
    y = g.like(torch.empty(shape, dtype=torch.float32, device="cuda"))
    Q.dq_current_scaling(out.q_row, out.scale, "e4m3", torch.float32, out=y)
    st = Q.DelayedScaling("e5m2", history_len=4)
    ds_out = g.wrap(Q.alloc_current_scaling(*shape, "cuda", "e5m2", True, colwise))
    slot = g.like(torch.empty(1, device="cuda"))
    Q.q_delayed_scaling(dev(x), st.ds, slot, "e5m2", True, colwise, out=ds_out)
    ds = g.like(torch.empty(2, device="cuda"))
    Q.q_delayed_scale_update(st.hist, 1, ds, "e5m2")
    g.check(f"current / delayed scaling {shape}")


@pytest.mark.parametrize("shape,bf16", [((96, 800), True), ((64, 416), False), ((32, 32), True)])
def test_mxfp8_and_requant_stay_in_bounds(shape, bf16):
    x = W.gen("lognormal_rows", shape, 2, bf16=bf16)
    g = Guards()
    out = g.wrap(Q.alloc_mxfp8(*shape, "cuda", "e4m3", True, True))
    Q.q_mxfp8(dev(x), "e4m3", True, True, out=out)
    rq = g.wrap(Q.alloc_mxfp8(*shape, "cuda", "e4m3", False, True))
    Q.q_mxfp8_requant_col(out.q_row, out.e8m0_row, "e4m3", out=rq)
    for d, q, e in ((Q.Q_ROW, out.q_row, out.e8m0_row), (Q.Q_COL, out.q_col, out.e8m0_col)):
        y = g.like(torch.empty(shape, dtype=torch.bfloat16, device="cuda"))
        Q.dq_mxfp8(q, e, "e4m3", d, torch.bfloat16, out=y)
    g.check(f"mxfp8 {shape}")


@pytest.mark.parametrize("tile,shape,colwise", [("1x128", (256, 384), True), ("1x128", (100, 256), False),
                                                ("128x128", (256, 384), True), ("128x128", (128, 128), True)])
def test_blockwise_stays_in_bounds(tile, shape, colwise):
    x = W.gen("normal", shape, 3, bf16=True)
    g = Guards()
    out = g.wrap(Q.alloc_blockwise(*shape, "cuda", tile, True, colwise))
    Q.q_blockwise(dev(x), tile, True, colwise, out=out)
    y = g.like(torch.empty(shape, dtype=torch.bfloat16, device="cuda"))
    Q.dq_blockwise(out.q_row, out.s_row, tile, torch.bfloat16, out=y)
    g.check(f"blockwise {tile} {shape}")


@pytest.mark.parametrize("tile,shape,colwise", [("1x128", (256, 384), True), ("1x128", (100, 256), False),
                                                ("128x128", (256, 384), True), ("128x128", (128, 128), True),
                                                ("128x128", (128, 512), True)])
def test_blockwise_mx_stays_in_bounds(tile, shape, colwise):
    x = W.gen("normal", shape, 3, bf16=True)
    g = Guards()
    out = g.wrap(Q.alloc_blockwise_mx(*shape, "cuda", tile, True, colwise))
    Q.q_blockwise_mx(dev(x), tile, True, colwise, out=out)
    y = g.like(torch.empty(shape, dtype=torch.bfloat16, device="cuda"))
    Q.dq_mxfp8(out.q_row, out.e8m0_row, "e4m3", Q.Q_ROW, torch.bfloat16, out=y)
    g.check(f"blockwise_mx {tile} {shape}")


@pytest.mark.parametrize("blk,rnd,shape", [("1x16", "rn", (272, 528)), ("1x16", "sr", (256, 512)),
                                           ("16x16", "rn", (144, 272)), ("1x16", "rn", (48, 160))])
def test_nvfp4_and_rht_stay_in_bounds(blk, rnd, shape):
    x = W.gen("t3", shape, 4, bf16=True)
    g = Guards()
    out = g.wrap(Q.alloc_nvfp4(*shape, "cuda", blk, True, True))
    Q.q_nvfp4(dev(x), blk, rnd, 3, 0, True, True, out=out)
    for q, sb in ((out.q_row, out.sb_row), (out.q_colT, out.sb_colT)):
        y = g.like(torch.empty((q.shape[0], q.shape[1] * 2), dtype=torch.bfloat16, device="cuda"))
        Q.dq_nvfp4(q, sb, out.s_global, blk, torch.bfloat16, out=y)
    if blk == "1x16":
        rw = g.wrap(Q.alloc_nvfp4(*shape, "cuda", "1x16", True, False))
        cl = g.wrap(Q.alloc_nvfp4(*shape, "cuda", "1x16", False, True))
        Q.q_nvfp4_recipe(dev(x), 0x3C5A, rnd, 3, 0, out=(rw, cl))
        h = g.wrap(Q.alloc_nvfp4(*shape, "cuda", "1x16", False, True))
        Q.q_nvfp4_rht_colT(dev(x), 0x3C5A, rnd, 3, 0, out=h)
        a = g.like(torch.empty(1, device="cuda"))
        Q.q_nvfp4_rht_amax(dev(x), 0x3C5A, out=a)
    g.check(f"nvfp4 {blk} {rnd} {shape}")
