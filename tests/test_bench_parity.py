"""The benchmark's full-size parity check on CPU: bench.parity_check runs
against a stand-in for the library whose every call is the oracle on the
whole tensor.  The check compares the whole-tensor results with the oracle
run band by band (with the whole tensor's maxima and the bands' counter
offsets), so it passes only if each recipe's outputs compose from row bands
exactly as the check slices them -- the property the GPU run relies on."""
import types

import numpy as np
import pytest
import torch

import bench
import oracle as O
import workloads as W

FMT = {"e4m3": O.E4M3, "e5m2": O.E5M2}


def t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(a.copy())


def h(x):
    return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()


def scalar(v):
    return torch.tensor([v], dtype=torch.float32)


def oracle_library():
    """Whole-tensor oracle calls with the library's Python signatures."""
    Q = types.SimpleNamespace(Q_ROW=O.ROW, Q_COL=O.COL)
    ns = types.SimpleNamespace

    def out(dtype):
        return O.BF16 if dtype == torch.bfloat16 else O.F32

    def q_current_scaling(x, fmt, rowwise, colwise):
        w = O.current_scaling(h(x), FMT[fmt], True, True)
        return ns(q_row=t(w.q_row), q_colT=t(w.q_colT), amax=scalar(w.amax), scale=scalar(w.scale))

    def dq_current_scaling(q, s, fmt, dtype):
        return t(O.dq_current_scaling(h(q), s.item(), FMT[fmt], out(dtype)))

    class DelayedScaling:
        def __init__(self, fmt, history_len):
            self.fmt, self.hist, self.t = FMT[fmt], np.zeros(history_len, np.float32), 0
            self.ds = torch.tensor([1.0, 1.0])

        def quantize(self, x, rowwise, colwise):
            q_row, q_colT, a = O.ds_cast(h(x), self.ds[0].item(), self.fmt, True, True)
            self.hist[self.t] = a
            self.ds = torch.tensor(O.ds_scale_update(self.hist, self.t, O.HIST_MAX, self.fmt), dtype=torch.float32)
            self.t += 1
            return ns(q_row=t(q_row), q_colT=t(q_colT), amax=scalar(a))

    def q_mxfp8(x):
        w = O.mxfp8(h(x))
        return ns(q_row=t(w.q_row), e8m0_row=t(w.e8m0_row), q_col=t(w.q_col), e8m0_col=t(w.e8m0_col))

    def q_mxfp8_requant_col(q_row, e_row):
        q, e = O.mxfp8_requant_col(h(q_row), h(e_row))
        return ns(q_col=t(q), e8m0_col=t(e))

    def dq_mxfp8(q, e, fmt, direction, dtype):
        return t(O.dq_mxfp8(h(q), h(e), FMT[fmt], direction, out(dtype)))

    tiles = {"1x128": O.T1x128, "128x128": O.T128x128}

    def q_blockwise(x, tile, rowwise, colwise):
        w = O.blockwise(h(x), tiles[tile], True, True)
        return ns(q_row=t(w.q_row), s_row=t(w.s_row), q_colT=t(w.q_colT), s_colT=t(w.s_colT))

    def dq_blockwise(q, s, tile, dtype):
        return t(O.dq_blockwise(h(q), h(s), tiles[tile], out(dtype)))

    def q_blockwise_mx(x, tile, rowwise, colwise):
        w = O.blockwise_mx(h(x), tiles[tile], True, True)
        return ns(q_row=t(w.q_row), e8m0_row=t(w.e8m0_row), q_colT=t(w.q_colT), e8m0_colT=t(w.e8m0_colT))

    blks = {"1x16": O.B1x16, "16x16": O.B16x16}
    rnds = {"rn": O.RN, "sr": O.SR}

    def q_nvfp4(x, blk, rnd, seed, offset, rowwise, colwise):
        w = O.nvfp4(h(x), blks[blk], rnds[rnd], seed=seed, offset=offset, rowwise=True, colwise=True)
        return ns(q_row=t(w.q_row), sb_row=t(w.sb_row), q_colT=t(w.q_colT), sb_colT=t(w.sb_colT),
                  amax=scalar(w.amax), s_global=scalar(w.s_global))

    def dq_nvfp4(q, sb, sg, blk, dtype):
        return t(O.dq_nvfp4(h(q), h(sb), sg.item(), blks[blk], out(dtype)))

    def q_nvfp4_rht_colT(x, mask, rnd, seed, offset):
        q, sb, a, sg = O.nvfp4_rht_colT(h(x), mask, rnds[rnd], seed=seed, offset=offset)
        return ns(q_colT=t(q), sb_colT=t(sb), amax=scalar(a), s_global=scalar(sg))

    def q_nvfp4_recipe(x, mask, rnd, seed, offset):
        r = q_nvfp4(x, "1x16", rnd, seed, offset, True, False)
        return r, q_nvfp4_rht_colT(x, mask, rnd, seed, offset)

    for f in (q_current_scaling, dq_current_scaling, q_mxfp8, q_mxfp8_requant_col, dq_mxfp8, q_blockwise,
              dq_blockwise, q_blockwise_mx, q_nvfp4, dq_nvfp4, q_nvfp4_rht_colT, q_nvfp4_recipe):
        setattr(Q, f.__name__, f)
    Q.DelayedScaling = DelayedScaling
    return Q


def small_workloads():
    """The step's tensors at 2176 x 256 (two full 1024-row bands and a 128-row
    tail; 17 tiles of 128 rows), same distributions."""
    shape = (2176, 256)
    spec = {"cs1": {"x": ("outliers", False)}, "mx2": {"act": ("lognormal_rows", True)},
            "bw3": {"act": ("normal", True), "w": ("weight", True)},
            "hy4": {"grad": ("grad", True), "w": ("weight", True)},
            "nv5": {"act": ("normal", True), "grad": ("t3", True), "w": ("weight", True)}}
    return {wl: {tn: W.gen(kind, shape, 900 + i, bf16=b) for i, (tn, (kind, b)) in enumerate(d.items())}
            for wl, d in spec.items()}


@pytest.mark.parametrize("full", [True, False])
def test_parity_check_composes_bands_into_the_whole_tensor(full, monkeypatch):
    monkeypatch.setattr(bench, "PARITY_BAND_ROWS", 1024)
    host_t = small_workloads()
    dev_t = {wl: {tn: t(a) for tn, a in d.items()} for wl, d in host_t.items()}
    fields, nbytes = bench.parity_check(host_t, dev_t, torch, oracle_library(), O, full=full, threads=4)
    assert fields > 0 and nbytes > 0
    if full:
        # every output byte of every call: e.g. the NVFP4 SR copies, 2 x 2176 x 256 / 2 bytes each
        assert nbytes > 2176 * 256 * 20


def test_parity_check_catches_a_wrong_band():
    """A library result with one wrong byte in the last band fails the check."""
    host_t = small_workloads()
    host_t = {"nv5": host_t["nv5"]}
    dev_t = {wl: {tn: t(a) for tn, a in d.items()} for wl, d in host_t.items()}
    Q = oracle_library()
    good = Q.q_nvfp4

    def bad(*a, **k):
        r = good(*a, **k)
        r.q_colT[5, -1] ^= 0x10
        return r
    Q.q_nvfp4 = bad
    with pytest.raises(AssertionError, match="q_colT"):
        bench.parity_check(host_t, dev_t, torch, Q, O, full=True, threads=2)
