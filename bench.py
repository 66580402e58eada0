#!/usr/bin/env python
"""Benchmark of the quantizer hot path on synthetic tensors shaped like the
pages' workloads.

One step = one pass of every recipe over its full-size tensors (all five
workloads of ``workloads.WORKLOADS``): current-scaling amax + cast (+ the
transposed copy), delayed scaling (one read + the window update), MXFP8
row + col and the row->col re-quantize, blockwise 1x128 (+ transposed) and
128x128 (+ transposed), both again with power-of-two tile scales held as
MXFP8, NVFP4 1x16 RTNE, 1x16 stochastic rounding and 16x16,
the dequantizer of each, and the random-Hadamard NVFP4 columnwise copies of
the NVFP4 activation and gradient (weight-gradient GEMM inputs), and the
NVFP4 recipe's two copies of the gradient (rowwise SR + random-Hadamard
columnwise SR, one amax pass for both).  Every call goes through the C ABI with
preallocated outputs.

Metric: quantize GB/s = algorithmic bytes (input bytes x reads + all output
bytes; reads = 2 for current scaling and NVFP4, whose amax pass reads the
tensor once more, 1 otherwise) / device time, summed over the step.  L2 is
flushed before every timed call: a 256 MiB write, then a 256 MiB read of
another buffer, which evicts the written lines so that their write-back is
not charged to the call.  The time of a call is taken with one pair of CUDA
events on the launching stream around that call only (its kernels overlap as
they do for a caller).  A second timed region of the same K steps records an
event after every kernel for the per-kernel breakdown and the roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the plain C reference
implementation) on a bounded row sample of the same workload instead.
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "quantize GB/s (bytes read+written) and % of GB300 HBM peak per recipe"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
CPU_SAMPLE_FRAC = 1.0 / 2.0
REF_BUDGET_S = 120.0
RHT_MASK = 0xB4E1   # the 16 random signs of the Hadamard transform (any fixed draw)

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu --set full capture of the kernel on the named call (key "workload.tensor:
# piece"), with the kernel, the commit the capture measured, and the hash of
# the kernel's source (file + shared device headers) at capture time;
# reported as null once the source has changed since.
TRAFFIC = {
    "bw3.w:bwmx_128x128_T": {"kernel": "qk::k_blockwise<0, 1, 1>", "capture_commit": "a00210f",
                             "bytes_per_launch": 485297664, "src_hash": "076d29a3116c64ea"},
}


def src_hash(fname):
    """Hash of a kernel's source file plus the shared device headers."""
    h = hashlib.sha256()
    for name in (fname, "q_common.cuh", "q_engine.cuh"):
        with open(os.path.join(ROOT, "nvfp4_quantization_current_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------
# the step: a list of calls, each a list of (kernel name, source file,
# algorithmic bytes, thunk issuing one C-ABI call)
# --------------------------------------------------------------------------

class Call:
    def __init__(self, name, recipe, pieces, h2d, d2h, e2e_thunk):
        self.name = name            # e.g. "hy4.grad cs_e5m2 row+colT"
        self.recipe = recipe        # current_scaling | mxfp8 | blockwise | nvfp4 | dequant
        self.pieces = pieces        # [(kernel, srcfile, alg_bytes, thunk)]
        self.h2d = h2d              # input tensors (device) whose bytes an end-to-end call copies in
        self.d2h = d2h              # output tensors copied back end to end
        self.e2e_thunk = e2e_thunk  # the single public-API call (amax computed inside)
        self.prime = None           # copies a producer call's outputs into this call's own inputs

    @property
    def alg_bytes(self):
        return sum(p[2] for p in self.pieces)


def nbytes(*ts):
    return sum(int(t.numel() * t.element_size()) for t in ts if t is not None)


def build_step(dev_tensors, torch, Q):
    """Preallocate every output and return the list of calls of one step.
    A call that consumes another call's outputs (a dequantizer, the MXFP8
    re-quantize) reads device buffers of its own, filled from the producer's
    outputs once before timing (``Call.prime``): its end-to-end upload then
    never waits for the producer's download of the same buffer."""
    calls = []
    d = dev_tensors

    def own(*ts):
        mine = [torch.empty_like(t) for t in ts]

        def prime():
            for m, t in zip(mine, ts):
                m.copy_(t)
        return mine, prime

    def cs(tag, x, fmt, colwise):
        out = Q.alloc_current_scaling(x.shape[0], x.shape[1], x.device, fmt, True, colwise)
        amax = out.amax
        ins = nbytes(x)
        outs = nbytes(out.q_row, out.q_colT, out.scale)
        pieces = [
            ("amax", "k_current_scaling.cu", ins, lambda: Q.q_amax(x, out=amax)),
            ("cs_cast" + ("_T" if colwise else ""), "k_current_scaling.cu", ins + outs + 4,
             lambda: Q.q_current_scaling(x, fmt, True, colwise, amax=amax, out=out)),
        ]

        def e2e():
            o = Q.q_current_scaling(x, fmt, True, colwise, out=out)
            o.amax = amax
            return o
        calls.append(Call(f"{tag} cs_{fmt} row{'+colT' if colwise else ''}", "current_scaling", pieces, [x],
                          [out.q_row, out.q_colT, out.scale], e2e))
        y = torch.empty(x.shape, dtype=torch.bfloat16 if x.dtype == torch.bfloat16 else torch.float32, device=x.device)
        (qd, sd), prime = own(out.q_row, out.scale)
        r = lambda: Q.dq_current_scaling(qd, sd, fmt, y.dtype, out=y)
        calls.append(Call(f"{tag} dq_cs row->{str(y.dtype)[6:]}", "dequant",
                          [("dq_cs", "k_dequant.cu", nbytes(qd, sd, y), r)], [qd, sd], [y], r))
        calls[-1].prime = prime

    def ds(tag, x, fmt, N=1024):
        st = Q.DelayedScaling(fmt, history_len=N, algo="max", device=x.device)
        out = Q.alloc_current_scaling(x.shape[0], x.shape[1], x.device, fmt, True, True)
        slot = st.hist[0:1]
        pieces = [
            ("ds_cast_T", "k_current_scaling.cu", nbytes(x, out.q_row, out.q_colT, out.scale, slot, st.ds),
             lambda: Q.q_delayed_scaling(x, st.ds, slot, fmt, True, True, out=out)),
            ("ds_update", "k_current_scaling.cu", nbytes(st.hist, st.ds),
             lambda: Q.q_delayed_scale_update(st.hist, 0, st.ds, fmt, "max")),
        ]
        calls.append(Call(f"{tag} ds_{fmt} row+colT", "delayed_scaling", pieces, [x],
                          [out.q_row, out.q_colT, out.scale], lambda: st.quantize(x, True, True, out=out)))

    def mx(tag, x):
        out = Q.alloc_mxfp8(x.shape[0], x.shape[1], x.device, "e4m3", True, True)
        b = nbytes(x, out.q_row, out.e8m0_row, out.q_col, out.e8m0_col)
        run = lambda: Q.q_mxfp8(x, "e4m3", True, True, out=out)
        calls.append(Call(f"{tag} mxfp8_e4m3 row+col", "mxfp8", [("mxfp8", "k_mxfp8.cu", b, run)], [x],
                          [out.q_row, out.e8m0_row, out.q_col, out.e8m0_col], run))
        rq = Q.alloc_mxfp8(x.shape[0], x.shape[1], x.device, "e4m3", False, True)
        (qr, er), prime = own(out.q_row, out.e8m0_row)
        rrun = lambda: Q.q_mxfp8_requant_col(qr, er, "e4m3", out=rq)
        calls.append(Call(f"{tag} mxfp8_requant row->col", "mxfp8",
                          [("mxfp8_requant", "k_mxfp8.cu", nbytes(qr, er, rq.q_col, rq.e8m0_col), rrun)],
                          [qr, er], [rq.q_col, rq.e8m0_col], rrun))
        calls[-1].prime = prime
        for direction, q0, e0 in ((Q.Q_ROW, out.q_row, out.e8m0_row), (Q.Q_COL, out.q_col, out.e8m0_col)):
            y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
            (q, e), prime = own(q0, e0)
            r = (lambda q=q, e=e, direction=direction, y=y: Q.dq_mxfp8(q, e, "e4m3", direction, torch.bfloat16, out=y))
            calls.append(Call(f"{tag} dq_mxfp8 {'row' if direction == Q.Q_ROW else 'col'}->bf16", "dequant",
                              [("dq_mxfp8", "k_dequant.cu", nbytes(q, e, y), r)], [q, e], [y], r))
            calls[-1].prime = prime

    def bw(tag, x, tile, colwise):
        out = Q.alloc_blockwise(x.shape[0], x.shape[1], x.device, tile, True, colwise)
        b = nbytes(x, out.q_row, out.s_row, out.q_colT, out.s_colT)
        run = lambda: Q.q_blockwise(x, tile, True, colwise, out=out)
        calls.append(Call(f"{tag} blockwise_{tile} row{'+colT' if colwise else ''}", "blockwise",
                          [("bw_" + tile + ("_T" if colwise else ""), "k_blockwise.cu", b, run)], [x],
                          [out.q_row, out.s_row, out.q_colT, out.s_colT], run))
        y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
        (qb, sb), prime = own(out.q_row, out.s_row)
        r = lambda: Q.dq_blockwise(qb, sb, tile, torch.bfloat16, out=y)
        calls.append(Call(f"{tag} dq_blockwise_{tile} row->bf16", "dequant",
                          [("dq_blockwise", "k_dequant.cu", nbytes(qb, sb, y), r)], [qb, sb], [y], r))
        calls[-1].prime = prime

    def bwmx(tag, x, tile):
        out = Q.alloc_blockwise_mx(x.shape[0], x.shape[1], x.device, tile, True, True)
        b = nbytes(x, out.q_row, out.e8m0_row, out.q_colT, out.e8m0_colT)
        run = lambda: Q.q_blockwise_mx(x, tile, True, True, out=out)
        calls.append(Call(f"{tag} blockwise_mx_{tile} row+colT", "blockwise_mx",
                          [("bwmx_" + tile + "_T", "k_blockwise.cu", b, run)], [x],
                          [out.q_row, out.e8m0_row, out.q_colT, out.e8m0_colT], run))

    def nv(tag, x, blk, rnd, seed):
        out = Q.alloc_nvfp4(x.shape[0], x.shape[1], x.device, blk, True, True)
        amax = out.amax
        ins = nbytes(x)
        outs = nbytes(out.q_row, out.sb_row, out.q_colT, out.sb_colT, out.s_global)
        pieces = [
            ("amax", "k_current_scaling.cu", ins, lambda: Q.q_amax(x, out=amax)),
            (f"nvfp4_{blk}_{rnd}", "k_nvfp4_bf16.cu" if x.dtype == torch.bfloat16 else "k_nvfp4.cu", ins + outs + 4,
             lambda: Q.q_nvfp4(x, blk, rnd, seed, 0, True, True, amax=amax, out=out)),
        ]

        def e2e():
            o = Q.q_nvfp4(x, blk, rnd, seed, 0, True, True, out=out)
            o.amax = amax
            return o
        calls.append(Call(f"{tag} nvfp4_{blk}_{rnd} row+colT", "nvfp4", pieces, [x],
                          [out.q_row, out.sb_row, out.q_colT, out.sb_colT, out.s_global], e2e))
        y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
        (qn, sbn, sgn), prime = own(out.q_row, out.sb_row, out.s_global)
        r = lambda: Q.dq_nvfp4(qn, sbn, sgn, blk, torch.bfloat16, out=y)
        calls.append(Call(f"{tag} dq_nvfp4_{blk} row->bf16", "dequant",
                          [("dq_nvfp4", "k_dequant.cu", nbytes(qn, sbn, sgn, y), r)], [qn, sbn, sgn], [y], r))
        calls[-1].prime = prime

    def rht(tag, x, rnd, seed, mask=RHT_MASK):
        out = Q.alloc_nvfp4(x.shape[0], x.shape[1], x.device, "1x16", rowwise=False, colwise=True)
        amax = out.amax
        ins = nbytes(x)
        pieces = [
            ("rht_amax", "k_nvfp4.cu", ins, lambda: Q.q_nvfp4_rht_amax(x, mask, out=amax)),
            (f"nvfp4_rht_colT_{rnd}", "k_nvfp4.cu", ins + nbytes(out.q_colT, out.sb_colT, out.s_global) + 4,
             lambda: Q.q_nvfp4_rht_colT(x, mask, rnd, seed, 0, amax=amax, out=out)),
        ]

        def e2e():
            o = Q.q_nvfp4_rht_colT(x, mask, rnd, seed, 0, out=out)
            o.amax = amax
            return o
        calls.append(Call(f"{tag} nvfp4_rht_{rnd} colT", "nvfp4_rht", pieces, [x],
                          [out.q_colT, out.sb_colT, out.s_global], e2e))

    def recipe(tag, x, rnd, seed, mask=RHT_MASK):
        M, K = x.shape
        row = Q.alloc_nvfp4(M, K, x.device, "1x16", rowwise=True, colwise=False)
        col = Q.alloc_nvfp4(M, K, x.device, "1x16", rowwise=False, colwise=True)
        ins = nbytes(x)
        pieces = [("rht_amax2", "k_nvfp4.cu", ins, lambda: Q.q_nvfp4_rht_amax2(x, mask, out=(col.amax, row.amax)))]
        if x.dtype == torch.bfloat16:
            # one kernel writes both copies from one read of x, the maxima given
            pieces.append((f"nvfp4_recipe_{rnd}", "k_nvfp4_bf16.cu",
                           ins + nbytes(row.q_row, row.sb_row, row.s_global, col.q_colT, col.sb_colT, col.s_global) + 8,
                           lambda: Q.q_nvfp4_recipe(x, mask, rnd, seed, 0, amax_row=row.amax, amax_col=col.amax,
                                                    out=(row, col))))
        else:
            pieces += [
                (f"nvfp4_row_{rnd}", "k_nvfp4.cu", ins + nbytes(row.q_row, row.sb_row, row.s_global) + 4,
                 lambda: Q.q_nvfp4(x, "1x16", rnd, seed, 0, True, False, amax=row.amax, out=row)),
                (f"nvfp4_rht_colT_{rnd}", "k_nvfp4.cu", ins + nbytes(col.q_colT, col.sb_colT, col.s_global) + 4,
                 lambda: Q.q_nvfp4_rht_colT(x, mask, rnd, seed, 0, amax=col.amax, out=col)),
            ]
        calls.append(Call(f"{tag} nvfp4_recipe_{rnd} row + RHT colT", "nvfp4_recipe", pieces, [x],
                          [row.q_row, row.sb_row, row.s_global, col.q_colT, col.sb_colT, col.s_global],
                          lambda: Q.q_nvfp4_recipe(x, mask, rnd, seed, 0, out=(row, col))))

    if "cs1" in d:
        cs("cs1.x", d["cs1"]["x"], "e4m3", True)
    if "mx2" in d:
        mx("mx2.act", d["mx2"]["act"])
    if "bw3" in d:
        bw("bw3.act", d["bw3"]["act"], "1x128", True)
        bw("bw3.w", d["bw3"]["w"], "128x128", True)
        bwmx("bw3.act", d["bw3"]["act"], "1x128")
        bwmx("bw3.w", d["bw3"]["w"], "128x128")
    if "hy4" in d:
        cs("hy4.grad", d["hy4"]["grad"], "e5m2", True)
        ds("hy4.grad", d["hy4"]["grad"], "e5m2")
        cs("hy4.w", d["hy4"]["w"], "e4m3", True)
    if "nv5" in d:
        nv("nv5.act", d["nv5"]["act"], "1x16", "rn", 0)
        nv("nv5.grad", d["nv5"]["grad"], "1x16", "sr", 4)
        nv("nv5.w", d["nv5"]["w"], "16x16", "rn", 0)
        rht("nv5.act", d["nv5"]["act"], "rn", 0)
        rht("nv5.grad", d["nv5"]["grad"], "sr", 4)
        recipe("nv5.grad", d["nv5"]["grad"], "sr", 4)
    return calls


# --------------------------------------------------------------------------
# 0-ULP parity of the full-size outputs against the oracle
# --------------------------------------------------------------------------

PARITY_BAND_ROWS = 1024


def parity_check(host_t, dev_t, torch, Q, O, full=True, threads=None, seed=0):
    """Every output of every call of the step on the full-size tensors,
    compared bit for bit with the oracle.  full=True compares every row band
    of every tensor (the whole outputs); full=False one random 128-row band
    per tensor.  The oracle runs over row bands on a pool of threads (its
    ctypes calls release the GIL), with the tensor-wide maxima given: a band
    of a current-scaling or NVFP4 tensor is quantized with the whole tensor's
    amax, and a stochastic band with the counter offset of its first row
    (r0 * K / 16), so that it is exactly that band of the whole-tensor result.
    Returns (fields compared, bytes compared)."""
    from concurrent.futures import ThreadPoolExecutor

    threads = threads or os.cpu_count() or 1
    pool = ThreadPoolExecutor(max_workers=threads)
    stats = {"fields": 0, "bytes": 0}

    def host(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()

    def eq(a, b, what):
        a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
        if a.dtype == np.float32:
            a, b = a.view(np.uint32), b.view(np.uint32)
        if a.shape != b.shape or not np.array_equal(a, b):
            raise AssertionError(f"parity failed: {what}")
        stats["fields"] += 1
        stats["bytes"] += a.nbytes

    def bands(M):
        if full:
            return [(r0, min(r0 + PARITY_BAND_ROWS, M)) for r0 in range(0, M, PARITY_BAND_ROWS)]
        r0 = int(np.random.default_rng(seed + M).integers(0, M // 128)) * 128
        return [(r0, r0 + 128)]

    def all_bands(M):
        return [(r0, min(r0 + PARITY_BAND_ROWS, M)) for r0 in range(0, M, PARITY_BAND_ROWS)]

    def tensor_max(fn, x):
        """max over row bands of fn(band) (a non-negative FP32 value)."""
        return np.float32(max(pool.map(lambda b: np.float32(fn(np.ascontiguousarray(x[b[0]:b[1]]))),
                                       all_bands(x.shape[0]))))

    def over_bands(xh, work):
        """work(r0, r1, band) -> list of (gpu slice, oracle array, name); all compared."""
        def one(b):
            r0, r1 = b
            return work(r0, r1, np.ascontiguousarray(xh[r0:r1]))
        for res in pool.map(one, bands(xh.shape[0])):
            for g, w, what in res:
                eq(g, w, what)

    f32eq = lambda a, b, what: eq(np.float32(a), np.float32(b), what)
    for wl, tn, kind in [("cs1", "x", "cs_e4m3"), ("hy4", "grad", "cs_e5m2"), ("hy4", "grad", "ds_e5m2"),
                         ("hy4", "w", "cs_e4m3"),
                         ("mx2", "act", "mx"), ("bw3", "act", "bw1"), ("bw3", "w", "bw128"),
                         ("bw3", "act", "bwmx1"), ("bw3", "w", "bwmx128"),
                         ("nv5", "act", "nv_rn"), ("nv5", "grad", "nv_sr"), ("nv5", "w", "nv16"),
                         ("nv5", "act", "rht_rn"), ("nv5", "grad", "rht_sr"), ("nv5", "grad", "recipe_sr")]:
        if wl not in host_t:
            continue
        xh, xd = host_t[wl][tn], dev_t[wl][tn]
        M, K = xh.shape
        tag = f"{wl}.{tn} {kind}"
        out_bf16 = torch.bfloat16 if xd.dtype == torch.bfloat16 else torch.float32
        o_out = O.BF16 if out_bf16 == torch.bfloat16 else O.F32
        if kind.startswith("cs"):
            fmt = O.E5M2 if kind == "cs_e5m2" else O.E4M3
            sfmt = "e5m2" if fmt == O.E5M2 else "e4m3"
            A = tensor_max(O.amax, xh)
            g = Q.q_current_scaling(xd, sfmt, True, True)
            y = host(Q.dq_current_scaling(g.q_row, g.scale, sfmt, out_bf16))
            qr, qc = host(g.q_row), host(g.q_colT)
            f32eq(g.amax.item(), A, f"{tag} amax")
            _, s_want = O.cs_scale(A, fmt)
            f32eq(g.scale.item(), s_want, f"{tag} scale")
            over_bands(xh, lambda r0, r1, band: (
                lambda w: [(qr[r0:r1], w.q_row, f"{tag} q_row"), (qc[:, r0:r1], w.q_colT, f"{tag} q_colT"),
                           (y[r0:r1], O.dq_current_scaling(w.q_row, w.scale, fmt, o_out), f"{tag} dq")])(
                O.current_scaling(band, fmt, True, True, amax_in=A)))
        elif kind.startswith("ds"):
            # two steps from an empty window: step 0 casts with alpha = 1, step 1
            # with the alpha of step 0's recorded amax
            st = Q.DelayedScaling("e5m2", history_len=1024)
            hist = np.zeros(1024, np.float32)
            alpha = np.float32(1.0)
            for t in range(2):
                g = st.quantize(xd, True, True)
                qr, qc = host(g.q_row), host(g.q_colT)

                def work(r0, r1, band, alpha=alpha, qr=qr, qc=qc, t=t):
                    w_row, w_colT, _ = O.ds_cast(band, alpha, O.E5M2, rowwise=True, colwise=True)
                    return [(qr[r0:r1], w_row, f"{tag} step {t} q_row"), (qc[:, r0:r1], w_colT, f"{tag} step {t} q_colT")]
                over_bands(xh, work)
                A = tensor_max(O.amax, xh)
                f32eq(g.amax.item(), A, f"{tag} step {t} amax")
                hist[t] = A
                alpha, s_next = O.ds_scale_update(hist, t, O.HIST_MAX, O.E5M2)
                eq(host(st.ds), np.array([alpha, s_next], np.float32), f"{tag} step {t} next scale")
        elif kind == "mx":
            g = Q.q_mxfp8(xd)
            rq = Q.q_mxfp8_requant_col(g.q_row, g.e8m0_row)
            yr = host(Q.dq_mxfp8(g.q_row, g.e8m0_row, "e4m3", Q.Q_ROW, torch.bfloat16))
            yc = host(Q.dq_mxfp8(g.q_col, g.e8m0_col, "e4m3", Q.Q_COL, torch.bfloat16))
            h = {k: host(getattr(g, k)) for k in ("q_row", "e8m0_row", "q_col", "e8m0_col")}
            rqq, rqe = host(rq.q_col), host(rq.e8m0_col)

            def work(r0, r1, band):
                w = O.mxfp8(band)
                wq, we = O.mxfp8_requant_col(w.q_row, w.e8m0_row)
                return [(h["q_row"][r0:r1], w.q_row, f"{tag} q_row"), (h["e8m0_row"][r0:r1], w.e8m0_row, f"{tag} e8m0_row"),
                        (h["q_col"][r0:r1], w.q_col, f"{tag} q_col"),
                        (h["e8m0_col"][r0 // 32:r1 // 32], w.e8m0_col, f"{tag} e8m0_col"),
                        (rqq[r0:r1], wq, f"{tag} requant q_col"), (rqe[r0 // 32:r1 // 32], we, f"{tag} requant e8m0_col"),
                        (yr[r0:r1], O.dq_mxfp8(w.q_row, w.e8m0_row, O.E4M3, O.ROW, O.BF16), f"{tag} dq row"),
                        (yc[r0:r1], O.dq_mxfp8(w.q_col, w.e8m0_col, O.E4M3, O.COL, O.BF16), f"{tag} dq col")]
            over_bands(xh, work)
        elif kind in ("bw1", "bw128"):
            tile, otile = ("1x128", O.T1x128) if kind == "bw1" else ("128x128", O.T128x128)
            g = Q.q_blockwise(xd, tile, True, True)
            y = host(Q.dq_blockwise(g.q_row, g.s_row, tile, torch.bfloat16))
            h = {k: host(getattr(g, k)) for k in ("q_row", "s_row", "q_colT", "s_colT")}

            def work(r0, r1, band):
                w = O.blockwise(band, otile, True, True)
                sr = h["s_row"][r0:r1] if kind == "bw1" else h["s_row"][r0 // 128:r1 // 128]
                return [(h["q_row"][r0:r1], w.q_row, f"{tag} q_row"), (sr, w.s_row, f"{tag} s_row"),
                        (h["q_colT"][:, r0:r1], w.q_colT, f"{tag} q_colT"),
                        (h["s_colT"][:, r0 // 128:r1 // 128], w.s_colT, f"{tag} s_colT"),
                        (y[r0:r1], O.dq_blockwise(w.q_row, w.s_row, otile, O.BF16), f"{tag} dq")]
            over_bands(xh, work)
        elif kind in ("bwmx1", "bwmx128"):
            tile, otile = ("1x128", O.T1x128) if kind == "bwmx1" else ("128x128", O.T128x128)
            g = Q.q_blockwise_mx(xd, tile, True, True)
            h = {k: host(getattr(g, k)) for k in ("q_row", "e8m0_row", "q_colT", "e8m0_colT")}

            def work(r0, r1, band):
                w = O.blockwise_mx(band, otile, True, True)
                return [(h["q_row"][r0:r1], w.q_row, f"{tag} q_row"), (h["e8m0_row"][r0:r1], w.e8m0_row, f"{tag} e8m0_row"),
                        (h["q_colT"][:, r0:r1], w.q_colT, f"{tag} q_colT"),
                        (h["e8m0_colT"][:, r0 // 32:r1 // 32], w.e8m0_colT, f"{tag} e8m0_colT")]
            over_bands(xh, work)
        elif kind.startswith("nv"):
            blk = O.B16x16 if kind == "nv16" else O.B1x16
            rnd = O.SR if kind == "nv_sr" else O.RN
            sd = 4 if rnd == O.SR else 0
            A = tensor_max(O.amax, xh)
            g = Q.q_nvfp4(xd, "16x16" if blk == O.B16x16 else "1x16", "sr" if rnd == O.SR else "rn", sd, 0, True, True)
            y = host(Q.dq_nvfp4(g.q_row, g.sb_row, g.s_global, "16x16" if blk == O.B16x16 else "1x16", torch.bfloat16))
            h = {k: host(getattr(g, k)) for k in ("q_row", "sb_row", "q_colT", "sb_colT")}
            f32eq(g.amax.item(), A, f"{tag} amax")
            f32eq(g.s_global.item(), O.nvfp4_global(A)[1], f"{tag} s_global")

            def work(r0, r1, band):
                w = O.nvfp4(band, blk, rnd, seed=sd, offset=r0 * K // 16, rowwise=True, colwise=True, amax_in=A)
                sbr = h["sb_row"][r0:r1] if blk == O.B1x16 else h["sb_row"][r0 // 16:r1 // 16]
                return [(h["q_row"][r0:r1], w.q_row, f"{tag} q_row"), (sbr, w.sb_row, f"{tag} sb_row"),
                        (h["q_colT"][:, r0 // 2:r1 // 2], w.q_colT, f"{tag} q_colT"),
                        (h["sb_colT"][:, r0 // 16:r1 // 16], w.sb_colT, f"{tag} sb_colT"),
                        (y[r0:r1], O.dq_nvfp4(w.q_row, w.sb_row, w.s_global, blk, O.BF16), f"{tag} dq")]
            over_bands(xh, work)
        elif kind.startswith("rht"):
            rnd = O.SR if kind == "rht_sr" else O.RN
            sd = 4 if rnd == O.SR else 0
            A = tensor_max(lambda b: O.amax(O.rht_cols(b, RHT_MASK)), xh)
            g = Q.q_nvfp4_rht_colT(xd, RHT_MASK, "sr" if rnd == O.SR else "rn", sd, 0)
            qc, sc = host(g.q_colT), host(g.sb_colT)
            f32eq(g.amax.item(), A, f"{tag} amax")
            f32eq(g.s_global.item(), O.nvfp4_global(A)[1], f"{tag} s_global")

            def work(r0, r1, band):
                q, sb, _, _ = O.nvfp4_rht_colT(band, RHT_MASK, rnd, seed=sd, offset=r0 * K // 16, amax_in=A)
                return [(qc[:, r0 // 2:r1 // 2], q, f"{tag} q_colT"), (sc[:, r0 // 16:r1 // 16], sb, f"{tag} sb_colT")]
            over_bands(xh, work)
        elif kind == "recipe_sr":
            A_x = tensor_max(O.amax, xh)
            A_r = tensor_max(lambda b: O.amax(O.rht_cols(b, RHT_MASK)), xh)
            row, col = Q.q_nvfp4_recipe(xd, RHT_MASK, "sr", 4, 0)
            f32eq(row.amax.item(), A_x, f"{tag} amax_row")
            f32eq(col.amax.item(), A_r, f"{tag} amax_colT")
            f32eq(row.s_global.item(), O.nvfp4_global(A_x)[1], f"{tag} s_global_row")
            f32eq(col.s_global.item(), O.nvfp4_global(A_r)[1], f"{tag} s_global_colT")
            qr, sr, qc, sc = host(row.q_row), host(row.sb_row), host(col.q_colT), host(col.sb_colT)

            def work(r0, r1, band):
                w = O.nvfp4(band, O.B1x16, O.SR, seed=4, offset=r0 * K // 16, rowwise=True, colwise=False, amax_in=A_x)
                q, sb, _, _ = O.nvfp4_rht_colT(band, RHT_MASK, O.SR, seed=4, offset=r0 * K // 16, amax_in=A_r)
                return [(qr[r0:r1], w.q_row, f"{tag} q_row"), (sr[r0:r1], w.sb_row, f"{tag} sb_row"),
                        (qc[:, r0 // 2:r1 // 2], q, f"{tag} q_colT"), (sc[:, r0 // 16:r1 // 16], sb, f"{tag} sb_colT")]
            over_bands(xh, work)
    if torch.cuda.is_available():
        torch.cuda.synchronize()
    pool.shutdown()
    return stats["fields"], stats["bytes"]


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# ours
# --------------------------------------------------------------------------

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def run_ours(args):
    import torch
    import torch.distributed as dist

    import nvfp4_quantization_current_gb300 as Q

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Q.lib()

    # ---- inputs: host (numpy, for the oracle checks and the end-to-end copies) and device
    host_t, dev_t, pinned = {}, {}, {}
    wanted = [wl for wl in WL.WORKLOADS if not args.only or args.only.split(".")[0] in wl]
    for wl in wanted:
        host_t[wl] = WL.workload(wl, args.scale_rows)
        dev_t[wl], pinned[wl] = {}, {}
        for tn, a in host_t[wl].items():
            t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
            pinned[wl][tn] = t.pin_memory()
            dev_t[wl][tn] = t.to(dev)
    torch.cuda.synchronize()

    parity = "not run"
    if not args.skip_parity and not args.only:
        import oracle as O
        t_par = time.perf_counter()
        fields, nbytes_cmp = parity_check(host_t, dev_t, torch, Q, O, full=not args.sampled_parity)
        what = "every output of every call on the full-size tensors" if not args.sampled_parity else \
            "one 128-row band per tensor"
        parity = (f"0-ULP: {what} ({nbytes_cmp / 1e9:.2f} GB compared in {fields} band fields, "
                  f"oracle on {os.cpu_count()} host threads, {time.perf_counter() - t_par:.0f} s)")

    calls = [c for c in build_step(dev_t, torch, Q) if args.only in c.name]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # A bounded GPU-side delay at the start of each step (outside every timed
    # event pair) lets the host queue the whole step ahead of the device, so
    # that no call's events include host submission latency.
    head_start = int(2e-3 * 2.0e9)

    def one_step(evs, per_kernel):
        """One pass over every call.  per_kernel False (the step): one event
        pair around each call, so the kernels of a call overlap as they do for
        a caller (programmatic dependent launch); True (the breakdown): an
        event after every kernel of a call, which serializes them."""
        torch.cuda._sleep(head_start)
        for ci, c in enumerate(calls):
            flush.fill_(float(ci))
            torch.sum(clean, dim=0, out=sink)   # clean lines replace the dirty ones
            evs[ci][0].record(stream)
            for pi, p in enumerate(c.pieces):
                p[3]()
                if per_kernel:
                    evs[ci][pi + 1].record(stream)
            if not per_kernel:
                evs[ci][1].record(stream)

    def new_events(per_kernel):
        return [[torch.cuda.Event(enable_timing=True) for _ in range((len(c.pieces) if per_kernel else 1) + 1)]
                for c in calls]

    for w in range(args.warmup):
        one_step(new_events(w % 2 == 1), w % 2 == 1)
        if w == 0:   # the producers' outputs exist now: fill the consumers' own inputs
            for c in calls:
                if c.prime is not None:
                    c.prime()
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)

    def timed(per_kernel):
        """K steps between a barrier + synchronize on both sides, with the SM
        clocks sampled meanwhile; returns (events, wall seconds, clocks)."""
        all_evs = [new_events(per_kernel) for _ in range(args.steps)]
        sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
        sampler.start()
        time.sleep(0.3)
        # no collector pass while the host queues the steps: a pause that
        # outlasts the queued work would leave the device idle inside a call
        gc.collect()
        gc_on = gc.isenabled()
        gc.disable()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(args.steps):
            one_step(all_evs[s], per_kernel)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if gc_on:
            gc.enable()
        if world > 1:
            dist.barrier()
        return all_evs, wall, sampler.stop()

    # the step: K steps timed call by call
    step_evs, wall, clocks = timed(False)
    call_ms = {ci: [step_evs[s][ci][0].elapsed_time(step_evs[s][ci][1]) for s in range(args.steps)]
               for ci in range(len(calls))}
    step_ms = sum(statistics.mean(v) for v in call_ms.values())
    step_bytes = sum(c.alg_bytes for c in calls)
    if world > 1:
        t = torch.tensor([step_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    value = step_bytes * world / (step_ms * 1e-3) / 1e9

    # the breakdown: K more steps with an event after every kernel
    brk_evs, brk_wall, brk_clocks = timed(True)
    kern_ms = {}      # (call index, piece index) -> list of ms
    for s in range(args.steps):
        for ci, c in enumerate(calls):
            ev = brk_evs[s][ci]
            for pi in range(len(c.pieces)):
                kern_ms.setdefault((ci, pi), []).append(ev[pi].elapsed_time(ev[pi + 1]))
    # per-kernel time: the median over the K steps.  With an event after
    # every kernel, a host stall long enough to drain the queued work leaves
    # the device idle inside one event interval; the median keeps such a
    # step from moving a kernel's time (and the choice of the dominant one).
    kern_med = {key: statistics.median(v) for key, v in kern_ms.items()}

    peak, peak_kind = measured_peak()
    per_call = []
    per_recipe = {}
    per_kernel = {}
    for ci, c in enumerate(calls):
        ms = statistics.mean(call_ms[ci])
        gbs = c.alg_bytes / (ms * 1e-3) / 1e9
        per_call.append({"call": c.name, "us": round(ms * 1e3, 2), "bytes": c.alg_bytes, "GB/s": round(gbs, 1),
                         "frac": round(gbs / peak, 3),
                         "kernels": [[p[0], round(kern_med[(ci, pi)] * 1e3, 2)]
                                     for pi, p in enumerate(c.pieces)]})
        r = per_recipe.setdefault(c.recipe, {"bytes": 0, "us": 0.0})
        r["bytes"] += c.alg_bytes
        r["us"] += ms * 1e3
        for pi, p in enumerate(c.pieces):
            k = per_kernel.setdefault(p[0], {"src": p[1], "bytes": 0, "us": 0.0, "launches": 0})
            k["bytes"] += p[2]
            k["us"] += kern_med[(ci, pi)] * 1e3
            k["launches"] += 1
    for r in per_recipe.values():
        r["GB/s"] = round(r["bytes"] / (r["us"] * 1e-6) / 1e9, 1)
        r["frac"] = round(r["GB/s"] / peak, 3)
        r["us"] = round(r["us"], 2)
    # dominant kernel: the single launch with the longest (median) time in the step
    (dci, dpi) = max(kern_med, key=lambda key: kern_med[key])
    dcall, dpiece = calls[dci], calls[dci].pieces[dpi]
    dom_us = kern_med[(dci, dpi)] * 1e3
    dom_bytes = dpiece[2]
    achieved = dom_bytes / (dom_us * 1e-6) / 1e9
    key = f"{dcall.name.split()[0]}:{dpiece[0]}"
    tr = TRAFFIC.get(key)
    traffic = None
    if tr is not None and tr.get("src_hash") == src_hash(dpiece[1]):
        traffic = tr["bytes_per_launch"]
    roofline = {"bound": "alu" if dpiece[0].endswith("_sr") else "hbm", "kernel": dpiece[0], "call": dcall.name,
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 3), "traffic": traffic,
                "alg_bytes_per_launch": int(dom_bytes), "us_per_launch": round(dom_us, 2),
                "share_of_step": round(dom_us / (step_ms * 1e3), 3), "peak_kind": peak_kind + " hbm_gbs"}
    # q_amax, the delayed-scaling cast and the transform's amax launch two
    # kernels (zero the amax word, then the pass); every other call one
    n_launches = args.steps * sum((2 if p[0] in ("amax", "ds_cast_T", "rht_amax", "rht_amax2") else 1) for c in calls for p in c.pieces)

    # ---- end to end: pinned host input -> device, the public call, outputs -> pinned host
    e2e = None
    if not args.skip_e2e:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        dev_to_pin = {}
        for wl in host_t:
            for tn in host_t[wl]:
                dev_to_pin[id(dev_t[wl][tn])] = pinned[wl][tn]
        out_host = {}
        for c in calls:
            for t in c.d2h:
                if t is not None and id(t) not in out_host:
                    out_host[id(t)] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        in_host = {}
        for c in calls:
            for t in c.h2d:
                if t is not None and id(t) not in in_host:
                    in_host[id(t)] = dev_to_pin.get(id(t))
                    if in_host[id(t)] is None:
                        in_host[id(t)] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        h2d_unique = {id(t): t for c in calls for t in c.h2d if t is not None}
        h2d_b = sum(nbytes(t) for t in h2d_unique.values())   # each input uploads once per step
        d2h_b = sum(nbytes(t) for c in calls for t in c.d2h if t is not None)
        # Three streams: host->device copies, the public calls, device->host
        # copies; call i+1's inputs upload while call i computes and call i-1's
        # results download.  Each input tensor uploads once per step (two calls
        # on one tensor share the upload); each device tensor keeps the event
        # of its last use (compute reading it, or the download of it), and an
        # upload into it waits for that event; a call waits for the uploads of
        # its inputs and its download for the call.  One event pair spans the
        # whole step.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_cmp = stream
        e_ms = []
        for s in range(e2e_steps + 1):
            torch.cuda.synchronize()
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(s_cmp)
            s_in.wait_event(start)
            s_out.wait_event(start)
            last, up = {}, {}
            for c in calls:
                for t in c.h2d:
                    if id(t) in up:
                        continue
                    if id(t) in last:
                        s_in.wait_event(last[id(t)])
                    with torch.cuda.stream(s_in):
                        t.copy_(in_host[id(t)], non_blocking=True)
                    up[id(t)] = torch.cuda.Event()
                    up[id(t)].record(s_in)
                for t in c.h2d:
                    s_cmp.wait_event(up[id(t)])
                for t in c.d2h:
                    if t is not None and id(t) in last:
                        s_cmp.wait_event(last[id(t)])
                with torch.cuda.stream(s_cmp):
                    c.e2e_thunk()
                e_c = torch.cuda.Event()
                e_c.record(s_cmp)
                s_out.wait_event(e_c)
                with torch.cuda.stream(s_out):
                    for t in c.d2h:
                        if t is not None:
                            out_host[id(t)].copy_(t, non_blocking=True)
                e_o = torch.cuda.Event()
                e_o.record(s_out)
                for t in c.h2d:
                    last[id(t)] = e_c
                for t in c.d2h:
                    if t is not None:
                        last[id(t)] = e_o
            s_cmp.wait_event(e_o)
            end.record(s_cmp)
            end.synchronize()
            if s > 0:          # the first pass warms the copy engines
                e_ms.append(start.elapsed_time(end))
        ems = statistics.mean(e_ms)
        if world > 1:
            t = torch.tensor([ems], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ems = float(t.item())

        # The host link in the same run, with the same pinned buffers: every
        # input of the step up alone, every output down alone, and both at once
        # (on two streams), no kernels.  The end-to-end step is bounded below by
        # the longer one-way time; it can beat the both-at-once figure, which
        # saturates the link in both directions for the whole time.
        def link(up, down, reps=3):
            ms = []
            for r in range(reps + 1):
                torch.cuda.synchronize()
                start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                start.record(s_cmp)
                s_in.wait_event(start)
                s_out.wait_event(start)
                if up:
                    with torch.cuda.stream(s_in):
                        for t in h2d_unique.values():
                            t.copy_(in_host[id(t)], non_blocking=True)
                if down:
                    with torch.cuda.stream(s_out):
                        for c in calls:
                            for t in c.d2h:
                                if t is not None:
                                    out_host[id(t)].copy_(t, non_blocking=True)
                e_i, e_o = torch.cuda.Event(), torch.cuda.Event()
                e_i.record(s_in)
                e_o.record(s_out)
                s_cmp.wait_event(e_i)
                s_cmp.wait_event(e_o)
                end.record(s_cmp)
                end.synchronize()
                if r > 0:
                    ms.append(start.elapsed_time(end))
            b = (h2d_b if up else 0) + (d2h_b if down else 0)
            return round(b / (statistics.mean(ms) * 1e-3) / 1e9, 1), round(statistics.mean(ms), 3)

        (up_gbs, up_ms), (down_gbs, down_ms), (both_gbs, both_ms) = link(True, False), link(False, True), link(True, True)
        e2e = {"value": round(step_bytes * world / (ems * 1e-3) / 1e9, 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b, "ms_per_step": round(ems, 3),
               "ms_per_step_each": [round(v, 3) for v in e_ms],
               "steps": e2e_steps, "schedule": "uploads, calls and downloads on three streams, overlapped across calls",
               "host_link": {"h2d_GBps": up_gbs, "h2d_ms": up_ms, "d2h_GBps": down_gbs, "d2h_ms": down_ms,
                             "both_GBps": both_gbs, "both_ms": both_ms,
                             "what": "the step's own copies alone (pinned host buffers, no kernels) in the same "
                                     "run: all uploads, all downloads, and both issued at once on two streams; the "
                                     "longer one-way time bounds the end-to-end step from below"}}

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu and not args.only:
        cpu = cpu_baseline_all_cores(host_t)
        cpu["single_core"] = cpu_baseline(host_t)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy; see workloads.WORKLOADS)",
            "config": {"workload": "all five workloads at full size per step: cs1 FP32 1024x1024 CS-E4M3+T; "
                                   "mx2 BF16 8192x4096 MXFP8 row+col, row->col requant; bw3 BF16 16384x7168 1x128+T and 7168x18432 "
                                   "128x128+T, each also held as MXFP8 (power-of-two scales); hy4 BF16 8192x14336 CS-E5M2+T, "
                                   "delayed-scaling E5M2+T (window 1024, max) and 14336x4096 CS-E4M3+T; nv5 BF16 8192x4096 NVFP4 "
                                   "1x16 RN+T, 1x16 SR+T, 4096x4096 16x16 RN+T; each with a dequant; nv5 act/grad random-Hadamard "
                                   "NVFP4 colT (RN / SR); nv5 grad NVFP4 recipe (row SR + RHT colT SR, one amax pass)",
                       "l2": "flushed before every timed call (256 MiB write, then a 256 MiB read that evicts the dirty lines)",
                       "timing": "one CUDA event pair around each call on its stream (the kernels of a call overlap "
                                 "as they do for a caller); value = step bytes / sum of call times",
                       "scale_rows": args.scale_rows, "parallelism": f"replicas x{world} (independent tensors)"},
            "parity": parity,
            "roofline": roofline,
            "per_recipe": per_recipe,
            "per_kernel": {k: {"launches_per_step": v["launches"], "us_per_launch": round(v["us"] / v["launches"], 2),
                               "GB/s": round(v["bytes"] / (v["us"] * 1e-6) / 1e9, 1),
                               "frac": round(v["bytes"] / (v["us"] * 1e-6) / 1e9 / peak, 3),
                               "share_of_step": round(v["us"] / (step_ms * 1e3), 3)}
                           for k, v in sorted(per_kernel.items(), key=lambda kv: -kv[1]["us"])},
            "per_call": per_call,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": n_launches,
            "clocks": clocks,
            "breakdown": {"what": "per_kernel, per_call kernels and roofline: K more steps with a CUDA event after "
                                  "every kernel (which serializes the kernels of a call); each kernel's time is "
                                  "the median over the K steps",
                          "steps": args.steps, "clocks": brk_clocks, "wall_s_timed": round(brk_wall, 3)},
            "wall_s_timed": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# the CPU oracle on a bounded row sample
# --------------------------------------------------------------------------

def oracle_sample_work(host_t, frac):
    """(thunk, algorithmic bytes) pairs over the first `frac` of the rows of
    every tensor (rows rounded to a multiple of 128), same recipes as a step."""
    import oracle as O
    work = []

    def rows(a):
        return max(128, int(a.shape[0] * frac) // 128 * 128)

    def isz(a):
        return a.dtype.itemsize

    def cs(a, fmt):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        work.append((lambda: O.current_scaling(s, fmt, True, True), 2 * s.nbytes + 2 * M * K + 4))
        r = O.current_scaling(s, fmt, True, False)
        work.append((lambda: O.dq_current_scaling(r.q_row, r.scale, fmt, O.BF16 if a.dtype == np.uint16 else O.F32),
                     M * K + M * K * isz(a) + 4))

    def ds(a, fmt):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        alpha, _ = O.ds_scale_update(np.array([O.amax(a)], np.float32), 0, O.HIST_MAX, fmt)
        hist = np.zeros(1024, np.float32)
        work.append((lambda: O.ds_cast(s, alpha, fmt, True, True), s.nbytes + 2 * M * K + 16))
        work.append((lambda: O.ds_scale_update(hist, 0, O.HIST_MAX, fmt), hist.nbytes + 8))

    def rht(a, rnd, seed):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        work.append((lambda: O.nvfp4_rht_colT(s, RHT_MASK, rnd, seed=seed), 2 * s.nbytes + M * K // 2 + M * K // 16 + 4))

    def mx(a):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        work.append((lambda: O.mxfp8(s), s.nbytes + 2 * M * K + M * K // 16))
        r = O.mxfp8(s)
        work.append((lambda: O.mxfp8_requant_col(r.q_row, r.e8m0_row), 2 * M * K + M * K // 16))
        work.append((lambda: O.dq_mxfp8(r.q_row, r.e8m0_row, O.E4M3, O.ROW, O.BF16), M * K * 3 + M * K // 32))
        work.append((lambda: O.dq_mxfp8(r.q_col, r.e8m0_col, O.E4M3, O.COL, O.BF16), M * K * 3 + M * K // 32))

    def bw(a, tile):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        sc = (M * K // 128) * 4 if tile == O.T1x128 else (M * K // 16384) * 4
        work.append((lambda: O.blockwise(s, tile, True, True), s.nbytes + 2 * M * K + 2 * sc))
        r = O.blockwise(s, tile, True, False)
        work.append((lambda: O.dq_blockwise(r.q_row, r.s_row, tile, O.BF16), M * K * 3 + sc))

    def bwmx(a, tile):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        work.append((lambda: O.blockwise_mx(s, tile, True, True), s.nbytes + 2 * M * K + 2 * (M * K // 32)))

    def nv(a, blk, rnd, seed):
        s = np.ascontiguousarray(a[:rows(a)])
        M, K = s.shape
        sb = M * K // 16 if blk == O.B1x16 else M * K // 256
        work.append((lambda: O.nvfp4(s, blk, rnd, seed=seed, rowwise=True, colwise=True), 2 * s.nbytes + M * K + 2 * sb + 4))
        r = O.nvfp4(s, blk, rnd, seed=seed)
        work.append((lambda: O.dq_nvfp4(r.q_row, r.sb_row, r.s_global, blk, O.BF16), M * K // 2 + sb + 2 * M * K + 4))

    cs(host_t["cs1"]["x"], O.E4M3)
    mx(host_t["mx2"]["act"])
    bw(host_t["bw3"]["act"], O.T1x128)
    bw(host_t["bw3"]["w"], O.T128x128)
    bwmx(host_t["bw3"]["act"], O.T1x128)
    bwmx(host_t["bw3"]["w"], O.T128x128)
    cs(host_t["hy4"]["grad"], O.E5M2)
    ds(host_t["hy4"]["grad"], O.E5M2)
    cs(host_t["hy4"]["w"], O.E4M3)
    nv(host_t["nv5"]["act"], O.B1x16, O.RN, 0)
    nv(host_t["nv5"]["grad"], O.B1x16, O.SR, 4)
    nv(host_t["nv5"]["w"], O.B16x16, O.RN, 0)
    rht(host_t["nv5"]["act"], O.RN, 0)
    rht(host_t["nv5"]["grad"], O.SR, 4)
    nv_rows = np.ascontiguousarray(host_t["nv5"]["grad"][:rows(host_t["nv5"]["grad"])])
    Mr, Kr = nv_rows.shape
    work.append((lambda: (O.amax(nv_rows), O.amax(O.rht_cols(nv_rows, RHT_MASK))), nv_rows.nbytes))
    work.append((lambda: O.nvfp4(nv_rows, O.B1x16, O.SR, seed=4, rowwise=True, colwise=False),
                 nv_rows.nbytes + Mr * Kr // 2 + Mr * Kr // 16 + 4))
    work.append((lambda: O.nvfp4_rht_colT(nv_rows, RHT_MASK, O.SR, seed=4), nv_rows.nbytes + Mr * Kr // 2 + Mr * Kr // 16 + 4))
    return work


def oracle_band_work(host_t, frac, nbands):
    """The recipes of a step on the first `frac` of every tensor's rows (a
    multiple of 128), as a list of (phase list, algorithmic bytes): each phase
    is a list of independent band thunks (row bands of 128-row multiples) to
    run in parallel, and a recipe's phases run in order -- first the band
    maxima of a tensor-wide amax, then the band casts given that amax (and
    the counter offset of the band's first row), as a row-sharded call does.
    The oracle functions are the plain, unmodified ones."""
    import oracle as O

    def rows(a):
        return max(128, int(a.shape[0] * frac) // 128 * 128)

    def split(M):
        step = max(128, (M // nbands + 127) // 128 * 128)
        return [(r0, min(r0 + step, M)) for r0 in range(0, M, step)]

    work = []

    def bands_of(a):
        s_ = np.ascontiguousarray(a[:rows(a)])
        return s_, [(r0, r1, np.ascontiguousarray(s_[r0:r1])) for r0, r1 in split(s_.shape[0])]

    class Max:
        """A tensor-wide maximum filled by the first phase."""
        def __init__(self, n):
            self.v = [np.float32(0)] * n

        def put(self, i, v):
            self.v[i] = np.float32(v)

        def get(self):
            return np.float32(max(self.v))

    def cs(a, fmt):
        s_, bs = bands_of(a)
        M, K = s_.shape
        A = Max(len(bs))
        work.append(([[lambda i=i, b=b: A.put(i, O.amax(b[2])) for i, b in enumerate(bs)],
                      [lambda b=b: O.current_scaling(b[2], fmt, True, True, amax_in=A.get()) for b in bs]],
                     2 * s_.nbytes + 2 * M * K + 4))
        r = O.current_scaling(s_, fmt, True, False)
        out = O.BF16 if a.dtype == np.uint16 else O.F32
        work.append(([[lambda r0=r0, r1=r1: O.dq_current_scaling(r.q_row[r0:r1], r.scale, fmt, out) for r0, r1, _ in bs]],
                     M * K + M * K * a.dtype.itemsize + 4))

    def ds(a, fmt):
        s_, bs = bands_of(a)
        M, K = s_.shape
        alpha, _ = O.ds_scale_update(np.array([O.amax(a)], np.float32), 0, O.HIST_MAX, fmt)
        hist = np.zeros(1024, np.float32)
        work.append(([[lambda b=b: O.ds_cast(b[2], alpha, fmt, True, True) for b in bs]], s_.nbytes + 2 * M * K + 16))
        work.append(([[lambda: O.ds_scale_update(hist, 0, O.HIST_MAX, fmt)]], hist.nbytes + 8))

    def mx(a):
        s_, bs = bands_of(a)
        M, K = s_.shape
        work.append(([[lambda b=b: O.mxfp8(b[2]) for b in bs]], s_.nbytes + 2 * M * K + M * K // 16))
        r = O.mxfp8(s_)
        work.append(([[lambda r0=r0, r1=r1: O.mxfp8_requant_col(r.q_row[r0:r1], r.e8m0_row[r0:r1]) for r0, r1, _ in bs]],
                     2 * M * K + M * K // 16))
        work.append(([[lambda r0=r0, r1=r1: O.dq_mxfp8(r.q_row[r0:r1], r.e8m0_row[r0:r1], O.E4M3, O.ROW, O.BF16)
                       for r0, r1, _ in bs]], M * K * 3 + M * K // 32))
        work.append(([[lambda r0=r0, r1=r1: O.dq_mxfp8(r.q_col[r0:r1], r.e8m0_col[r0 // 32:r1 // 32], O.E4M3, O.COL, O.BF16)
                       for r0, r1, _ in bs]], M * K * 3 + M * K // 32))

    def bw(a, tile):
        s_, bs = bands_of(a)
        M, K = s_.shape
        sc = (M * K // 128) * 4 if tile == O.T1x128 else (M * K // 16384) * 4
        work.append(([[lambda b=b: O.blockwise(b[2], tile, True, True) for b in bs]], s_.nbytes + 2 * M * K + 2 * sc))
        r = O.blockwise(s_, tile, True, False)
        srow = (lambda r0, r1: r.s_row[r0:r1]) if tile == O.T1x128 else (lambda r0, r1: r.s_row[r0 // 128:r1 // 128])
        work.append(([[lambda r0=r0, r1=r1: O.dq_blockwise(r.q_row[r0:r1], srow(r0, r1), tile, O.BF16) for r0, r1, _ in bs]],
                     M * K * 3 + sc))

    def bwmx(a, tile):
        s_, bs = bands_of(a)
        M, K = s_.shape
        work.append(([[lambda b=b: O.blockwise_mx(b[2], tile, True, True) for b in bs]], s_.nbytes + 2 * M * K + 2 * (M * K // 32)))

    def nv(a, blk, rnd, seed):
        s_, bs = bands_of(a)
        M, K = s_.shape
        A = Max(len(bs))
        sb = M * K // 16 if blk == O.B1x16 else M * K // 256
        work.append(([[lambda i=i, b=b: A.put(i, O.amax(b[2])) for i, b in enumerate(bs)],
                      [lambda b=b: O.nvfp4(b[2], blk, rnd, seed=seed, offset=b[0] * K // 16, rowwise=True, colwise=True,
                                           amax_in=A.get()) for b in bs]],
                     2 * s_.nbytes + M * K + 2 * sb + 4))
        r = O.nvfp4(s_, blk, rnd, seed=seed)
        sbr = (lambda r0, r1: r.sb_row[r0:r1]) if blk == O.B1x16 else (lambda r0, r1: r.sb_row[r0 // 16:r1 // 16])
        work.append(([[lambda r0=r0, r1=r1: O.dq_nvfp4(r.q_row[r0:r1], sbr(r0, r1), r.s_global, blk, O.BF16)
                       for r0, r1, _ in bs]], M * K // 2 + sb + 2 * M * K + 4))

    def rht(a, rnd, seed, row_copy=False):
        s_, bs = bands_of(a)
        M, K = s_.shape
        Ar, Ax = Max(len(bs)), Max(len(bs))

        def maxima(i, b):
            Ar.put(i, O.amax(O.rht_cols(b[2], RHT_MASK)))
            if row_copy:
                Ax.put(i, O.amax(b[2]))
        phases = [[lambda i=i, b=b: maxima(i, b) for i, b in enumerate(bs)]]
        if row_copy:
            phases.append([lambda b=b: O.nvfp4(b[2], O.B1x16, rnd, seed=seed, offset=b[0] * K // 16, rowwise=True,
                                               colwise=False, amax_in=Ax.get()) for b in bs])
        phases.append([lambda b=b: O.nvfp4_rht_colT(b[2], RHT_MASK, rnd, seed=seed, offset=b[0] * K // 16,
                                                     amax_in=Ar.get()) for b in bs])
        copies = (2 if row_copy else 1) * (M * K // 2 + M * K // 16 + 4)
        work.append((phases, (3 if row_copy else 2) * s_.nbytes + copies))

    cs(host_t["cs1"]["x"], O.E4M3)
    mx(host_t["mx2"]["act"])
    bw(host_t["bw3"]["act"], O.T1x128)
    bw(host_t["bw3"]["w"], O.T128x128)
    bwmx(host_t["bw3"]["act"], O.T1x128)
    bwmx(host_t["bw3"]["w"], O.T128x128)
    cs(host_t["hy4"]["grad"], O.E5M2)
    ds(host_t["hy4"]["grad"], O.E5M2)
    cs(host_t["hy4"]["w"], O.E4M3)
    nv(host_t["nv5"]["act"], O.B1x16, O.RN, 0)
    nv(host_t["nv5"]["grad"], O.B1x16, O.SR, 4)
    nv(host_t["nv5"]["w"], O.B16x16, O.RN, 0)
    rht(host_t["nv5"]["act"], O.RN, 0)
    rht(host_t["nv5"]["grad"], O.SR, 4)
    rht(host_t["nv5"]["grad"], O.SR, 4, row_copy=True)
    return work


def run_band_work(work, threads):
    """Runs the phases of every recipe in order, the bands of a phase on the
    pool; returns (seconds, algorithmic bytes)."""
    from concurrent.futures import ThreadPoolExecutor
    total = sum(b for _, b in work)
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        for phases, _ in work:
            for phase in phases:
                for f in [pool.submit(fn) for fn in phase]:
                    f.result()
        return time.perf_counter() - t0, total


def cpu_baseline_all_cores(host_t, frac=1.0):
    threads = os.cpu_count() or 1
    work = oracle_band_work(host_t, frac, threads)
    dt, total = run_band_work(work, threads)
    return {"value": round(total / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {frac:.3f} of the rows of every tensor of the step, all recipes and dequants; the "
                      f"unmodified C oracle on {threads} host threads over row bands (tensor-wide maxima computed "
                      f"first, then given); {total / 1e9:.3f} GB in {dt:.1f} s",
            "seconds": round(dt, 2)}


def cpu_baseline(host_t, frac=CPU_SAMPLE_FRAC):
    work = oracle_sample_work(host_t, frac)
    t0 = time.perf_counter()
    total = 0
    for fn, b in work:
        fn()
        total += b
    dt = time.perf_counter() - t0
    return {"value": round(total / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {frac:.3f} of the rows (multiple of 128) of every tensor of the step, all recipes "
                      f"and dequants, single-threaded C oracle; {total / 1e9:.3f} GB in {dt:.1f} s",
            "seconds": round(dt, 2)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    host_t = {wl: WL.workload(wl, args.scale_rows) for wl in WL.WORKLOADS}
    import oracle as O
    O.build()
    threads = os.cpu_count() or 1
    # each step is a bounded row sample, sized so that warm-up + steps take
    # about REF_BUDGET_S seconds (never less than 128 rows of every tensor)
    t_small, _ = run_band_work(oracle_band_work(host_t, 0.0, threads), threads)
    budget = REF_BUDGET_S / max(1, args.steps + args.warmup)
    frac = min(1.0, max(0.0, budget / max(t_small, 1e-6)) * min(
        128 / a.shape[0] for d in host_t.values() for a in d.values()))
    work = oracle_band_work(host_t, frac, threads)
    for _ in range(args.warmup):
        run_band_work(work, threads)
    times, total = [], sum(b for _, b in work)
    for _ in range(args.steps):
        dt, _ = run_band_work(work, threads)
        times.append(dt)
    ms = statistics.mean(times) * 1e3
    value = total / (ms * 1e-3) / 1e9
    sample = (f"first {frac:.4f} of the rows (multiple of 128) of every tensor of the step, all recipes and "
              f"dequants; the unmodified C oracle on {threads} host threads over row bands")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy)",
        "config": {"workload": "same five workloads as the library arm, bounded row sample per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--skip-parity", action="store_true", help="skip the oracle check of the full-size outputs")
    ap.add_argument("--sampled-parity", action="store_true",
                    help="check one 128-row band per tensor instead of every output byte")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--scale-rows", type=float, default=1.0, help="shrink every tensor's rows (debug only)")
    ap.add_argument("--only", default="", help="time only the calls whose name contains this text (profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
