"""The N > 1 path on CPU: two gloo ranks each hold a row shard, agree on the
amax through the library's MAX all-reduce helper, quantize their shard with
the CPU oracle, and the gathered codes must equal the unsharded oracle
result bit for bit (per-tensor current scaling, NVFP4 with round-to-nearest
and with stochastic rounding (each rank's counter offset moved to its first
global row), two steps of delayed scaling with all-reduced window slots, and
the random-Hadamard NVFP4 columnwise copy with the all-reduced amax of the
transform)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        import workloads as W
        from nvfp4_quantization_current_gb300.distributed import allreduce_amax_, shard_row_base, sr_offset

        x = W.gen("outliers", (256, 96), 17, bf16=True)
        cut = [0, 64, 256]                                  # uneven shards on 16-row boundaries
        shard = np.ascontiguousarray(x[cut[rank]:cut[rank + 1]])
        a = torch.tensor([O.amax(shard)], dtype=torch.float32)
        allreduce_amax_(a)
        glob = float(a.item())
        cs = O.current_scaling(shard, O.E5M2, rowwise=True, colwise=True, amax_in=glob)
        nv = O.nvfp4(shard, O.B1x16, O.RN, rowwise=True, colwise=True, amax_in=glob)
        # delayed scaling: the window slot of each step is all-reduced before the update
        hist = np.zeros(4, np.float32)
        alpha = np.float32(1.0)
        ds = []
        for t, sc in enumerate([1.0, 0.25]):
            xs = O.bf16_round((W.bf16_bits_to_f32(shard) * np.float32(sc)).astype(np.float32))
            q_row, q_colT, a_loc = O.ds_cast(xs, alpha, O.E4M3, rowwise=True, colwise=True)
            slot = torch.tensor([a_loc], dtype=torch.float32)
            allreduce_amax_(slot)
            hist[t] = slot.item()
            alpha, _ = O.ds_scale_update(hist, t)
            ds += [q_row, q_colT]
        # random-Hadamard NVFP4 colT: the amax of the transformed shard is all-reduced
        mask = 0x6B1D
        ra = torch.tensor([O.amax(O.rht_cols(shard, mask))], dtype=torch.float32)
        allreduce_amax_(ra)
        rq, rsb, _, rsg = O.nvfp4_rht_colT(shard, mask, O.RN, amax_in=float(ra.item()))
        # stochastic rounding: each rank moves the unsharded call's counter
        # offset by its first global row, so its draws are the whole tensor's
        r0 = shard_row_base(shard.shape[0])
        assert r0 == cut[rank]
        off = sr_offset(77, r0, shard.shape[1])
        sr1 = O.nvfp4(shard, O.B1x16, O.SR, seed=9, offset=off, rowwise=True, colwise=True, amax_in=glob)
        sr2 = O.nvfp4(shard, O.B16x16, O.SR, seed=9, offset=off, rowwise=True, colwise=True, amax_in=glob)
        srq, srsb, _, _ = O.nvfp4_rht_colT(shard, mask, O.SR, seed=9, offset=off, amax_in=float(ra.item()))
        np.savez(os.path.join(result_dir, f"r{rank}.npz"), amax=np.float32(glob), cs_row=cs.q_row, cs_colT=cs.q_colT,
                 cs_s=cs.scale, nv_row=nv.q_row, nv_sb=nv.sb_row, nv_colT=nv.q_colT, nv_sbT=nv.sb_colT,
                 nv_sg=nv.s_global, ds0_row=ds[0], ds0_colT=ds[1], ds1_row=ds[2], ds1_colT=ds[3],
                 rht_q=rq, rht_sb=rsb, rht_sg=np.float32(rsg), sr1_row=sr1.q_row, sr1_colT=sr1.q_colT,
                 sr2_row=sr2.q_row, sr2_colT=sr2.q_colT, srrht_q=srq, srrht_sb=srsb)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_amax_allreduce_matches_unsharded(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    import oracle as O
    import workloads as W

    x = W.gen("outliers", (256, 96), 17, bf16=True)
    r = [np.load(os.path.join(tmp_path, f"r{i}.npz")) for i in range(world)]
    assert r[0]["amax"] == r[1]["amax"] == np.float32(O.amax(x))
    whole = O.current_scaling(x, O.E5M2, rowwise=True, colwise=True)
    assert np.array_equal(np.concatenate([q["cs_row"] for q in r]), whole.q_row)
    assert np.array_equal(np.concatenate([q["cs_colT"] for q in r], axis=1), whole.q_colT)
    assert r[0]["cs_s"] == r[1]["cs_s"] == whole.scale
    nv = O.nvfp4(x, O.B1x16, O.RN, rowwise=True, colwise=True)
    assert np.array_equal(np.concatenate([q["nv_row"] for q in r]), nv.q_row)
    assert np.array_equal(np.concatenate([q["nv_sb"] for q in r]), nv.sb_row)
    assert np.array_equal(np.concatenate([q["nv_colT"] for q in r], axis=1), nv.q_colT)
    assert np.array_equal(np.concatenate([q["nv_sbT"] for q in r], axis=1), nv.sb_colT)
    assert r[0]["nv_sg"] == nv.s_global
    # delayed scaling, unsharded: the same two steps
    hist = np.zeros(4, np.float32)
    alpha = np.float32(1.0)
    for t, sc in enumerate([1.0, 0.25]):
        xs = O.bf16_round((W.bf16_bits_to_f32(x) * np.float32(sc)).astype(np.float32))
        q_row, q_colT, a = O.ds_cast(xs, alpha, O.E4M3, rowwise=True, colwise=True)
        assert np.array_equal(np.concatenate([q[f"ds{t}_row"] for q in r]), q_row), t
        assert np.array_equal(np.concatenate([q[f"ds{t}_colT"] for q in r], axis=1), q_colT), t
        hist[t] = a
        alpha, _ = O.ds_scale_update(hist, t)
    # random-Hadamard NVFP4 colT, unsharded
    rq, rsb, _, rsg = O.nvfp4_rht_colT(x, 0x6B1D, O.RN)
    assert np.array_equal(np.concatenate([q["rht_q"] for q in r], axis=1), rq)
    assert np.array_equal(np.concatenate([q["rht_sb"] for q in r], axis=1), rsb)
    assert r[0]["rht_sg"] == r[1]["rht_sg"] == rsg
    # stochastic rounding: the gathered shards equal the unsharded call (seed 9, offset 77)
    for blk, key in ((O.B1x16, "sr1"), (O.B16x16, "sr2")):
        w = O.nvfp4(x, blk, O.SR, seed=9, offset=77, rowwise=True, colwise=True)
        assert np.array_equal(np.concatenate([q[f"{key}_row"] for q in r]), w.q_row), key
        assert np.array_equal(np.concatenate([q[f"{key}_colT"] for q in r], axis=1), w.q_colT), key
    sq, ssb, _, _ = O.nvfp4_rht_colT(x, 0x6B1D, O.SR, seed=9, offset=77)
    assert np.array_equal(np.concatenate([q["srrht_q"] for q in r], axis=1), sq)
    assert np.array_equal(np.concatenate([q["srrht_sb"] for q in r], axis=1), ssb)


def test_allreduce_amax_single_process_is_identity():
    from nvfp4_quantization_current_gb300.distributed import allreduce_amax_
    a = torch.tensor([3.5])
    assert allreduce_amax_(a).item() == 3.5
    with pytest.raises(ValueError):
        allreduce_amax_(torch.tensor([1.0, 2.0]))


def test_sr_offset_counts_sixteen_draws_per_philox_block():
    """A shard at global row r0 moves the counter offset by the r0*K draws
    ahead of it, 16 per Philox block; rows that split a 16-row block (or a K
    that splits a 1x16 block) have no such offset."""
    from nvfp4_quantization_current_gb300.distributed import sr_offset
    assert sr_offset(5, 0, 64) == 5
    assert sr_offset(5, 32, 64) == 5 + 32 * 64 // 16
    assert sr_offset(0, 8192, 4096) == 8192 * 4096 // 16
    for r0, K in ((8, 64), (24, 64), (16, 40)):
        with pytest.raises(ValueError):
            sr_offset(0, r0, K)


def _gather_worker(rank, world, port, result_dir):
    """Each rank quantizes its row shard (uneven: 128 and 256 rows, on 128-row
    boundaries) with the CPU oracle, wraps the outputs in the library's
    result classes and all-gathers them with ``all_gather_quantized``."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        import workloads as W
        import nvfp4_quantization_current_gb300 as Q
        from nvfp4_quantization_current_gb300.distributed import all_gather_quantized, allreduce_amax_

        x = W.gen("outliers", (384, 256), 23, bf16=True)
        cut = [0, 128, 384]
        shard = np.ascontiguousarray(x[cut[rank]:cut[rank + 1]])
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a))
        a = torch.tensor([O.amax(shard)], dtype=torch.float32)
        allreduce_amax_(a)
        glob = float(a.item())
        cs = O.current_scaling(shard, O.E4M3, rowwise=True, colwise=True, amax_in=glob)
        mx = O.mxfp8(shard, O.E5M2)
        bw1 = O.blockwise(shard, O.T1x128, rowwise=True, colwise=True)
        bw2 = O.blockwise(shard, O.T128x128, rowwise=True, colwise=True)
        nv1 = O.nvfp4(shard, O.B1x16, O.RN, rowwise=True, colwise=True, amax_in=glob)
        nv2 = O.nvfp4(shard, O.B16x16, O.RN, rowwise=True, colwise=True, amax_in=glob)
        got = {
            "cs": all_gather_quantized(Q.CurrentScalingTensor(t(cs.q_row), t(cs.q_colT), a.clone(),
                                                              torch.tensor([cs.scale]), Q.Q_E4M3)),
            "mx": all_gather_quantized(Q.MXFP8Tensor(t(mx.q_row), t(mx.e8m0_row), t(mx.q_col), t(mx.e8m0_col),
                                                     Q.Q_E5M2)),
            "bw1": all_gather_quantized(Q.BlockwiseTensor(t(bw1.q_row), t(bw1.s_row), t(bw1.q_colT), t(bw1.s_colT),
                                                          Q.Q_T1x128)),
            "bw2": all_gather_quantized(Q.BlockwiseTensor(t(bw2.q_row), t(bw2.s_row), t(bw2.q_colT), t(bw2.s_colT),
                                                          Q.Q_T128x128)),
            "nv1": all_gather_quantized(Q.NVFP4Tensor(t(nv1.q_row), t(nv1.sb_row), t(nv1.q_colT), t(nv1.sb_colT),
                                                      a.clone(), torch.tensor([nv1.s_global]), Q.Q_B1x16)),
            "nv2": all_gather_quantized(Q.NVFP4Tensor(t(nv2.q_row), t(nv2.sb_row), t(nv2.q_colT), t(nv2.sb_colT),
                                                      a.clone(), torch.tensor([nv2.s_global]), Q.Q_B16x16)),
        }
        if rank == 0:
            flat = {}
            for k, v in got.items():
                for f in ("q_row", "q_colT", "q_col", "e8m0_row", "e8m0_col", "s_row", "s_colT", "sb_row", "sb_colT"):
                    if getattr(v, f, None) is not None:
                        flat[f"{k}.{f}"] = getattr(v, f).numpy()
            np.savez(os.path.join(result_dir, "gathered.npz"), **flat)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_all_gather_of_quantized_shards_matches_unsharded(tmp_path):
    world = 2
    mp.start_processes(_gather_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    import oracle as O
    import workloads as W

    x = W.gen("outliers", (384, 256), 23, bf16=True)
    g = np.load(os.path.join(tmp_path, "gathered.npz"))
    want = {
        "cs": O.current_scaling(x, O.E4M3, rowwise=True, colwise=True),
        "mx": O.mxfp8(x, O.E5M2),
        "bw1": O.blockwise(x, O.T1x128, rowwise=True, colwise=True),
        "bw2": O.blockwise(x, O.T128x128, rowwise=True, colwise=True),
        "nv1": O.nvfp4(x, O.B1x16, O.RN, rowwise=True, colwise=True),
        "nv2": O.nvfp4(x, O.B16x16, O.RN, rowwise=True, colwise=True),
    }
    n = 0
    for key in g.files:
        rec, field = key.split(".")
        w = getattr(want[rec], field)
        assert g[key].shape == w.shape, key
        assert np.array_equal(g[key].view(np.uint8), np.ascontiguousarray(w).view(np.uint8)), key
        n += 1
    assert n == 2 + 4 + 4 + 4 + 4 + 4


def test_all_gather_single_process_is_identity():
    from nvfp4_quantization_current_gb300.distributed import all_gather_shards
    a = torch.arange(6).reshape(2, 3)
    assert all_gather_shards(a, 1) is a
