"""The N > 1 path on CPU: two gloo ranks each hold a row shard, agree on the
amax through the library's MAX all-reduce helper, quantize their shard with
the CPU oracle, and the gathered codes must equal the unsharded oracle
result bit for bit (per-tensor current scaling, NVFP4, two steps of delayed
scaling with all-reduced window slots, and the random-Hadamard NVFP4
columnwise copy with the all-reduced amax of the transform)."""
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
        from nvfp4_quantization_current_gb300.distributed import allreduce_amax_

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
        np.savez(os.path.join(result_dir, f"r{rank}.npz"), amax=np.float32(glob), cs_row=cs.q_row, cs_colT=cs.q_colT,
                 cs_s=cs.scale, nv_row=nv.q_row, nv_sb=nv.sb_row, nv_colT=nv.q_colT, nv_sbT=nv.sb_colT,
                 nv_sg=nv.s_global, ds0_row=ds[0], ds0_colT=ds[1], ds1_row=ds[2], ds1_colT=ds[3],
                 rht_q=rq, rht_sb=rsb, rht_sg=np.float32(rsg))
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


def test_allreduce_amax_single_process_is_identity():
    from nvfp4_quantization_current_gb300.distributed import allreduce_amax_
    a = torch.tensor([3.5])
    assert allreduce_amax_(a).item() == 3.5
    with pytest.raises(ValueError):
        allreduce_amax_(torch.tensor([1.0, 2.0]))
