"""The N > 1 path on CPU: two gloo ranks each hold a row shard, agree on the
amax through the library's MAX all-reduce helper, quantize their shard with
the CPU oracle, and the gathered codes must equal the unsharded oracle
result bit for bit (per-tensor current scaling and NVFP4)."""
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
        np.savez(os.path.join(result_dir, f"r{rank}.npz"), amax=np.float32(glob), cs_row=cs.q_row, cs_colT=cs.q_colT,
                 cs_s=cs.scale, nv_row=nv.q_row, nv_sb=nv.sb_row, nv_colT=nv.q_colT, nv_sbT=nv.sb_colT,
                 nv_sg=nv.s_global)
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


def test_allreduce_amax_single_process_is_identity():
    from nvfp4_quantization_current_gb300.distributed import allreduce_amax_
    a = torch.tensor([3.5])
    assert allreduce_amax_(a).item() == 3.5
    with pytest.raises(ValueError):
        allreduce_amax_(torch.tensor([1.0, 2.0]))
