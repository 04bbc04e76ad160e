"""The multi-GPU path on CPU: two gloo ranks run the bench's partition and timing logic.

Every (sequence, v-head) unit is independent, so ranks shard by sequence with no
exchange on the data path (weak scaling); the only collectives are the barrier
and the max over ranks of the timed region. Run here as two spawned processes.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from gated_deltanet_linear_scan_gb300 import inputs as I

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for cid in (3, 4, 2):
            cfg = I.get_config(cid)
            work = bench.rank_work(cfg, rank)
            gathered = [None] * world
            dist.all_gather_object(gathered, work)
            seqs = [s for w in gathered for s in w["seqs"]]
            pools = [s for w in gathered for s in w["pool_ids"]]
            assert len(set(seqs)) == len(seqs) == world * cfg.n_seqs
            assert len(set(pools)) == len(pools) == world * cfg.pool_size
            assert len(work["seqs"]) == cfg.n_seqs  # fixed work per rank: weak scaling
        # each rank's inputs are its own seeded streams, regenerable anywhere
        cfg = I.get_config(3, n_seqs=2, n_k_heads=1, n_v_heads=2, state_size=32)
        work = bench.rank_work(cfg, rank)
        mine = I.block_step(cfg, 0, seqs=work["seqs"])["qkv"]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        assert not np.array_equal(gathered[0], gathered[1])
        np.testing.assert_array_equal(gathered[rank], mine)
        # the timed region is the max over ranks
        t = bench.reduce_max(0.25 + rank, dist, "cpu")
        assert t == 0.25 + (world - 1)
        dist.barrier()
        with open(os.path.join(out_dir, f"ok{rank}"), "w") as f:
            f.write("ok")
    finally:
        dist.destroy_process_group()


def test_two_rank_partition_and_timing(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        assert (tmp_path / f"ok{r}").read_text() == "ok"


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5, None, "cpu") == 3.5
