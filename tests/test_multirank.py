"""Host-side logic of bench.py's multi-replica path on CPU: two gloo ranks,
each with its own seeded batch, the slowest rank's time and the weak-scaling
aggregate (no GPU, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import bench
    import oracle
    import workloads

    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each replica draws its own batch (seed = rank) of the ragged workload shape
    inp = workloads.make_workload("ragged_v2_bf16", seed=rank, num_seqs=8)
    lens = inp["seq_lens_list"]
    splits = oracle.num_kv_splits(lens, 1, 32, 8, 16, 148)
    elapsed = 1.0 + rank  # stand-in per-rank step time
    slowest = bench.max_over_ranks(elapsed, dist, "cpu")
    kv = sum(lens) * 8 * 2 * 128 * 2
    kv_all = torch.tensor([kv], dtype=torch.float64)
    dist.all_reduce(kv_all)
    value = bench.aggregate_gbs(kv, world, slowest)
    torch.save({"rank": rank, "lens": lens, "splits": splits, "slowest": slowest, "value": value,
                "kv": kv, "kv_all": float(kv_all.item())},
               os.path.join(out_dir, f"r{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [torch.load(os.path.join(tmp_path, f"r{i}.pt")) for i in range(world)]
    assert r[0]["lens"] != r[1]["lens"]  # independent batches
    assert r[0]["slowest"] == r[1]["slowest"] == 2.0
    assert r[0]["value"] == pytest.approx(world * r[0]["kv"] / 2.0 / 1e9)
    assert r[0]["kv_all"] == pytest.approx(r[0]["kv"] + r[1]["kv"])
    for x in r:
        assert all(1 <= v <= 16 for v in x["splits"])
