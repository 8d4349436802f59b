"""The multi-GPU path is replicas only: each rank compresses its own pool, the
ranks meet at a barrier around the timed region and the slowest rank's time
sets the job's throughput.  These tests run that plumbing as two gloo ranks on
the CPU (no GPU, no data-path collective)."""
import json
import os
import socket
import tempfile

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    w, r, local = bench.dist_env()
    dist = bench.init_group(w, "gloo")
    bench.barrier(dist)
    slowest = bench.reduce_max(dist, 1.0 + rank)          # rank 1 is the slow one
    value = bench.replica_value(w, 10, 8192, slowest)
    bench.barrier(dist)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "slowest": slowest, "value": value}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_slowest_rank():
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(2, port, d), nprocs=2, join=True, start_method="spawn")
        res = [json.load(open(os.path.join(d, f"rank{r}.json"))) for r in range(2)]
    for r, x in enumerate(res):
        assert x["world"] == 2 and x["rank"] == r and x["local"] == r
        assert x["slowest"] == 2.0                          # the max over ranks, seen by every rank
        assert x["value"] == pytest.approx(2 * 10 * 8192 / 2.0 / 1e6)


def test_single_process_needs_no_group():
    assert bench.init_group(1, "gloo") is None
    bench.barrier(None)
    assert bench.reduce_max(None, 3.5) == 3.5
    assert bench.replica_value(1, 4, 1000, 2.0) == pytest.approx(4 * 1000 / 2.0 / 1e6)


def test_reference_arm_prints_only_on_rank_0(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_each_rank_compresses_its_own_pool():
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS["single_head_n512_d64"]
    a, b = synth.make_layer(wl, layer=0), synth.make_layer(wl, layer=1)
    assert not (a["K"] == b["K"]).all()
