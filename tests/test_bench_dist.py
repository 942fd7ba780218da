"""The bench's multi-rank host logic on CPU: two gloo ranks agree on the slowest time and
on the whole-job throughput (no GPU involved)."""
from __future__ import annotations

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    secs = 1.0 + rank  # rank 1 is the slow one
    mx = bench.max_over_ranks(secs, w)
    val = bench.aggregate_value(1e12, mx, w)
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_two_rank_max_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, mx, val in res:
        assert mx == 2.0                      # max over ranks
        assert val == pytest.approx(1.0)      # 2 ranks x 1e12 ops / 2 s = 1 TOPS


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_value(2e12, 2.0, 1) == pytest.approx(1.0)


def test_traffic_data_file_and_hash_guard(monkeypatch):
    """bench.py takes its DRAM traffic figures from bench_traffic.json and reports one only while
    the attention kernel's source has the hash that the figure was captured on."""
    import json

    import bench
    from bit_exact_attention_gb300 import workloads as W
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    data = json.load(open(bench.TRAFFIC_FILE))
    assert data["entries"]
    for e in data["entries"]:
        assert e["dram_read_bytes"] > 0 and e["dram_write_bytes"] > 0
        assert len(e["source_sha16"]) == 16 and int(e["source_sha16"], 16) >= 0
        assert os.path.exists(os.path.join(root, e["profile"])), e["profile"]
    digest, nbytes = bench.MEASURED_TRAFFIC[(W.GQA_LONG.name, "sage2")]
    monkeypatch.setattr(bench, "kernel_source_sha16", lambda: digest)
    assert bench.measured_traffic(W.GQA_LONG) == nbytes
    monkeypatch.setattr(bench, "kernel_source_sha16", lambda: "0" * 16)
    assert bench.measured_traffic(W.GQA_LONG) is None


def test_visited_keys_by_enumeration():
    """The DeltaS entries counted for the prepass's algorithmic bytes: every key of every KV tile
    a Q block visits, checked against a per-row enumeration of the bottom-right causal rule."""
    import bench
    for nq, nkv in [(1, 1), (300, 100), (100, 300), (256, 256), (1000, 777), (5, 4000)]:
        for causal in (False, True):
            want = 0
            for qb in range((nq + 127) // 128):
                last = -1
                for i in range(qb * 128, min(nq, qb * 128 + 128)):
                    jmax = nkv - 1 if not causal else min(nkv - 1, i + nkv - nq)
                    last = max(last, jmax)
                want += 0 if last < 0 else min(nkv, (last // 128 + 1) * 128)
            assert bench.visited_keys(nq, nkv, causal) == want, (nq, nkv, causal)
