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


def test_traffic_figures_match_their_profiles():
    """The DRAM bytes that bench.py reports come from the captures summarised under profiles/:
    the same kernel-source hash and the same counter values, one profile per path."""
    import re

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    files = {"sage2": "traffic_attn_pp_gqa_long_causal_B1_Hq32_Hkv8_N32768_D128.md",
             "sage1": "traffic_attn_fwd_gqa_long_causal_B1_Hq32_Hkv8_N32768_D128.md"}
    for (workload, quant), (digest, nbytes) in bench.MEASURED_TRAFFIC.items():
        text = open(os.path.join(root, "profiles", files[quant])).read()
        assert f"sha256 prefix `{digest}`" in text, (quant, digest)
        rows = dict(re.findall(r"\| (dram__bytes_(?:read|write)\.sum) \| ([0-9.]+) MB \|", text))
        got = (float(rows["dram__bytes_read.sum"]) + float(rows["dram__bytes_write.sum"])) * 1e6
        assert abs(got - nbytes) <= 0.01e6, (quant, got, nbytes)
