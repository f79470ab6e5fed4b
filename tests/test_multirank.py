"""The N > 1 path on the CPU: two gloo ranks.

Tokens are independent through the whole layer (routing, both GEMMs and the
combine act per slot row / per token), so the work shards by batch with no
data-path collective. These tests check, without a GPU:
  * the only cross-rank operation of the bench (max of the elapsed times);
  * that token shards run separately reproduce the full batch bit for bit
    (the property weak scaling relies on), using the oracle on each rank;
  * that the reference arm under torchrun prints one line from rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    return dist


def _max_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    dist = _init(rank, world, port)
    total, e2e = [(3.0, 7.5), (4.5, 2.0)][rank]
    got = bench.max_over_ranks(dist, total, e2e, device="cpu")
    none_case = bench.max_over_ranks(dist, 1.0 + rank, None, device="cpu")
    q.put((rank, got, none_case))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, got, none_case in res:
        assert got == (4.5, 7.5)
        assert none_case == (2.0, None)


def _shard_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import oracle
    import workloads
    dist = _init(rank, world, port)
    w = workloads.CONFIGS["tiny"]
    d = workloads.host_inputs(w)
    lo, hi = rank * w.T // world, (rank + 1) * w.T // world
    dims = dict(T=hi - lo, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S, clamp=w.clamp)
    res = oracle.get().forward(dims, d["x"][lo:hi], d["x_sf"][lo:hi], d["topk_idx"][lo:hi], d["topk_w"][lo:hi],
                               d["w1"], d["w1_sf"], d["w2"], d["w2_sf"], nthreads=2)
    mine = torch.from_numpy(res["out"].astype(np.int32))
    parts = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine)
    if rank == 0:
        q.put(torch.cat(parts).numpy().astype(np.uint16))
    dist.destroy_process_group()


def test_token_shards_reproduce_the_full_batch(orc):
    import workloads
    w = workloads.CONFIGS["tiny"]
    d = workloads.host_inputs(w)
    dims = dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S, clamp=w.clamp)
    full = orc.forward(dims, d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"],
                       d["w2_sf"])["out"]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    sharded = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sharded.shape == full.shape
    assert np.array_equal(sharded, full)


def test_reference_arm_under_torchrun_prints_once(orc):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
