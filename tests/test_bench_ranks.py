"""Multi-rank host logic of bench.py on CPU: two gloo processes (world size 2).

bench.py runs one process per GPU under torchrun; the path shards by batch with
no data exchange, so the only cross-rank steps are the barrier around the timed
region and the max over ranks of the elapsed time. These run here with the
gloo backend on 127.0.0.1; the GPU step itself is not involved."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.rank_env()
        dev = torch.device("cpu")
        # every rank times a different step; the job's time is the slowest rank's
        elapsed = 10.0 + 5.0 * rank
        dist.barrier()
        slowest = bench.max_over_ranks(elapsed, w, dev)
        dist.barrier()
        flops = 1e12
        res = {"world": w, "rank": r, "local": local, "slowest": slowest,
               "value": bench.job_tflops(w, flops, slowest), "seeds": bench.rank_seeds(r)}
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_seeds(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        # both ranks agree on the slowest rank's time (rank 1: 15 ms)
        assert d["slowest"] == 15.0
        # whole-job throughput: 2 ranks x 1 TFLOP in 15 ms
        assert d["value"] == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
    # weak scaling: each rank draws its own inputs
    assert res[0]["seeds"] != res[1]["seeds"]
    assert set(res[0]["seeds"]) == {"q", "k", "v", "do"}


def test_single_rank_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for v in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)


def test_reference_arm_only_on_rank0(monkeypatch, capsys):
    """Under torchrun the reference arm runs on rank 0 alone; other ranks exit without work."""
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.reference_arm(argparse.Namespace(steps=1, warmup=0))
    assert capsys.readouterr().out == ""


def _shard_worker(rank, world, port, out_dir):
    """One rank of a scope-sharded step, with the oracle standing in for the GPU
    calls: the rank computes its round-robin scopes and writes only their rows;
    the ranks' rows are then gathered (no exchange is needed by the method;
    this only checks the partition and the assembled result)."""
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import numpy as np
    import torch
    import torch.distributed as dist
    import sparse_spatiotemporal_attention_gb300 as skp
    from oracle import skiparse_oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, heads, D, T, H, W, k, mode = 1, 2, 16, 2, 5, 7, 3, O.GROUP       # N = 70: unequal scopes
        N = T * H * W
        rs = np.random.default_rng(5)
        q, kk, v, do = (rs.standard_normal((B, N, heads, D)) for _ in range(4))
        first, step = skp.scope_shard(k, world, rank)
        out = np.zeros((B, N, heads, D))
        owner = np.zeros(N)
        for s in range(first, k, step):
            for h in range(heads):
                r = O.skiparse_scope(q, kk, v, do, T, H, W, k, mode, 0, h, s)
                out[0, r["tokens"], h] = r["dq"]
            owner[O.scope_tokens(N, k, mode, s)] += 1
        t_out, t_own = torch.from_numpy(out), torch.from_numpy(owner)
        dist.all_reduce(t_out)
        dist.all_reduce(t_own)
        dq, _, _, _, _ = O.skiparse_bwd(q, kk, v, do, T, H, W, k, mode)
        res = {"covered_once": bool((t_own == 1).all()), "err": float(np.abs(t_out.numpy() - dq).max()),
               "mine": list(range(first, k, step))}
        with open(os.path.join(out_dir, f"shard{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_scope_shards(tmp_path):
    """Two ranks split the scopes of one batch round-robin: every token's rows
    come from exactly one rank and the gathered gradients equal the whole
    backward's."""
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_shard_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"shard{r}.json")) for r in range(2)]
    assert res[0]["mine"] == [0, 2] and res[1]["mine"] == [1]
    for d in res:
        assert d["covered_once"]
        assert d["err"] < 1e-12
