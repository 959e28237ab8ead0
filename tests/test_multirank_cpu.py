"""Multi-rank host logic on CPU (gloo, world size 2).

Two uses of more than one GPU are covered here without a GPU:
* independent caches per rank (the bench's weak-scaling mode): the job
  throughput is the total work over the max time across ranks;
* one cache sharded by layer: each rank holds L/2 layers, computes the
  KeyDiff partial sum over its heads, and a single all-reduce(sum) of N
  floats gives the global token score -- the only exchange step of the
  path; after it the selection is replicated, the scoring and eviction are
  shard-local and the sink pin needs one scalar all-reduce(max).
The merged results must equal the unsharded oracle.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import kv_synth as ks
from oracle import kv2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = ks.scaled(ks.TINY, L=4, Hkv=2, Hq=4, N=600, m=128, rho=0.2, budget=0.05, needles_per_layer=3)
        x = ks.gen_kv2(cfg)
        L, H, N, S = cfg.L, cfg.Hkv, cfg.N, cfg.sinks
        mine = list(range(rank * L // world, (rank + 1) * L // world))
        # partial sum of per-head KeyDiff scores over this rank's layers
        _, s_local = kv2.proxy_scores(x.K[mine])
        part = torch.from_numpy(s_local.reshape(-1, N).sum(axis=0))
        dist.all_reduce(part, op=dist.ReduceOp.SUM)
        p = part.numpy() / (L * H)
        sel, chunks = kv2.select_queries(p, N, S, cfg.m, cfg.rho)
        score, _ = kv2.recon_scores(x.K[mine], x.Q[mine], sel, chunks)
        local_max = torch.tensor([np.nanmax(score[:, :, S:])], dtype=torch.float64)
        dist.all_reduce(local_max, op=dist.ReduceOp.MAX)
        score[:, :, :S] = local_max.item()
        k = kv2.budget_count(cfg.budget, N)
        kept = kv2.evict(score, S, [k] * len(mine))
        # weak-scaling timing rule: job time is the max over ranks
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        q.put((rank, p, sel, [kk.tolist() for kk in kept], local_max.item(), t.item()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_layer_sharded_merge_equals_unsharded():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=240) for _ in range(world)], key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg = ks.scaled(ks.TINY, L=4, Hkv=2, Hq=4, N=600, m=128, rho=0.2, budget=0.05, needles_per_layer=3)
    x = ks.gen_kv2(cfg)
    ref = kv2.kv2_compress(x.K, x.V, x.Q, cfg.sinks, cfg.m, cfg.rho, [kv2.budget_count(cfg.budget, cfg.N)] * cfg.L)
    for r in res:
        np.testing.assert_allclose(r[1], ref["p"], rtol=1e-12, atol=1e-15)
        assert r[2].tolist() == ref["sel"][0].tolist()
        assert r[4] == pytest.approx(float(ref["score"][:, :, cfg.sinks:].max()), rel=0, abs=0)
        assert r[5] == 2.0
    merged = res[0][3] + res[1][3]
    assert merged == [kk.tolist() for kk in ref["kept"]]
