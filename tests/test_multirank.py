"""Multi-rank host logic on CPU (gloo, world size 2).

1. Replicas: sequences are independent, so sharding a batch's sequences over ranks and
   gathering the per-rank selections reproduces the single-process result (no data exchange).
2. Context-parallel indexer design ("local Top-K compression before communication", Inference
   Optimization for Kimi K3.1 Pro ..., section 5.1): each rank scores its own slice of a long
   sequence's positions, keeps its local top-K as (score, position) candidates, the candidates are
   all-gathered (the one exchange step), and a merge by (score desc, position asc) gives exactly
   the unsharded selection.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import dsa_inputs as di
import oracle


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _workload():
    return di.Workload("mr", [300, 1200, 77, 640, 2000], [1, 2, 1, 3, 1], H_I=4, d_I=16, K=64,
                       H=2, d_qk=32, d_v=16, page_size=16, seed=41)


def local_topk(scores, positions, K):
    """Local candidates of one shard: the K best (score, position) pairs in selection order."""
    order = np.lexsort((positions, -scores))[:K]
    return scores[order], positions[order]


def merge_candidates(cand_scores, cand_pos, K):
    """Merge all shards' candidates by (score desc, position asc); return ascending positions."""
    order = np.lexsort((cand_pos, -cand_scores))[:K]
    return np.sort(cand_pos[order])


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = _workload()
        inp = di.generate(wl)
        # 1. replicas over sequences
        qs = inp["q_start"].tolist()
        mine = [t for b in range(wl.B) if b % world == rank for t in range(qs[b], qs[b + 1])]
        idx, _, _ = oracle.li_topk(inp, mine)
        rows = torch.full((wl.n_q, wl.K), -2, dtype=torch.int32)
        rows[mine] = torch.from_numpy(idx)
        gathered = [torch.empty_like(rows) for _ in range(world)]
        dist.all_gather(gathered, rows)
        merged = torch.stack(gathered).max(0).values  # each token owned by exactly one rank
        # 2. context-parallel candidates for the last token of the longest sequence
        t = qs[4 + 1] - 1
        s, _ = oracle.li_scores(inp, t)
        n = len(s)
        lo, hi = rank * n // world, (rank + 1) * n // world
        cs, cp = local_topk(s[lo:hi], np.arange(lo, hi), wl.K)
        pad = wl.K - len(cs)
        cs = torch.from_numpy(np.concatenate([cs, np.full(pad, -np.inf)]))
        cp = torch.from_numpy(np.concatenate([cp, np.full(pad, -1)]).astype(np.int64))
        gs = [torch.empty_like(cs) for _ in range(world)]
        gp = [torch.empty_like(cp) for _ in range(world)]
        dist.all_gather(gs, cs)
        dist.all_gather(gp, cp)
        allc = torch.cat(gs).numpy()
        allp = torch.cat(gp).numpy()
        keep = allp >= 0
        cp_sel = merge_candidates(allc[keep], allp[keep], wl.K)
        if rank == 0:
            q.put((merged.numpy(), t, cp_sel))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_and_context_parallel_merge():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    merged, t, cp_sel = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = _workload()
    inp = di.generate(wl)
    full, _, _ = oracle.li_topk(inp)
    assert np.array_equal(merged, full)
    assert np.array_equal(cp_sel, full[t][full[t] >= 0])
