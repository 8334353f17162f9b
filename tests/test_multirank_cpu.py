"""Multi-rank logic on CPU (gloo, world size 2), with the oracle standing in for the GPU.

1. Data parallel over sequences: each rank scores and ranks its own sequences; the
   union of the ranks' results equals the single-process result, with no collective on
   the data path (only the final comparison gathers results).
2. Context parallel over one long sequence: each rank ranks its half of the keys; one
   all-gather of the (value, index) lists and an exact re-selection under the tie rule
   reproduce the global top-k.  This is the same exactness argument the GPU path uses
   when it splits a row's keys over CTAs and merges the partial lists.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import parity
from oracle import dsa_oracle as orc


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
        # ---- 1. DP over sequences
        wl = parity.make_case(7, [300, 517, 64, 1000], next_n=2, block_size=16, topk=40)
        seqs = [b for b in range(wl.B) if b % world == rank]
        rows = np.concatenate([np.arange(b * wl.next_n, (b + 1) * wl.next_n) for b in seqs])
        lg = parity.oracle_logits(wl, rows=rows)
        idx, _ = orc.topk_select(lg, wl.topk)
        gathered = [None] * world
        dist.all_gather_object(gathered, (rows.tolist(), idx.tolist()))
        # ---- 2. CP over keys of one sequence
        wl2 = parity.make_case(8, [2000], next_n=3, paged=False, topk=64)
        full = parity.oracle_logits(wl2)
        L = full.shape[1]
        lo, hi = rank * L // world, (rank + 1) * L // world
        part = np.full_like(full, -np.inf)
        part[:, lo:hi] = full[:, lo:hi]
        pidx, pval = orc.topk_select(part, wl2.topk)
        lists = [None] * world
        dist.all_gather_object(lists, (pidx.tolist(), pval.tolist()))
        if rank == 0:
            q.put(("dp", gathered))
            q.put(("cp", lists))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_sharding_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=240) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # DP: the union equals one process over the whole batch
    wl = parity.make_case(7, [300, 517, 64, 1000], next_n=2, block_size=16, topk=40)
    want, _ = orc.topk_select(parity.oracle_logits(wl), wl.topk)
    merged = np.full_like(want, -2)
    for rows, idx in got["dp"]:
        merged[np.array(rows)] = np.array(idx)
    assert np.array_equal(merged, want)
    # CP: exact merge of the per-rank lists == global top-k
    wl2 = parity.make_case(8, [2000], next_n=3, paged=False, topk=64)
    full = parity.oracle_logits(wl2)
    want2, _ = orc.topk_select(full, wl2.topk)
    T = full.shape[0]
    cand = np.full((T, full.shape[1]), -np.inf)
    for pidx, pval in got["cp"]:
        pidx, pval = np.array(pidx), np.array(pval)
        for t in range(T):
            live = pidx[t] >= 0
            cand[t, pidx[t][live]] = pval[t][live]
    merged2, _ = orc.topk_select(cand, wl2.topk)
    assert np.array_equal(merged2, want2)
