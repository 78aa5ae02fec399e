"""Host logic of expert parallelism over two gloo ranks on the CPU: each rank
routes its own token shard (the oracle's routing), the per-rank expert
counts are all-gathered over the process group, and each rank's plan pulls
exactly the rows routed to its experts, so the ranks together pull every
(source rank, slot) exactly once."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from combine_router_top_expert_gb300 import ep, synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, G, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=G)
    try:
        wl = synth.small("epd", T=64, H=128, I=64, E=8, k=2, zipf_s=1.2)
        inp = synth.make_inputs(wl, shard=rank)
        r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
        counts_all = ep.gather_counts(torch.from_numpy(r["counts"].astype(np.int32)))
        # the sources' layouts, as the peer table would expose them
        offs = [None] * G
        rsrc = [None] * G
        dist.all_gather_object(offs, r["offsets"].tolist())
        dist.all_gather_object(rsrc, r["row_src"].tolist())
        offs = [np.array(o) for o in offs]
        rsrc = [np.array(o) for o in rsrc]
        cl, ol, seg = ep.plan_host(counts_all.numpy(), rank)
        pulled = ep.pulled_slots_host(counts_all.numpy(), rank, offs, rsrc)
        # each pulled slot chose one of this rank's experts
        mine = set(ep.local_experts(rank, G, wl.E))
        idx_all = [None] * G
        dist.all_gather_object(idx_all, r["idx"].tolist())
        ok_local = all(idx_all[s][slot // wl.k][slot % wl.k] in mine for s, slot in pulled)
        q.put((rank, counts_all.numpy().tolist(), int(ol[-1]), len(pulled), ok_local, pulled))
    finally:
        dist.destroy_process_group()


def test_counts_all_gather_and_plan_partition():
    G = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, G, port, q)) for r in range(G)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(G))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks hold the same gathered counts; rank s's row is its own routing
    assert res[0][1] == res[1][1]
    counts = np.array(res[0][1])
    assert counts.shape == (G, 8) and counts.sum() == G * 64 * 2
    for rank, _, n_local, n_pulled, ok_local, pulled in res:
        assert n_local == n_pulled and ok_local
    union = [x for r in res for x in r[5]]
    assert sorted(union) == sorted((s, j) for s in range(G) for j in range(64 * 2))
