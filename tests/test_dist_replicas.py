"""Data-parallel replicas across ranks, on CPU with the gloo backend.

Each rank of a multi-GPU benchmark holds the same weights and its own token
shard, and no collective touches the data path: the routed layer maps every
token through its own top-k experts and fixed-order weighted sum, so a token's
output depends on that token alone. These tests run two gloo ranks that
compute their shard with the oracle and check (a) the shards share weights
and differ in tokens, (b) the concatenated shard outputs equal the oracle on
all tokens at once, bit for bit, and (c) the benchmark's max-over-ranks
timing reduction and whole-job rate.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WL_KW = dict(T=48, H=256, I=128, E=8, k=2, zipf_s=1.2, shared_I=128)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from combine_router_top_expert_gb300 import synth
        wl = synth.small("dp_shard", **WL_KW)
        inp = synth.make_inputs(wl, shard=rank)
        r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
        y = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, shared=inp.shared)
        ys = [torch.empty(y.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(ys, torch.from_numpy(np.ascontiguousarray(y)))
        xs = [torch.empty(inp.x.shape, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(xs, torch.from_numpy(inp.x.astype(np.int32)))
        wsum = torch.tensor([float(inp.Wg.astype(np.int64).sum()), float(inp.Wd.astype(np.int64).sum()),
                             float(inp.W_r.astype(np.float64).sum())], dtype=torch.float64)
        wsums = [torch.empty_like(wsum) for _ in range(world)]
        dist.all_gather(wsums, wsum)
        # per-rank timings as the benchmark reduces them: the slowest rank wins
        mx = bench.max_over_ranks([10.0 + rank, 5.0 - rank], torch.device("cpu"))
        if rank == 0:
            np.save(os.path.join(out_dir, "y.npy"), torch.cat(ys).numpy())
            np.save(os.path.join(out_dir, "x.npy"), torch.cat(xs).numpy().astype(np.uint16))
            np.save(os.path.join(out_dir, "wsums.npy"), torch.stack(wsums).numpy())
            np.save(os.path.join(out_dir, "mx.npy"), np.array(mx))
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    import oracle
    oracle.build()
    out = str(tmp_path_factory.mktemp("dp"))
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    return {n: np.load(os.path.join(out, n + ".npy")) for n in ("y", "x", "wsums", "mx")}


def test_shards_share_weights_and_differ_in_tokens(two_ranks):
    T = WL_KW["T"]
    w = two_ranks["wsums"]
    assert np.array_equal(w[0], w[1])
    x = two_ranks["x"]
    assert not np.array_equal(x[:T], x[T:])
    from combine_router_top_expert_gb300 import synth
    wl = synth.small("dp_shard", **WL_KW)
    assert np.array_equal(x[:T], synth.make_inputs(wl).x)    # shard 0 is the single-GPU input


def test_sharded_outputs_equal_the_whole_batch(two_ranks):
    import oracle
    from combine_router_top_expert_gb300 import synth
    wl = synth.small("dp_shard", **WL_KW)
    inp = synth.make_inputs(wl)
    x_all = two_ranks["x"]
    r = oracle.route(x_all, inp.W_r, wl.k, inp.bias)
    y_all = oracle.moe_forward(x_all, inp.Wg, inp.Wu, inp.Wd, r, shared=inp.shared)
    assert np.array_equal(y_all, two_ranks["y"])


def test_max_over_ranks_and_rate(two_ranks):
    assert list(two_ranks["mx"]) == [11.0, 5.0]
    import sys
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 2560 tokens x 100 steps in 1.6 s of the slowest rank
    assert bench.whole_job_rate(2, 2560, 100, 1600.0) == pytest.approx(320000.0)
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu")) == [3.0, 4.0]   # no process group
