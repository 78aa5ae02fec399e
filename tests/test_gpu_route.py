"""Router / top-k / layout on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import dev_f32, to_dev_bf16

CASES = [
    dict(T=64, H=128, E=8, k=2),
    dict(T=300, H=512, E=32, k=8),
    dict(T=1000, H=7168, E=32, k=8, zipf_s=1.2),
    dict(T=1, H=256, E=16, k=4),
    dict(T=257, H=384, E=256, k=16),
    dict(T=40, H=128, E=5, k=5),
    dict(T=33, H=1152, E=64, k=1),
    # enough tokens for the 18- and 28-token CTA tiles on a 152-SM part
    dict(T=2600, H=256, E=64, k=6),
    dict(T=4096, H=384, E=32, k=8),
]


def _run(x, W_r, k, bias=None):
    xd = to_dev_bf16(x)
    r = mok.route_layout(xd, dev_f32(W_r), k, None if bias is None else dev_f32(bias))
    torch.cuda.synchronize()
    return {n: v.cpu().numpy() for n, v in r.items()}


def _compare(g, ref, T, k):
    assert np.array_equal(g["topk_idx"], ref["idx"])
    assert np.array_equal(g["counts"], ref["counts"])
    assert np.array_equal(g["offsets"], ref["offsets"])
    assert np.array_equal(g["row_src"][:T * k], ref["row_src"])
    assert np.array_equal(g["slot_row"][:T * k], ref["slot_row"])
    assert np.max(np.abs(g["topk_w"].astype(np.float64) - ref["w"])) <= 1e-6
    assert np.all(np.abs(g["topk_w"].sum(1) - 1.0) <= 1e-6)


@pytest.mark.gpu
@pytest.mark.parametrize("c", CASES, ids=[f"T{c['T']}_H{c['H']}_E{c['E']}_k{c['k']}" for c in CASES])
def test_route_layout_bit_exact(c):
    wl = synth.small("r", T=c["T"], H=c["H"], I=64, E=c["E"], k=c["k"], zipf_s=c.get("zipf_s", 0.0))
    g = torch.Generator().manual_seed(c["T"] * 7 + c["E"])
    x = synth._normal_bf16(g, (wl.T, wl.H), 1.0)
    W_r = (torch.randn((wl.H, wl.E), generator=g) * 0.02).numpy()
    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    ref = oracle.route(x, W_r, wl.k, bias)
    _compare(_run(x, W_r, wl.k, bias), ref, wl.T, wl.k)


@pytest.mark.gpu
def test_route_ties_and_zero_input():
    """All-zero x: every logit is 0 (or the bias); ties go to the lower index."""
    T, H, E, k = 50, 256, 16, 4
    x = np.zeros((T, H), np.uint16)
    W_r = np.random.default_rng(0).standard_normal((H, E)).astype(np.float32)
    ref = oracle.route(x, W_r, k)
    assert np.all(ref["idx"] == np.arange(k))
    _compare(_run(x, W_r, k), ref, T, k)
    bias = np.zeros(E, np.float32)
    bias[[3, 9]] = 1.0
    ref = oracle.route(x, W_r, k, bias)
    _compare(_run(x, W_r, k, bias), ref, T, k)


@pytest.mark.gpu
def test_route_all_tokens_one_expert():
    T, H, E, k = 200, 256, 8, 1
    g = torch.Generator().manual_seed(5)
    x = synth._normal_bf16(g, (T, H), 1.0)
    W_r = (torch.randn((H, E), generator=g) * 0.02).numpy()
    bias = np.full(E, -100.0, np.float32)
    bias[6] = 100.0
    ref = oracle.route(x, W_r, k, bias)
    assert ref["counts"][6] == T
    _compare(_run(x, W_r, k, bias), ref, T, k)


@pytest.mark.gpu
def test_route_follows_the_fixed_summation_order():
    """The hand-built input of tests/golden/router_order.json, whose fp32
    logits are (1, 2) only in the fixed chain/butterfly order (exact
    arithmetic and chains over h mod 32 tie at (2, 2), which would rank
    expert 0 first): the kernel must rank expert 1 first, with and without
    the bias, and weight the two experts softmax(2, 1)."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "router_order.json")))
    x = np.zeros((1, g["H"]), np.float32)
    for h, v in g["x_nonzero"]:
        x[0, h] = v
    W = np.zeros((g["H"], g["E"]), np.float32)
    for h, e, v in g["W_r_nonzero"]:
        W[h, e] = v
    xb = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for bias in (None, np.array(g["bias"], np.float32)):
        got = _run(xb, W, 2, bias)
        assert got["topk_idx"][0].tolist() == g["k2"]["idx"]
        if bias is None:
            assert np.max(np.abs(got["topk_w"][0] - np.array(g["k2"]["w"]))) <= 1e-6
        ref = oracle.route(xb, W, 2, bias)
        _compare(got, ref, 1, 2)


@pytest.mark.gpu
def test_route_wait_that_gives_up_is_reported():
    """A router copy withheld by the test hook: the chunk wait runs out after
    the short limit, the workspace status reports MOK_ERR_TIMEOUT (detail 7)
    and the outputs are still a valid layout; without the hook the same call
    routes bit-exactly again."""
    T, H, E, k = 700, 2048, 32, 8
    g = torch.Generator().manual_seed(9)
    x = synth._normal_bf16(g, (T, H), 1.0)
    W_r = (torch.randn((H, E), generator=g) * 0.02).numpy()
    xd, wd = to_dev_bf16(x), dev_f32(W_r)
    ws = mok.alloc_bytes(mok.route_workspace_size(T, H, E, k))
    mok.route_test_hook(1, timeout_ms=50)
    try:
        r = mok.route_layout(xd, wd, k, workspace=ws)
        torch.cuda.synchronize()
        assert mok.device_status(ws) == (mok.ERR_TIMEOUT, 7)
        idx = r["topk_idx"].cpu().numpy()
        assert idx.min() >= 0 and idx.max() < E and all(len(set(row)) == k for row in idx.tolist())
        assert int(r["counts"].sum()) == T * k
    finally:
        mok.route_test_hook(0, 0)
    r = mok.route_layout(xd, wd, k, workspace=ws)
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    _compare({n: v.cpu().numpy() for n, v in r.items()}, oracle.route(x, W_r, k), T, k)
