"""mok_route_layout_static: routing for callers that cannot allocate device
memory (their allocations must go through a framework allocator they cannot
reach, or their process has no device memory left to reserve). It must give
exactly the outputs of mok_route_layout, call after call, using only the
library's fixed scratch array. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import dev_f32, to_dev_bf16


def _inputs(T, H, E, seed, zipf=0.0):
    g = torch.Generator().manual_seed(seed)
    x = synth._normal_bf16(g, (T, H), 1.0)
    W_r = (torch.randn((H, E), generator=g) * 0.02).numpy()
    bias = synth.zipf_bias(E, zipf) if zipf else None
    return x, W_r, bias


@pytest.mark.gpu
def test_static_scratch_routing_matches_workspace_routing_twice():
    cases = [dict(T=2560, H=7168, E=32, k=8, seed=0, zipf=0.0),
             dict(T=1000, H=7168, E=32, k=8, seed=1, zipf=1.2)]
    for c in cases:   # two calls in a row through the C ABI
        x, W_r, bias = _inputs(c["T"], c["H"], c["E"], c["seed"], c["zipf"])
        xd, wd = to_dev_bf16(x), dev_f32(W_r)
        bd = None if bias is None else dev_f32(bias)
        ref = mok.route_layout(xd, wd, c["k"], bd)
        got = mok.route_layout_static(xd, wd, c["k"], bd)
        torch.cuda.synchronize()
        R = c["T"] * c["k"]
        for n in ("topk_idx", "counts", "offsets"):
            assert torch.equal(got[n], ref[n]), n
        for n in ("row_src", "slot_row"):
            assert torch.equal(got[n][:R], ref[n][:R]), n
        # the routing weights are the same kernel's fp32 values: bit-identical
        assert torch.equal(got["topk_w"].view(torch.int32), ref["topk_w"].view(torch.int32))
        o = oracle.route(x, W_r, c["k"], bias)
        assert np.array_equal(got["topk_idx"].cpu().numpy(), o["idx"])
        assert mok.device_status(None) == (mok.OK, 0)


@pytest.mark.gpu
def test_static_scratch_calls_leave_device_memory_unchanged():
    """After the first call (which looks up the array's address), further
    calls allocate nothing: the device's free memory does not move."""
    T, H, E, k = 2560, 7168, 32, 8
    x, W_r, _ = _inputs(T, H, E, 3)
    xd, wd = to_dev_bf16(x), dev_f32(W_r)
    out = mok.route_layout_static(xd, wd, k)           # first call: outputs allocated here
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        mok.route_layout_static(xd, wd, k, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert mok.device_status(None) == (mok.OK, 0)


@pytest.mark.gpu
def test_static_scratch_reports_a_router_wait_that_gave_up():
    """The status block of the library's array is readable through
    mok_device_status(NULL): a router copy withheld by the test hook makes a
    wait run out, the call reports MOK_ERR_TIMEOUT (detail 7, the router's
    chunk wait) and still returns valid routing arrays; the next call without
    the hook clears the report and routes correctly again."""
    T, H, E, k = 1000, 7168, 32, 8
    x, W_r, _ = _inputs(T, H, E, 4)
    xd, wd = to_dev_bf16(x), dev_f32(W_r)
    mok.route_test_hook(1, timeout_ms=50)
    try:
        got = mok.route_layout_static(xd, wd, k)
        torch.cuda.synchronize()
        assert mok.device_status(None) == (mok.ERR_TIMEOUT, 7)
        # the withheld CTA's tokens fall back to the lowest-index experts, so
        # the arrays stay a valid layout
        idx = got["topk_idx"].cpu().numpy()
        assert idx.min() >= 0 and idx.max() < E
        assert all(len(set(row)) == k for row in idx.tolist())
        assert int(got["counts"].sum()) == T * k
    finally:
        mok.route_test_hook(0, 0)
    ref = mok.route_layout(xd, wd, k)
    got = mok.route_layout_static(xd, wd, k)
    torch.cuda.synchronize()
    assert mok.device_status(None) == (mok.OK, 0)
    assert torch.equal(got["topk_idx"], ref["topk_idx"])
    assert torch.equal(got["row_src"][:T * k], ref["row_src"][:T * k])


@pytest.mark.gpu
def test_static_scratch_rejects_problems_beyond_its_size():
    # E * H * 4 bytes of transposed router weights alone exceed 8 MiB here
    T, H, E, k = 64, 16384, 256, 2
    assert mok.route_workspace_size(T, H, E, k) > mok.ROUTE_STATIC_SCRATCH_BYTES
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    W_r = torch.zeros((H, E), dtype=torch.float32, device="cuda")
    with pytest.raises(mok.MokError) as ei:
        mok.route_layout_static(x, W_r, k)
    assert ei.value.code == mok.ERR_INVALID
