"""Full-size layers (H=7168, I=2048, E=32, k=8) against the oracle.

Routing is compared bit for bit over every token; layer outputs on sampled
tokens the oracle computes one by one; weight gradients on sampled columns;
determinism over ten reruns. These run the same kernels bench.py times.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import TOL, assert_close, dtype_of, host_bf16_f64, layer_for, to_dev_bf16


def _sample_tokens(T, n=24, seed=0):
    rng = np.random.default_rng(seed)
    s = set([0, T - 1]) | set(rng.choice(T, n - 2, replace=False).tolist())
    return np.array(sorted(s), dtype=np.int32)


def _check_routing(layer, ref, T, k):
    g = {n: v.cpu().numpy() for n, v in layer.buffers(T)["routing"].items()}
    assert np.array_equal(g["topk_idx"], ref["idx"])
    assert np.array_equal(g["counts"], ref["counts"])
    assert np.array_equal(g["offsets"], ref["offsets"])
    assert np.array_equal(g["row_src"][:T * k], ref["row_src"])
    assert np.array_equal(g["slot_row"][:T * k], ref["slot_row"])
    assert np.max(np.abs(g["topk_w"].astype(np.float64) - ref["w"])) <= 1e-6


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["bf16_fwd_T2560", "mxfp8_zipf_T512", "mxfp8_zipf_T2560", "mxfp8_zipf_T4096",
                                  "mxfp8_zipf_T8192"])
def test_fullsize_forward(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl)
    dt = dtype_of(wl)
    layer = layer_for(inp, dt)
    x = to_dev_bf16(inp.x)
    out = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert layer.status(wl.T) == (mok.OK, 0)
    ref_r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    _check_routing(layer, ref_r, wl.T, wl.k)
    toks = _sample_tokens(wl.T)
    mode = oracle.MODE_MXFP8 if dt == mok.MXFP8 else oracle.MODE_BF16
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, ref_r, mode=mode, tokens=toks)
    assert_close(host_bf16_f64(out[toks]), ref, TOL[dt], name)
    for _ in range(9):
        again = layer.forward(x)
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))


@pytest.mark.gpu
def test_fullsize_backward_T4096():
    wl = synth.WORKLOADS["bf16_bwd_T4096"]
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    dY = to_dev_bf16(inp.dY)
    layer.forward(x, training=True)
    g = layer.backward(x, dY)
    torch.cuda.synchronize()
    assert layer.status(wl.T, training=True) == (mok.OK, 0)
    r = oracle.route(inp.x, inp.W_r, wl.k)
    toks = _sample_tokens(wl.T, n=6, seed=1)
    rng = np.random.default_rng(2)
    cols = [(int(e), int(i)) for e, i in zip(rng.integers(0, wl.E, 6), rng.integers(0, wl.I, 6))]
    sX, sG, sU, sD = oracle.moe_backward_sampled(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, toks, cols)
    c = TOL[mok.BF16]
    assert_close(host_bf16_f64(g["dX"][toks]), sX, c, "dX")
    gG = np.stack([host_bf16_f64(g["dW_gate"][e, :, i]) for e, i in cols])
    gU = np.stack([host_bf16_f64(g["dW_up"][e, :, i]) for e, i in cols])
    gD = np.stack([host_bf16_f64(g["dW_down"][e, i, :]) for e, i in cols])
    assert_close(gG, sG, c, "dW_gate columns")
    assert_close(gU, sU, c, "dW_up columns")
    assert_close(gD, sD, c, "dW_down rows")
    # router gradient: each row of dW_r sums to zero (sum_j dl_j = 0 per token),
    # and the column of the least-loaded expert against the oracle's column
    dWr = g["dW_r"].double().cpu().numpy()
    assert np.max(np.abs(dWr.sum(1))) <= 1e-4 * np.abs(dWr).max() * wl.E
    e_min = int(np.argmin(r["counts"]))
    col = oracle.router_grad_columns(inp.x, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, [e_min])
    assert_close(dWr[:, e_min][None], col, c, f"dW_r[:, {e_min}]", bf16_out=False)
    # bitwise determinism of every gradient over ten runs
    first = {n: t.clone() for n, t in g.items()}
    for _ in range(9):
        layer.forward(x, training=True)
        again = layer.backward(x, dY)
        for n in first:
            assert torch.equal(again[n].view(torch.uint8), first[n].view(torch.uint8)), n


@pytest.mark.gpu
def test_fullsize_ring_stream_16x4096():
    """The 16-batch stream (T=4096 each, MXFP8 routed experts with Zipf-skewed
    routing, one BF16 shared expert, a ring of 16384 rows = half the
    worst-case routed rows) through one megakernel launch, as bench.py times
    it: routing of the first and last batch bit for bit, sampled tokens of
    both against the oracle (shared expert included), and a rerun bit for
    bit."""
    wl = synth.WORKLOADS["ring_stream_16x4096"]
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.MXFP8)
    xs = [to_dev_bf16(xb) for xb in inp.xs]
    routings = []
    for xb in xs:
        routings.append({n: v.clone() for n, v in layer.route(xb).items()})
    p = layer.problem(wl.T)
    cfg = mok.make_config(ring_rows=wl.ring_rows)
    ws = mok.alloc_bytes(mok.workspace_size_batches(p, len(xs), cfg))
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda") for _ in xs]
    mok.moe_forward_batches(p, xs, layer.packed, routings, outs, ws, packed_shared=layer.packed_shared, cfg=cfg)
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    first = [o.clone() for o in outs]
    mok.moe_forward_batches(p, xs, layer.packed, routings, outs, ws, packed_shared=layer.packed_shared, cfg=cfg)
    torch.cuda.synchronize()
    for b in range(len(xs)):
        assert torch.equal(outs[b].view(torch.int16), first[b].view(torch.int16)), b
    xsel, got = [], []
    for b in (0, len(xs) - 1):
        ref_r = oracle.route(inp.xs[b], inp.W_r, wl.k, inp.bias)
        g = {n: v.cpu().numpy() for n, v in routings[b].items()}
        assert np.array_equal(g["topk_idx"], ref_r["idx"])
        assert np.array_equal(g["counts"], ref_r["counts"])
        assert np.array_equal(g["row_src"][:wl.R], ref_r["row_src"])
        toks = _sample_tokens(wl.T, n=8, seed=b)
        xsel.append(inp.xs[b][toks])
        got.append(host_bf16_f64(first[b][toks]))
    # each token's output depends on that token alone: route and run the
    # sampled tokens of both batches as one small batch through the oracle
    xcat = np.ascontiguousarray(np.concatenate(xsel))
    r = oracle.route(xcat, inp.W_r, wl.k, inp.bias)
    ref = oracle.moe_forward(xcat, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_MXFP8, shared=inp.shared)
    assert_close(np.concatenate(got), ref, TOL[mok.MXFP8], "ring stream, batches 0 and 15")


@pytest.mark.gpu
def test_fullsize_mxfp8_backward_T4096():
    """The MXFP8 training step at T=4096 (H=7168, I=2048, E=32, k=8): sampled
    dX rows and weight-gradient columns against the oracle's MXFP8 backward,
    and ten bitwise reruns."""
    wl = synth.WORKLOADS["mxfp8_bwd_T4096"]
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    dY = to_dev_bf16(inp.dY)
    layer.forward(x, training=True)
    g = layer.backward(x, dY)
    torch.cuda.synchronize()
    assert layer.status(wl.T, training=True) == (mok.OK, 0)
    r = oracle.route(inp.x, inp.W_r, wl.k)
    toks = _sample_tokens(wl.T, n=4, seed=3)
    rng = np.random.default_rng(4)
    cols = [(int(e), int(i)) for e, i in zip(rng.integers(0, wl.E, 4), rng.integers(0, wl.I, 4))]
    sX, sG, sU, sD = oracle.moe_backward_sampled(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, toks, cols,
                                                 mode=oracle.MODE_MXFP8)
    c = TOL[mok.MXFP8]
    assert_close(host_bf16_f64(g["dX"][toks]), sX, c, "dX (MXFP8)")
    gG = np.stack([host_bf16_f64(g["dW_gate"][e, :, i]) for e, i in cols])
    gU = np.stack([host_bf16_f64(g["dW_up"][e, :, i]) for e, i in cols])
    gD = np.stack([host_bf16_f64(g["dW_down"][e, i, :]) for e, i in cols])
    assert_close(gG, sG, c, "dW_gate columns (MXFP8)")
    assert_close(gU, sU, c, "dW_up columns (MXFP8)")
    assert_close(gD, sD, c, "dW_down rows (MXFP8)")
    first = {n: t.clone() for n, t in g.items()}
    for _ in range(9):
        layer.forward(x, training=True)
        again = layer.backward(x, dY)
        for n in first:
            assert torch.equal(again[n].view(torch.uint8), first[n].view(torch.uint8)), n
