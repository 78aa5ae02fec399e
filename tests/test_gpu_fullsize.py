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
@pytest.mark.parametrize("name", ["bf16_fwd_T2560", "mxfp8_zipf_T512", "mxfp8_zipf_T8192"])
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
    # router gradient: each row of dW_r sums to zero (sum_j dl_j = 0 per token)
    dWr = g["dW_r"].double().cpu().numpy()
    assert np.max(np.abs(dWr.sum(1))) <= 1e-4 * np.abs(dWr).max() * wl.E
    # bitwise determinism of every gradient
    first = {n: t.clone() for n, t in g.items()}
    layer.forward(x, training=True)
    again = layer.backward(x, dY)
    for n in first:
        assert torch.equal(again[n].view(torch.uint8), first[n].view(torch.uint8)), n
