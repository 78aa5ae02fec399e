"""Backward layer on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import TOL, assert_close, host_bf16_f64, layer_for, to_dev_bf16

BWD_CASES = [
    synth.small("bwd_tiny", T=64, H=128, I=64, E=8, k=2, backward=True),
    synth.small("bwd_ragged", T=500, H=512, I=256, E=4, k=2, backward=True),
    synth.small("bwd_skew", T=300, H=256, I=512, E=8, k=4, zipf_s=1.2, backward=True),
    # one expert, k = 1: a dense SwiGLU FFN (router gradient is zero)
    synth.small("bwd_dense", T=130, H=256, I=128, E=1, k=1, backward=True),
    # k = E: every token through every expert
    synth.small("bwd_all_experts", T=96, H=256, I=128, E=4, k=4, backward=True),
]


def _run(wl, seed=0):
    inp = synth.make_inputs(wl, seed=seed)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    dY = to_dev_bf16(inp.dY)
    out = layer.forward(x, training=True).clone()
    g = layer.backward(x, dY)
    torch.cuda.synchronize()
    assert layer.status(wl.T, training=True) == (mok.OK, 0)
    return inp, layer, x, dY, out, g


@pytest.mark.gpu
@pytest.mark.parametrize("wl", BWD_CASES, ids=[w.name for w in BWD_CASES])
def test_backward_matches_oracle(wl):
    inp, layer, x, dY, out, g = _run(wl)
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    ref_out = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16)
    assert_close(host_bf16_f64(out), ref_out, TOL[mok.BF16], "out")
    dX, dWg, dWu, dWd, dWr = oracle.moe_backward(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r,
                                                  mode=oracle.MODE_BF16)
    c = TOL[mok.BF16]
    assert_close(host_bf16_f64(g["dX"]), dX, c, "dX")
    assert_close(host_bf16_f64(g["dW_gate"]), dWg, c, "dW_gate")
    assert_close(host_bf16_f64(g["dW_up"]), dWu, c, "dW_up")
    assert_close(host_bf16_f64(g["dW_down"]), dWd, c, "dW_down")
    assert_close(g["dW_r"].cpu().numpy().astype(np.float64), dWr, c, "dW_r", bf16_out=False)


@pytest.mark.gpu
def test_backward_bitwise_deterministic():
    wl = BWD_CASES[1]
    inp, layer, x, dY, out, g = _run(wl, seed=2)
    first = {n: t.clone() for n, t in g.items()}
    for _ in range(9):
        layer.forward(x, training=True)
        again = layer.backward(x, dY)
        for n in first:
            assert torch.equal(again[n].view(torch.uint8), first[n].view(torch.uint8)), n


@pytest.mark.gpu
def test_router_gradient_rows_sum_to_zero():
    """sum_e dW_r[h, e] = sum_t x[t,h] sum_j dl[t,j] = 0 because
    sum_j w_j (gw_j - sum_i w_i gw_i) = 0 - a property at any size."""
    wl = BWD_CASES[2]
    inp, layer, x, dY, out, g = _run(wl, seed=5)
    dWr = g["dW_r"].double().cpu().numpy()
    scale = np.abs(dWr).max()
    assert np.max(np.abs(dWr.sum(1))) <= 1e-4 * scale * wl.E


MX_BWD_CASES = [
    synth.small("mxbwd_small", T=256, H=256, I=128, E=4, k=2, dtype="mxfp8", backward=True),
    synth.small("mxbwd_ragged", T=500, H=512, I=256, E=4, k=2, dtype="mxfp8", zipf_s=1.2, backward=True),
    synth.small("mxbwd_all_experts", T=96, H=256, I=128, E=4, k=4, dtype="mxfp8", backward=True),
    # H = 384: the down weight gradient's 384 columns take the 128-wide tiles,
    # the gate/up one's 256 columns the 256-wide tiles
    synth.small("mxbwd_h384", T=200, H=384, I=128, E=4, k=2, dtype="mxfp8", zipf_s=1.2, backward=True),
]


def _run_mx(wl, seed=0):
    inp = synth.make_inputs(wl, seed=seed)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    dY = to_dev_bf16(inp.dY)
    out_inf = layer.forward(x).clone()
    out = layer.forward(x, training=True).clone()
    g = layer.backward(x, dY)
    torch.cuda.synchronize()
    assert layer.status(wl.T, training=True) == (mok.OK, 0)
    return inp, layer, x, dY, out_inf, out, g


@pytest.mark.gpu
@pytest.mark.parametrize("wl", MX_BWD_CASES, ids=[w.name for w in MX_BWD_CASES])
def test_mxfp8_backward_matches_oracle(wl):
    """MXFP8 backward (every backward GEMM on MXFP8 operands blocked along
    its own reduction dimension) against the oracle's MXFP8 mode; the MXFP8
    training forward gives the inference forward's bits."""
    inp, layer, x, dY, out_inf, out, g = _run_mx(wl)
    assert torch.equal(out.view(torch.int16), out_inf.view(torch.int16))
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    dX, dWg, dWu, dWd, dWr = oracle.moe_backward(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r,
                                                  mode=oracle.MODE_MXFP8)
    c = TOL[mok.MXFP8]
    assert_close(host_bf16_f64(g["dX"]), dX, c, "dX (MXFP8)")
    assert_close(host_bf16_f64(g["dW_gate"]), dWg, c, "dW_gate (MXFP8)")
    assert_close(host_bf16_f64(g["dW_up"]), dWu, c, "dW_up (MXFP8)")
    assert_close(host_bf16_f64(g["dW_down"]), dWd, c, "dW_down (MXFP8)")
    assert_close(g["dW_r"].cpu().numpy().astype(np.float64), dWr, c, "dW_r (MXFP8)", bf16_out=False)


@pytest.mark.gpu
def test_mxfp8_backward_bitwise_deterministic():
    wl = MX_BWD_CASES[1]
    inp, layer, x, dY, out_inf, out, g = _run_mx(wl, seed=2)
    first = {n: t.clone() for n, t in g.items()}
    for _ in range(9):
        layer.forward(x, training=True)
        again = layer.backward(x, dY)
        for n in first:
            assert torch.equal(again[n].view(torch.uint8), first[n].view(torch.uint8)), n


@pytest.mark.gpu
def test_mxfp8_backward_weight_copies_packed_or_per_call():
    """The weights' MXFP8 backward copies packed once (mok_pack_weights_bwd)
    or quantised inside the call (packed_bwd NULL) give the same bits."""
    wl = MX_BWD_CASES[0]
    inp, layer, x, dY, out_inf, out, g = _run_mx(wl, seed=4)
    first = {n: t.clone() for n, t in g.items()}
    b = layer.buffers(wl.T, True)
    grads = {n: torch.empty_like(t) for n, t in first.items()}
    mok.moe_backward(layer.problem(wl.T), x, layer.W_r, layer.Wg, layer.Wu, layer.Wd, layer.packed, dY,
                     b["routing"], b["saved"], grads, b["ws"], packed_bwd=None)
    torch.cuda.synchronize()
    for n in first:
        assert torch.equal(grads[n].view(torch.uint8), first[n].view(torch.uint8)), n
