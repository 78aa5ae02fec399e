"""Forward layer on the GPU against the oracle (small and medium shapes)."""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import (TOL, assert_close, dtype_of, host_bf16_f64, layer_for, to_dev_bf16, untile_sf)

FWD_CASES = [
    # tiny layer of the pages' shape family, BF16
    synth.small("tiny", T=64, H=128, I=64, E=8, k=2),
    # several 128-row tiles per expert with ragged tails, BF16
    synth.small("ragged_bf16", T=1000, H=512, I=256, E=4, k=2),
    # wide expert (I=2048) at small H, skewed routing, BF16
    synth.small("skew_bf16", T=300, H=256, I=2048, E=8, k=2, zipf_s=1.2),
    # MXFP8 operands, skewed routing
    synth.small("ragged_mx", T=600, H=512, I=256, E=8, k=2, dtype="mxfp8", zipf_s=1.2),
    synth.small("mx_k8", T=200, H=1024, I=512, E=32, k=8, dtype="mxfp8"),
    # MXFP8 down GEMM on 224-wide tiles (H = 4 x 224), scales per 224-row tile
    synth.small("mx_h896", T=700, H=896, I=256, E=8, k=2, dtype="mxfp8", zipf_s=1.2),
    # BF16 shared expert added to MXFP8 routed experts
    synth.small("mx_shared", T=300, H=512, I=256, E=8, k=2, dtype="mxfp8", zipf_s=1.2, shared_I=256),
    # one token; one expert with k=1 (dense SwiGLU)
    synth.small("one_token", T=1, H=256, I=128, E=16, k=4),
    synth.small("dense", T=130, H=256, I=128, E=1, k=1),
    # more experts than tokens can fill: several experts get zero rows
    synth.small("sparse", T=8, H=256, I=128, E=64, k=1),
    # every token to every expert (k = E: the weights are the full softmax)
    synth.small("all_experts", T=100, H=256, I=128, E=4, k=4),
    # the largest expert count the routing kernels take (256), BF16 and MXFP8
    synth.small("e256", T=300, H=256, I=128, E=256, k=8, zipf_s=1.2),
    synth.small("mx_e256", T=200, H=512, I=128, E=256, k=4, dtype="mxfp8"),
]


def _oracle_mode(dtype):
    return oracle.MODE_MXFP8 if dtype == mok.MXFP8 else oracle.MODE_BF16


def _run_case(wl, seed=0):
    inp = synth.make_inputs(wl, seed=seed)
    dt = dtype_of(wl)
    layer = layer_for(inp, dt)
    x = to_dev_bf16(inp.x)
    out = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert layer.status(wl.T) == (mok.OK, 0)
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=_oracle_mode(dt), shared=inp.shared)
    return inp, layer, x, out, ref


@pytest.mark.gpu
@pytest.mark.parametrize("wl", FWD_CASES, ids=[w.name for w in FWD_CASES])
def test_forward_matches_oracle(wl):
    inp, layer, x, out, ref = _run_case(wl)
    assert_close(host_bf16_f64(out), ref, TOL[dtype_of(wl)], wl.name)


@pytest.mark.gpu
def test_forward_bitwise_deterministic():
    wl = synth.small("det", T=700, H=512, I=256, E=8, k=4, zipf_s=1.2)
    inp = synth.make_inputs(wl, seed=3)
    for dt in (mok.BF16, mok.MXFP8):
        layer = layer_for(inp, dt)
        x = to_dev_bf16(inp.x)
        first = layer.forward(x).clone()
        for _ in range(9):
            again = layer.forward(x)
            assert torch.equal(again.view(torch.int16), first.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("dt", [mok.BF16, mok.MXFP8])
def test_dispatch_bytes(dt):
    """The gather reproduces x rows (BF16) or the oracle's MXFP8 bytes and
    scales (MXFP8) bit for bit; pad rows are zero."""
    wl = synth.small("disp", T=333, H=1024, I=128, E=8, k=3, zipf_s=1.2)
    inp = synth.make_inputs(wl, seed=1)
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    layer = layer_for(inp, dt)
    x = to_dev_bf16(inp.x)
    rt = layer.route(x)
    p = layer.problem(wl.T)
    rows = mok.padded_rows_max(wl.T, wl.E, wl.k)
    if dt == mok.BF16:
        A = mok.alloc_bytes(rows * wl.H * 2).view(torch.bfloat16).view(rows, wl.H)
        mok.dispatch(p, x, rt, A)
    else:
        A = mok.alloc_bytes(rows * wl.H).view(rows, wl.H)
        A_sf = mok.alloc_bytes(rows * wl.H // 32)
        mok.dispatch(p, x, rt, A, A_sf)
    torch.cuda.synchronize()
    counts = r["counts"]
    poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    src_rows = np.full(poff[-1], -1)
    for e in range(wl.E):
        src_rows[poff[e]:poff[e] + counts[e]] = r["row_src"][r["offsets"][e]:r["offsets"][e + 1]] // wl.k
    live = src_rows >= 0
    if dt == mok.BF16:
        got = A[:poff[-1]].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got[live], inp.x[src_rows[live]])
        assert np.all(got[~live] == 0)
    else:
        codes, scales = oracle.mx_quantize_bf16_rows(inp.x)
        got = A[:poff[-1]].cpu().numpy()
        assert np.array_equal(got[live], codes[src_rows[live]])
        assert np.all(got[~live] == 0)
        sf = untile_sf(A_sf.cpu().numpy(), poff[-1], wl.H)
        assert np.array_equal(sf[live], scales[src_rows[live]])
        assert np.all(sf[~live] == 0)


@pytest.mark.gpu
def test_quantize_once_then_gather():
    """mok_quantize_rows gives the oracle's MXFP8 codes and scales per token;
    mok_dispatch_quantized then writes the same routed rows and scales as the
    quantising mok_dispatch."""
    wl = synth.small("disp_q", T=333, H=1024, I=128, E=8, k=3, zipf_s=1.2)
    inp = synth.make_inputs(wl, seed=2)
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    rt = layer.route(x)
    p = layer.problem(wl.T)
    xq = mok.alloc_bytes(wl.T * wl.H).view(wl.T, wl.H)
    xsf = mok.alloc_bytes(wl.T * wl.H // 32).view(wl.T, wl.H // 32)
    mok.quantize_rows(x, xq, xsf)
    torch.cuda.synchronize()
    codes, scales = oracle.mx_quantize_bf16_rows(inp.x)
    assert np.array_equal(xq.cpu().numpy(), codes)
    assert np.array_equal(xsf.cpu().numpy(), scales)
    rows = mok.padded_rows_max(wl.T, wl.E, wl.k)
    A1, A2 = mok.alloc_bytes(rows * wl.H).view(rows, wl.H), mok.alloc_bytes(rows * wl.H).view(rows, wl.H)
    S1, S2 = mok.alloc_bytes(rows * wl.H // 32), mok.alloc_bytes(rows * wl.H // 32)
    mok.dispatch(p, x, rt, A1, S1)
    mok.dispatch_quantized(p, xq, xsf, rt, A2, S2)
    torch.cuda.synchronize()
    counts = r["counts"]
    poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    live = np.zeros(poff[-1], bool)
    for e in range(wl.E):
        live[poff[e]:poff[e] + counts[e]] = True
    assert np.array_equal(A2[:poff[-1]].cpu().numpy()[live], A1[:poff[-1]].cpu().numpy()[live])
    sf1 = untile_sf(S1.cpu().numpy(), poff[-1], wl.H)
    sf2 = untile_sf(S2.cpu().numpy(), poff[-1], wl.H)
    assert np.array_equal(sf2[live], sf1[live])
    # the one-pass token-major dispatch writes the same routed bytes and scales
    A3, S3 = mok.alloc_bytes(rows * wl.H).view(rows, wl.H), mok.alloc_bytes(rows * wl.H // 32)
    mok.dispatch_tokens(p, x, rt, A3, S3)
    torch.cuda.synchronize()
    assert np.array_equal(A3[:poff[-1]].cpu().numpy()[live], A1[:poff[-1]].cpu().numpy()[live])
    assert np.array_equal(untile_sf(S3.cpu().numpy(), poff[-1], wl.H)[live], sf1[live])
    with pytest.raises(mok.MokError):
        mok.quantize_rows(x[:, :1000], xq, xsf)     # H % 128 != 0


@pytest.mark.gpu
def test_token_major_dispatch_many_slots():
    """k = 40 > 32 slots per token (each slot's row looked up directly rather
    than shuffled from lane j): the same routed bytes as mok_dispatch."""
    wl = synth.small("disp_k40", T=50, H=256, I=128, E=64, k=40)
    inp = synth.make_inputs(wl, seed=3)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    rt = layer.route(x)
    p = layer.problem(wl.T)
    rows = mok.padded_rows_max(wl.T, wl.E, wl.k)
    A1, A3 = mok.alloc_bytes(rows * wl.H).view(rows, wl.H), mok.alloc_bytes(rows * wl.H).view(rows, wl.H)
    S1, S3 = mok.alloc_bytes(rows * wl.H // 32), mok.alloc_bytes(rows * wl.H // 32)
    mok.dispatch(p, x, rt, A1, S1)
    mok.dispatch_tokens(p, x, rt, A3, S3)
    torch.cuda.synchronize()
    counts = rt["counts"].cpu().numpy()
    poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    live = np.zeros(poff[-1], bool)
    for e in range(wl.E):
        live[poff[e]:poff[e] + counts[e]] = True
    assert np.array_equal(A3[:poff[-1]].cpu().numpy()[live], A1[:poff[-1]].cpu().numpy()[live])
    assert np.array_equal(untile_sf(S3.cpu().numpy(), poff[-1], wl.H)[live],
                          untile_sf(S1.cpu().numpy(), poff[-1], wl.H)[live])


@pytest.mark.gpu
def test_stages_compose_to_forward():
    """dispatch -> expert_ffn -> combine gives the same bits as moe_forward."""
    wl = synth.small("stages", T=256, H=512, I=256, E=8, k=2, dtype="mxfp8")
    inp = synth.make_inputs(wl, seed=4)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    full = layer.forward(x).clone()
    rt = layer.buffers(wl.T)["routing"]
    p = layer.problem(wl.T)
    rows = mok.padded_rows_max(wl.T, wl.E, wl.k)
    A = mok.alloc_bytes(rows * wl.H)
    A_sf = mok.alloc_bytes(rows * wl.H // 32)
    h = mok.alloc_bytes(rows * wl.I)
    h_sf = mok.alloc_bytes(rows * wl.I // 32)
    part = torch.empty((wl.T * wl.k, wl.H), dtype=torch.bfloat16, device="cuda")
    ws = mok.alloc_bytes(256)
    out = torch.empty_like(full)
    mok.dispatch(p, x, rt, A, A_sf)
    mok.expert_ffn(p, A, A_sf, layer.packed, rt, h, h_sf, part, ws)
    mok.combine(p, part, rt["topk_w"], out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_stages_behind_a_producer_kernel_on_the_stream(dtype):
    """The library's kernels are launched with programmatic stream
    serialization: each waits for the kernel before it on the stream before
    touching memory. Here a torch kernel rewrites x on the stream right before
    routing and the stages run, with no synchronisation in between, for
    alternating inputs; every output must equal the one computed after a
    full synchronisation."""
    wl = synth.small("pdl", T=512, H=1024, I=256, E=8, k=2, dtype=dtype)
    inp = synth.make_inputs(wl, seed=21)
    mode = mok.MXFP8 if dtype == "mxfp8" else mok.BF16
    layer = layer_for(inp, mode)
    g = torch.Generator().manual_seed(3)
    xs = [to_dev_bf16(synth._normal_bf16(g, (wl.T, wl.H), 1.0)) for _ in range(2)]
    refs = []
    for xv in xs:
        refs.append(layer.forward(xv.clone()).clone())
        torch.cuda.synchronize()
    p = layer.problem(wl.T)
    rt = layer.buffers(wl.T)["routing"]
    rows = mok.padded_rows_max(wl.T, wl.E, wl.k)
    eb = 1 if dtype == "mxfp8" else 2
    A = mok.alloc_bytes(rows * wl.H * eb)
    A_sf = mok.alloc_bytes(rows * wl.H // 32) if dtype == "mxfp8" else None
    h = mok.alloc_bytes(rows * wl.I * eb)
    h_sf = mok.alloc_bytes(rows * wl.I // 32) if dtype == "mxfp8" else None
    part = torch.empty((wl.T * wl.k, wl.H), dtype=torch.bfloat16, device="cuda")
    ws = mok.alloc_bytes(256)
    x = torch.empty_like(xs[0])
    outs = [torch.empty_like(refs[0]) for _ in range(20)]
    for i in range(20):
        x.copy_(xs[i % 2])                       # a torch kernel writes the input
        layer.route(x)                            # ... and the routing reads it
        if dtype == "mxfp8":
            mok.dispatch_tokens(p, x, rt, A, A_sf)
        else:
            mok.dispatch(p, x, rt, A, None)
        mok.expert_ffn(p, A, A_sf, layer.packed, rt, h, h_sf, part, ws)
        mok.combine(p, part, rt["topk_w"], outs[i])
        x.zero_()                                 # and is overwritten behind them
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    for i in range(20):
        assert torch.equal(outs[i].view(torch.int16), refs[i % 2].view(torch.int16)), i


@pytest.mark.gpu
def test_invalid_arguments_rejected_on_host():
    wl = synth.small("inv", T=16, H=256, I=128, E=4, k=2)
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    b = layer.buffers(wl.T)
    p = mok.make_problem(wl.T, wl.H, wl.I, wl.E, 9, mok.BF16)  # k > E
    with pytest.raises(mok.MokError) as ei:
        mok.moe_forward(p, x, layer.packed, b["routing"], b["out"], b["ws"])
    assert ei.value.code == mok.ERR_INVALID
    small_ws = b["ws"][:1024]
    with pytest.raises(mok.MokError) as ei:
        mok.moe_forward(layer.problem(wl.T), x, layer.packed, b["routing"], b["out"], small_ws)
    assert ei.value.code == mok.ERR_INVALID
    # a backward with a shared expert is not built
    p_sh = mok.make_problem(wl.T, wl.H, wl.I, wl.E, wl.k, mok.BF16, 128)
    g = {n: torch.empty(1, device="cuda") for n in ("dX", "dW_gate", "dW_up", "dW_down", "dW_r")}
    with pytest.raises(mok.MokError) as ei:
        mok.moe_backward(p_sh, x, layer.W_r, layer.Wg, layer.Wu, layer.Wd, layer.packed, x, b["routing"], b["ws"], g,
                         b["ws"])
    assert ei.value.code == mok.ERR_UNSUPPORTED


@pytest.mark.gpu
def test_empty_batch():
    """T = 0: routing yields zero counts and offsets, forward and training
    forward + backward run no tile and report MOK_OK."""
    wl = synth.small("empty", T=8, H=256, I=128, E=4, k=2)
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x0 = torch.empty((0, wl.H), dtype=torch.bfloat16, device="cuda")
    r = layer.route(x0)
    torch.cuda.synchronize()
    assert int(r["counts"].abs().sum()) == 0 and int(r["offsets"].abs().sum()) == 0
    out = layer.forward(x0, route=False)
    torch.cuda.synchronize()
    assert out.shape[0] == 0 and layer.status(0) == (mok.OK, 0)
    layer.forward(x0, training=True)
    g = layer.backward(x0, torch.empty_like(x0))
    torch.cuda.synchronize()
    assert layer.status(0, training=True) == (mok.OK, 0)
    assert g["dX"].shape[0] == 0
    # nothing routed: every weight gradient is zero
    for n in ("dW_gate", "dW_up", "dW_down", "dW_r"):
        assert float(g[n].float().abs().max()) == 0.0, n
