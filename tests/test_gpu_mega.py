"""The persistent forward megakernel (mover / compute SM split, GPU-local
counters, minibatches through a two-region ring).

It runs the same tile shapes and the same arithmetic as the staged kernels,
so its output must be bit-identical to theirs for every minibatch size, ring
size and mover count (the result must not depend on how the work is cut),
and within tolerance of the oracle."""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import TOL, assert_close, dtype_of, host_bf16_f64, layer_for, to_dev_bf16

CASES = [
    synth.small("mega_bf16", T=1000, H=512, I=256, E=8, k=2),
    synth.small("mega_bf16_skew", T=600, H=256, I=2048, E=8, k=4, zipf_s=1.2),
    synth.small("mega_mx", T=1000, H=512, I=256, E=8, k=2, dtype="mxfp8", zipf_s=1.2),
    synth.small("mega_mx_k8", T=300, H=1024, I=512, E=32, k=8, dtype="mxfp8"),
    synth.small("mega_mx_h896", T=700, H=896, I=256, E=8, k=2, dtype="mxfp8", zipf_s=1.2),
]


def _forward(layer, x, cfg, T):
    cfg.flags |= mok.FLAG_MEGAKERNEL
    p = layer.problem(T)
    b = layer.buffers(T)
    ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
    out = torch.empty((T, layer.H), dtype=torch.bfloat16, device="cuda")
    mok.moe_forward(p, x, layer.packed, b["routing"], out, ws, packed_shared=layer.packed_shared, cfg=cfg)
    torch.cuda.synchronize()
    return out, mok.device_status(ws)


def _staged(layer, x, T):
    """The stage kernels on 128-row token tiles, the tile shapes the
    megakernel runs."""
    p = layer.problem(T)
    cfg = mok.make_config(flags=mok.FLAG_ROW_TILES)
    ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
    out = torch.empty((T, layer.H), dtype=torch.bfloat16, device="cuda")
    mok.moe_forward(p, x, layer.packed, layer.buffers(T)["routing"], out, ws, packed_shared=layer.packed_shared,
                    cfg=cfg)
    torch.cuda.synchronize()
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_megakernel_matches_staged_bitwise_and_oracle(wl):
    inp = synth.make_inputs(wl)
    dt = dtype_of(wl)
    layer = layer_for(inp, dt)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    ref = _staged(layer, x, wl.T)
    out, st = _forward(layer, x, mok.make_config(), wl.T)
    assert st == (mok.OK, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    mode = oracle.MODE_MXFP8 if dt == mok.MXFP8 else oracle.MODE_BF16
    o = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=mode)
    assert_close(host_bf16_f64(out), o, TOL[dt], wl.name)


@pytest.mark.gpu
@pytest.mark.parametrize("wl", [CASES[0], CASES[2]], ids=["bf16", "mxfp8"])
def test_megakernel_independent_of_minibatch_ring_and_movers(wl):
    inp = synth.make_inputs(wl, seed=7)
    layer = layer_for(inp, dtype_of(wl))
    x = to_dev_bf16(inp.x)
    layer.route(x)
    ref = _staged(layer, x, wl.T)
    configs = [
        mok.make_config(minibatch_tokens=64),                        # many minibatches, both regions reused
        mok.make_config(minibatch_tokens=160, ring_rows=2 * 1536),   # ring forces the cut
        mok.make_config(mover_ctas=1),
        mok.make_config(mover_ctas=24, minibatch_tokens=300),
        # token-range minibatches: each pads its experts' rows separately
        mok.make_config(minibatch_tokens=64, flags=mok.FLAG_MB_TOKEN_RANGES),
        mok.make_config(minibatch_tokens=160, ring_rows=2 * 1536, flags=mok.FLAG_MB_TOKEN_RANGES),
    ]
    for cfg in configs:
        out, st = _forward(layer, x, cfg, wl.T)
        what = (cfg.minibatch_tokens, cfg.ring_rows, cfg.mover_ctas, cfg.flags)
        assert st == (mok.OK, 0), (what, st)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), what


@pytest.mark.gpu
def test_megakernel_bitwise_reruns():
    wl = CASES[2]
    inp = synth.make_inputs(wl, seed=9)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    cfg = mok.make_config(minibatch_tokens=128)
    first, _ = _forward(layer, x, cfg, wl.T)
    for _ in range(9):
        again, st = _forward(layer, x, cfg, wl.T)
        assert st == (mok.OK, 0)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("cut_flags", [0, mok.FLAG_MB_TOKEN_RANGES], ids=["tile_cuts", "token_ranges"])
def test_macro_batches_through_one_ring_with_shared_expert(cut_flags):
    """Several macro-batches (own tokens, same weights) stream through one
    launch and a small ring; each output equals that batch's staged forward,
    shared BF16 expert included."""
    wl = synth.small("stream", T=400, H=512, I=256, E=8, k=2, dtype="mxfp8", zipf_s=1.2, shared_I=256,
                     batches=3)
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.MXFP8)
    xs = [to_dev_bf16(x) for x in inp.xs]
    routings, refs = [], []
    for x in xs:
        r = layer.route(x)
        routings.append({n: v.clone() for n, v in r.items()})
        refs.append(_staged(layer, x, wl.T).clone())
    p = layer.problem(wl.T)
    cfg = mok.make_config(ring_rows=2 * 1024, minibatch_tokens=128, flags=cut_flags)
    ws = mok.alloc_bytes(mok.workspace_size_batches(p, len(xs), cfg))
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda") for _ in xs]
    mok.moe_forward_batches(p, xs, layer.packed, routings, outs, ws, packed_shared=layer.packed_shared, cfg=cfg)
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    for b in range(len(xs)):
        assert torch.equal(outs[b].view(torch.int16), refs[b].view(torch.int16)), b
    r = oracle.route(inp.xs[1], inp.W_r, wl.k, inp.bias)
    o = oracle.moe_forward(inp.xs[1], inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_MXFP8, shared=inp.shared)
    assert_close(host_bf16_f64(outs[1]), o, TOL[mok.MXFP8], "batch 1")


@pytest.mark.gpu
def test_ring_of_one_tile():
    """A ring region of one 128-row tile: token-range minibatches cannot hold
    a 16-token block's padded rows (capacity error, device still usable);
    expert-tile runs still fit, one tile per minibatch."""
    wl = CASES[0]
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    out, st = _forward(layer, x, mok.make_config(ring_rows=2 * 128, flags=mok.FLAG_MB_TOKEN_RANGES), wl.T)
    assert st[0] == mok.ERR_CAPACITY
    ref = _staged(layer, x, wl.T)       # the device is still usable
    for cfg in (mok.make_config(), mok.make_config(ring_rows=2 * 128)):
        out, st = _forward(layer, x, cfg, wl.T)
        assert st == (mok.OK, 0) and torch.equal(out.view(torch.int16), ref.view(torch.int16)), cfg.ring_rows


@pytest.mark.gpu
def test_too_many_minibatches_reports_capacity():
    """Expert-tile runs of one tile each: 40000 tokens x 2 rows need more
    than 512 minibatches per macro-batch, which the plan refuses."""
    wl = synth.small("mega_many_mb", T=40000, H=128, I=128, E=8, k=2)
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    out, st = _forward(layer, x, mok.make_config(ring_rows=2 * 128), wl.T)
    assert st[0] == mok.ERR_CAPACITY
    ref = _staged(layer, x, wl.T)
    out, st = _forward(layer, x, mok.make_config(), wl.T)
    assert st == (mok.OK, 0) and torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
def test_withheld_publish_times_out_cleanly():
    """A mover that never publishes one chunk: the waiting tiles give up
    after timeout_ms, the call reports MOK_ERR_TIMEOUT, nothing hangs, and the
    next call works."""
    wl = CASES[0]
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    cfg = mok.make_config(timeout_ms=300, flags=mok.FLAG_TEST_WITHHOLD_PUBLISH)
    out, st = _forward(layer, x, cfg, wl.T)
    assert st[0] == mok.ERR_TIMEOUT
    ref = _staged(layer, x, wl.T)
    out, st = _forward(layer, x, mok.make_config(), wl.T)
    assert st == (mok.OK, 0) and torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("cut_flags", [0, mok.FLAG_MB_TOKEN_RANGES], ids=["tile_cuts", "token_ranges"])
def test_trace_records_and_unchanged_output(cut_flags):
    """MOK_FLAG_TRACE: one record per CTA (movers first), ordered timestamps,
    every gate/up and down tile counted once, output bit-identical."""
    wl = CASES[2]
    inp = synth.make_inputs(wl, seed=3)
    layer = layer_for(inp, mok.MXFP8)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    ref = _staged(layer, x, wl.T)
    movers = 8
    cfg = mok.make_config(mover_ctas=movers, minibatch_tokens=256, flags=mok.FLAG_TRACE | cut_flags)
    cfg.flags |= mok.FLAG_MEGAKERNEL
    p = layer.problem(wl.T)
    ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
    out = torch.empty((wl.T, layer.H), dtype=torch.bfloat16, device="cuda")
    mok.moe_forward(p, x, layer.packed, layer.buffers(wl.T)["routing"], out, ws, packed_shared=layer.packed_shared,
                    cfg=cfg)
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    n = torch.cuda.get_device_properties(0).multi_processor_count
    rec = mok.megakernel_trace(ws, n)
    assert np.all(rec[:movers, 0] == 0) and np.all(rec[movers:, 0] == 1)
    assert np.all(rec[:, 1] <= rec[:, 4]) and np.all(rec[:, 3] <= rec[:, 4])
    # waiting and weighted sums are disjoint spans of the CTA's lifetime
    assert np.all(rec[:, 5] + rec[:, 7] <= rec[:, 4] - rec[:, 1] + 2000)
    work = rec[:, 6] > 0
    assert np.all(rec[work, 1] <= rec[work, 2]) and np.all(rec[work, 2] <= rec[work, 3])
    counts = layer.buffers(wl.T)["routing"]["counts"].cpu().numpy()
    n_mb = int(np.max(rec[:movers, 6]))
    assert n_mb >= 2   # 1000 tokens in minibatches of at most 256
    # down tiles: 256 wide when H allows, else 224, else 128 (MXFP8)
    bn2 = 256 if wl.H % 256 == 0 else 224 if wl.H % 224 == 0 else 128
    nt1, nt2 = 2 * wl.I // 256, wl.H // bn2
    mtiles = int(np.sum((counts + 127) // 128))
    tiles_min = mtiles * (nt1 + nt2)
    if cut_flags:
        # token ranges: tiles per minibatch sum to at least the whole batch's,
        # since each minibatch pads its experts' rows separately
        assert int(rec[movers:, 6].sum()) >= tiles_min
    else:
        # tile cuts: exactly the staged GEMMs' tiles, in runs of at most
        # 256 * k rows
        assert int(rec[movers:, 6].sum()) == tiles_min
        assert n_mb == -(-mtiles // -(-256 * wl.k // 128))
