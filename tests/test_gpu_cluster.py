"""Grouped GEMMs as 2-SM CTA pairs (tcgen05 cta_group::2: one M=256 MMA over
two CTAs' 128-row A halves and 128-row B halves) against the single-CTA
kernels. Every output element is still one K-ordered tensor-core dot product
with fp32 accumulation, so the results must be bit-identical. Experts with
an odd number of 128-row tiles exercise the last pair: in BF16 it shares the
expert's last tile as an M=128 pair MMA (64 rows per CTA, the accumulator
spread over all 128 lanes with half the columns each); the MXFP8 gate/up
pairs leave its second half idle (rows outside the expert must not be
written)."""
import pytest
import torch

from combine_router_top_expert_gb300 import mok, synth
from helpers import dtype_of, layer_for, to_dev_bf16


def _staged(layer, x, T, extra=0):
    p = layer.problem(T)
    cfg = mok.make_config(flags=extra)
    ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
    out = torch.empty((T, layer.H), dtype=torch.bfloat16, device="cuda")
    mok.moe_forward(p, x, layer.packed, layer.buffers(T)["routing"], out, ws, packed_shared=layer.packed_shared,
                    cfg=cfg)
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("wl", [
    synth.small("cl_bf16", T=700, H=512, I=256, E=8, k=2, zipf_s=1.2, shared_I=256),
    synth.small("cl_bf16_odd", T=600, H=768, I=512, E=4, k=2),
    synth.small("cl_mx", T=700, H=1024, I=256, E=8, k=4, dtype="mxfp8", zipf_s=1.2),
], ids=["bf16_shared", "bf16_odd_tiles", "mxfp8"])
def test_cluster_pairs_forward_bitwise(wl):
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, dtype_of(wl))
    x = to_dev_bf16(inp.x)
    layer.route(x)
    pairs = _staged(layer, x, wl.T, mok.FLAG_GEMM_PAIRS)
    single = _staged(layer, x, wl.T, mok.FLAG_ROW_TILES)
    assert torch.equal(pairs.view(torch.int16), single.view(torch.int16))


@pytest.mark.gpu
def test_cluster_pairs_backward_bitwise():
    # about 300 rows per expert: three 128-row tiles, so the last pair of every
    # GEMM (training gate/up with G|U saved, down, both dgrads) is an M=128 pair
    wl = synth.small("cl_bwd", T=600, H=512, I=512, E=4, k=2, backward=True)
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    dY = to_dev_bf16(inp.dY)
    res = []
    for flags in (mok.FLAG_GEMM_PAIRS, mok.FLAG_ROW_TILES):
        cfg = mok.make_config(flags=flags)
        layer.forward(x, training=True, cfg=cfg)
        g = layer.backward(x, dY, cfg=cfg)
        torch.cuda.synchronize()
        res.append({n: t.clone() for n, t in g.items()})
    for n in res[0]:
        assert torch.equal(res[0][n].view(torch.uint8), res[1][n].view(torch.uint8)), n


@pytest.mark.gpu
def test_last_tiles_of_at_most_64_rows():
    """Experts of 64, 65, 1, 127, 192, 129, 0, 320, 385 and 640 rows
    (hand-made routing, k = 1): the single-CTA kernels run an M=64 MMA for
    last tiles of at most 64 rows; the 2-SM pair kernels run an expert's odd
    last tile (one tile of 1-128 rows, or the third or fifth of 320 and 640
    rows) as an M=128 pair and an even count's short last tile (385 rows)
    inside an M=256 pair. Both equal the oracle and each other bit for bit."""
    import numpy as np
    import oracle
    from helpers import TOL, assert_close, host_bf16_f64

    counts = [64, 65, 1, 127, 192, 129, 0, 320, 385, 640]
    E, T = len(counts), sum(counts)
    wl = synth.small("m64_tiles", T=T, H=512, I=256, E=E, k=1)
    inp = synth.make_inputs(wl, seed=5)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    idx = np.repeat(np.arange(E), counts).astype(np.int32)[:, None]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    order = np.arange(T, dtype=np.int32)            # tokens are already in expert order
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    rt = {"topk_idx": dev(idx), "topk_w": dev(np.ones((T, 1), np.float32)), "counts": dev(np.array(counts, np.int32)),
          "offsets": dev(offsets), "row_src": dev(order), "slot_row": dev(order)}
    p = layer.problem(T)
    outs = []
    for flags in (mok.FLAG_ROW_TILES, mok.FLAG_GEMM_PAIRS):
        cfg = mok.make_config(flags=flags)
        ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
        mok.moe_forward(p, x, layer.packed, rt, out, ws, cfg=cfg)
        torch.cuda.synchronize()
        assert mok.device_status(ws) == (mok.OK, 0)
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    r = {"idx": idx, "w": np.ones((T, 1)), "offsets": offsets, "row_src": order}
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16)
    assert_close(host_bf16_f64(outs[0]), ref, TOL[mok.BF16], "M=64 last tiles")


SWEEP = [
    synth.small("sw_e16_t333", T=333, H=256, I=256, E=16, k=2),
    synth.small("sw_e64_t1000", T=1000, H=512, I=128, E=64, k=4, zipf_s=1.2),
    synth.small("sw_e4_t100", T=100, H=768, I=384, E=4, k=1),
    synth.small("sw_e8_t777", T=777, H=512, I=512, E=8, k=3, zipf_s=0.8, shared_I=384),
    synth.small("sw_e32_t2000", T=2000, H=256, I=256, E=32, k=8),
]


@pytest.mark.gpu
@pytest.mark.parametrize("wl", SWEEP, ids=[w.name for w in SWEEP])
def test_pairs_bitwise_sweep(wl):
    """BF16 layers of assorted shapes and routings (uniform and Zipf, k from
    1 to 8, 4 to 64 experts, with and without a shared expert): the default
    2-SM pairs (odd last tiles as M=128 pairs) against single CTAs, forward
    bit for bit, and the training step's gradients bit for bit."""
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    outs = [_staged(layer, x, wl.T, f).clone() for f in (0, mok.FLAG_ROW_TILES)]
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    if wl.shared_I:
        return   # no backward for the shared expert
    dY = torch.randn((wl.T, wl.H), device="cuda").to(torch.bfloat16)
    res = []
    for flags in (0, mok.FLAG_ROW_TILES):
        cfg = mok.make_config(flags=flags)
        layer.forward(x, training=True, cfg=cfg)
        g = layer.backward(x, dY, cfg=cfg)
        torch.cuda.synchronize()
        res.append({n: t.clone() for n, t in g.items()})
    for n in res[0]:
        assert torch.equal(res[0][n].view(torch.uint8), res[1][n].view(torch.uint8)), n
