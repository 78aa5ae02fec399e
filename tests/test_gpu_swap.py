"""BF16 inference GEMMs with the operands swapped: weight rows as the M side
of 2-SM pair tiles (256 rows over two CTAs), each expert's tokens cut into
tiles of any multiple of 32 rows as the N side.

Each output element is still one K-ordered tensor-core dot product with
fp32 accumulation; how an expert's tokens are cut into tiles cannot change
it, so both cuts (balanced tiles; 256 rows plus a remainder) must give the
same bits. Against the oracle the layer stays within the BF16 tolerance, and
against the 128-row token tiles (the other operand order) too. The tests
force the swapped tiles (MOK_FLAG_SWAPPED_TILES); by default the library
picks them only for shapes where they measured faster."""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import mok, synth
from helpers import TOL, assert_close, host_bf16_f64, layer_for, to_dev_bf16

CASES = [
    synth.small("sw_ragged", T=1000, H=512, I=256, E=4, k=2),
    synth.small("sw_skew", T=700, H=256, I=2048, E=8, k=4, zipf_s=1.2),
    synth.small("sw_sparse", T=8, H=256, I=128, E=64, k=1),
    synth.small("sw_e256", T=300, H=256, I=128, E=256, k=8, zipf_s=1.2),
    synth.small("sw_shared", T=500, H=768, I=384, E=8, k=2, zipf_s=1.2, shared_I=256),
]


def _forward(layer, x, T, flags, routing=None):
    p = layer.problem(T)
    cfg = mok.make_config(flags=flags)
    ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
    out = torch.empty((T, layer.H), dtype=torch.bfloat16, device="cuda")
    mok.moe_forward(p, x, layer.packed, routing or layer.buffers(T)["routing"], out, ws,
                    packed_shared=layer.packed_shared, cfg=cfg)
    torch.cuda.synchronize()
    assert mok.device_status(ws) == (mok.OK, 0)
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_swapped_tiles_match_oracle_and_both_cuts(wl):
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    layer.route(x)
    bal = _forward(layer, x, wl.T, mok.FLAG_SWAPPED_TILES)
    bal2 = _forward(layer, x, wl.T, mok.FLAG_SWAPPED_TILES | mok.FLAG_TOKEN_TILES_BALANCED)
    rows = _forward(layer, x, wl.T, mok.FLAG_ROW_TILES)
    assert torch.equal(bal.view(torch.int16), bal2.view(torch.int16))
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16, shared=inp.shared)
    assert_close(host_bf16_f64(bal), ref, TOL[mok.BF16], wl.name)
    assert_close(host_bf16_f64(rows), ref, TOL[mok.BF16], wl.name + " (token tiles)")
    same = torch.equal(bal.view(torch.int16), rows.view(torch.int16))
    print(f"[swap] {wl.name}: bit-identical to the 128-row token tiles: {same}")


@pytest.mark.gpu
def test_swapped_tiles_edge_counts():
    """Hand-made routing (k = 1) giving experts 0, 1, 15, 16, 17, 31, 32,
    33, 255, 256, 257 and 513 rows: token tiles of 32-row multiples with ragged ends, and
    an empty expert, against the oracle."""
    counts = [0, 1, 15, 16, 17, 31, 32, 33, 255, 256, 257, 513]
    E, T = len(counts), sum(counts)
    wl = synth.small("sw_edges", T=T, H=512, I=256, E=E, k=1)
    inp = synth.make_inputs(wl, seed=7)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    idx = np.repeat(np.arange(E), counts).astype(np.int32)[:, None]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    order = np.arange(T, dtype=np.int32)            # tokens are already in expert order
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    rt = {"topk_idx": dev(idx), "topk_w": dev(np.ones((T, 1), np.float32)), "counts": dev(np.array(counts, np.int32)),
          "offsets": dev(offsets), "row_src": dev(order), "slot_row": dev(order)}
    bal = _forward(layer, x, T, mok.FLAG_SWAPPED_TILES, rt)
    bal2 = _forward(layer, x, T, mok.FLAG_SWAPPED_TILES | mok.FLAG_TOKEN_TILES_BALANCED, rt)
    assert torch.equal(bal.view(torch.int16), bal2.view(torch.int16))
    r = {"idx": idx, "w": np.ones((T, 1)), "offsets": offsets, "row_src": order}
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16)
    assert_close(host_bf16_f64(bal), ref, TOL[mok.BF16], "edge counts")


@pytest.mark.gpu
def test_swapped_tiles_bitwise_reruns():
    wl = CASES[0]
    inp = synth.make_inputs(wl, seed=2)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    cfg = mok.make_config(flags=mok.FLAG_SWAPPED_TILES)
    first = layer.forward(x, cfg=cfg).clone()
    for _ in range(9):
        assert torch.equal(layer.forward(x, cfg=cfg).view(torch.int16), first.view(torch.int16))
