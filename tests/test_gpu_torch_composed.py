"""The PyTorch-composed layer that bench.py times beside the library as a
context arm computes the same layer: on tokens whose top-k experts agree
with the oracle's fixed-order routing, its output is close to the oracle.
Stock BF16 ops round more intermediates than the library does (G, U,
silu(G), h and every expert output y each to BF16, against h alone), so the
bar is 5e-2 * rms rather than the library's 2e-2."""
import numpy as np
import pytest
import torch

import bench
import oracle
from combine_router_top_expert_gb300 import synth
from combine_router_top_expert_gb300.layer import to_dev_bf16
from helpers import assert_close, host_bf16_f64


@pytest.mark.gpu
def test_torch_composed_layer_matches_oracle():
    wl = synth.small("tc", T=600, H=512, I=256, E=8, k=2, zipf_s=1.2)
    inp = synth.make_inputs(wl)
    x = to_dev_bf16(inp.x)
    W_r = torch.from_numpy(inp.W_r).cuda()
    bias = torch.from_numpy(inp.bias).cuda()
    Wg, Wu, Wd = (to_dev_bf16(a) for a in (inp.Wg, inp.Wu, inp.Wd))
    out = bench.torch_composed_forward(x, W_r, bias, Wg, Wu, Wd, wl.k)
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_EXACT)
    lg = (torch.from_numpy(synth.bf16_to_f32(inp.x)).cuda() @ W_r + bias)
    same = np.array([set(a) == set(b) for a, b in zip(torch.topk(lg, wl.k, dim=1).indices.cpu().numpy().tolist(),
                                                      r["idx"].tolist())])
    assert same.mean() > 0.99
    assert_close(host_bf16_f64(out)[same], ref[same], 5e-2, "torch-composed layer")
