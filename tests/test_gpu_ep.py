"""Expert parallelism with G logical ranks on one GPU (separate allocations
of one device, stream-ordered): rank g owns E/G experts, pulls the rows of
its experts from every rank through the peer table and pushes each result
to its source rank's slot buffer. Every output row is computed from the same
input row and expert weights as in the single-GPU layer, so each rank's
output must equal the single-GPU forward of its tokens bit for bit, and the
oracle within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from combine_router_top_expert_gb300 import ep, mok, synth
from helpers import TOL, assert_close, host_bf16_f64, layer_for, to_dev_bf16


def _run(G, E, k, Ts, H=512, I=256, zipf=0.0, flags=0):
    wl = synth.small("ep", T=max(Ts), H=H, I=I, E=E, k=k, zipf_s=zipf)
    inp = synth.make_inputs(wl)
    xs_host = [synth.make_x(synth.small("epx", T=T, H=H, I=I, E=E, k=k), 0, 0, shard=r) for r, T in enumerate(Ts)]
    xs = [to_dev_bf16(x) for x in xs_host]
    ranks = [ep.EPRank(r, G, inp.W_r, inp.Wg, inp.Wu, inp.Wd, k, max(Ts), bias=inp.bias) for r in range(G)]
    outs = ep.forward_logical(ranks, xs, cfg=mok.make_config(flags=flags))
    torch.cuda.synchronize()
    for rk in ranks:
        assert mok.device_status(rk.ffn_ws) == (mok.OK, 0)
    return inp, wl, xs_host, xs, ranks, outs


@pytest.mark.gpu
@pytest.mark.parametrize("G,E,k,Ts,zipf", [(2, 8, 2, [300, 300], 0.0), (4, 16, 4, [100, 0, 257, 64], 1.2)],
                         ids=["2ranks", "4ranks_uneven"])
def test_expert_parallel_matches_single_gpu_and_oracle(G, E, k, Ts, zipf):
    inp, wl, xs_host, xs, ranks, outs = _run(G, E, k, Ts, zipf=zipf)
    full = layer_for(inp, mok.BF16)
    for r in range(G):
        # the plan built on the device equals the host reference of the plan
        counts_all = np.stack([rk.routing["counts"].cpu().numpy() for rk in ranks])
        cl, ol, _ = ep.plan_host(counts_all, r)
        assert np.array_equal(ranks[r].counts_local.cpu().numpy(), cl)
        assert np.array_equal(ranks[r].offsets_local.cpu().numpy(), ol)
        if Ts[r] == 0:
            continue
        single = full.forward(xs[r]).clone()
        assert torch.equal(outs[r].view(torch.int16), single.view(torch.int16)), r
        ro = oracle.route(xs_host[r], inp.W_r, k, inp.bias)
        ref = oracle.moe_forward(xs_host[r], inp.Wg, inp.Wu, inp.Wd, ro, mode=oracle.MODE_BF16)
        assert_close(host_bf16_f64(outs[r]), ref, TOL[mok.BF16], f"rank {r}")


@pytest.mark.gpu
def test_expert_parallel_pull_bookkeeping():
    """src_rank / src_slot of every local row equal the host reference built
    from the sources' layouts (rows ordered by expert, source rank, source
    order), so every (rank, slot) is pulled by exactly one owner."""
    G, E, k, Ts = 2, 8, 2, [200, 150]
    inp, wl, xs_host, xs, ranks, outs = _run(G, E, k, Ts, zipf=1.2)
    counts_all = np.stack([rk.routing["counts"].cpu().numpy() for rk in ranks])
    offs = [rk.routing["offsets"].cpu().numpy() for rk in ranks]
    rsrc = [rk.routing["row_src"].cpu().numpy() for rk in ranks]
    seen = set()
    for r in range(G):
        ref = ep.pulled_slots_host(counts_all, r, offs, rsrc)
        n = len(ref)
        got = list(zip(ranks[r].src_rank[:n].cpu().numpy().tolist(), ranks[r].src_slot[:n].cpu().numpy().tolist()))
        assert got == ref
        seen |= set(got)
    assert seen == {(s, j) for s in range(G) for j in range(Ts[s] * k)}
