"""The per-shape autotuner: candidate enumeration, selection and caching
(host logic, on the CPU with a fake timer) and, on the GPU, a tuned
configuration that runs the layer within tolerance of the oracle."""
import pytest

from combine_router_top_expert_gb300 import mok, tune


def _p(T=2560, H=7168, I=2048, E=32, k=8, dtype=mok.BF16, I_shared=0):
    return mok.make_problem(T, H, I, E, k, dtype, I_shared)


def test_candidates_cover_paths_and_megakernel_knobs():
    c = tune.candidates(_p(), num_sms=152)
    names = [x.name for x in c]
    assert names[0] == "staged"
    assert any(x.flags == mok.FLAG_ROW_TILES for x in c)
    assert any(x.flags == mok.FLAG_SWAPPED_TILES for x in c)
    assert any(x.flags & mok.FLAG_TOKEN_TILES_BALANCED for x in c)
    mk = [x for x in c if x.megakernel]
    assert {x.mover_ctas for x in mk} == {4, 8, 16}
    assert {x.minibatch_tokens for x in mk} == {0, 1280}
    # MXFP8: no BF16-only tilings; shapes the megakernel cannot tile get none
    cm = tune.candidates(_p(dtype=mok.MXFP8), num_sms=152)
    assert not any(x.flags & (mok.FLAG_ROW_TILES | mok.FLAG_SWAPPED_TILES) for x in cm)
    assert not any(x.megakernel for x in tune.candidates(_p(H=384, I=64), num_sms=152))
    # few SMs: mover counts that leave no compute half are dropped
    assert all(x.mover_ctas < 8 for x in tune.candidates(_p(), num_sms=16) if x.megakernel)
    # ring capacity is passed through to the megakernel candidates
    assert all(x.ring_rows == 4096 for x in tune.candidates(_p(), 4, 4096) if x.megakernel)


def test_pick_and_cache():
    cands = tune.candidates(_p(), num_sms=152)
    fake = {c: 10.0 + i for i, c in enumerate(cands)}
    fake[cands[3]] = 1.0
    fake[cands[1]] = None                        # could not run
    calls = []

    def time_fn(c):
        calls.append(c)
        if c is cands[2]:
            raise mok.MokError(mok.ERR_INVALID, "x")
        return fake[c]
    t = tune.Tuner()
    key = tune.shape_key(_p())
    assert t.choose(key, cands, time_fn) is cands[3]
    assert len(calls) == len(cands)
    assert t.tables[key][cands[2].name] is None
    assert t.choose(key, cands, time_fn) is cands[3]   # cached: no new timings
    assert len(calls) == len(cands)
    with pytest.raises(RuntimeError):
        tune.pick({cands[0]: None})


@pytest.mark.gpu
def test_tuned_forward_runs_and_matches_oracle():
    import oracle
    from combine_router_top_expert_gb300 import synth
    from helpers import TOL, assert_close, host_bf16_f64, layer_for, to_dev_bf16
    import torch
    wl = synth.small("tune", T=600, H=512, I=256, E=8, k=2, zipf_s=1.2)
    inp = synth.make_inputs(wl)
    layer = layer_for(inp, mok.BF16)
    x = to_dev_bf16(inp.x)
    best, table = tune.tune_forward(layer, [x], steps=3, warmup=1, tuner=tune.Tuner())
    assert table[best.name] is not None and table[best.name] == min(v for v in table.values() if v is not None)
    out = layer.forward(x, cfg=best.config()).clone()
    torch.cuda.synchronize()
    assert layer.status(wl.T) == (mok.OK, 0)
    r = oracle.route(inp.x, inp.W_r, wl.k, inp.bias)
    ref = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16)
    assert_close(host_bf16_f64(out), ref, TOL[mok.BF16], "tuned: " + best.name)
