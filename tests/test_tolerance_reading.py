"""The tolerance measure the GPU parity tests use (tests/helpers.py), checked
on the CPU against the oracle's own output.

The layer's output is BF16, so even an exact result, rounded once to BF16,
differs from the fp64 reference by up to half a BF16 ulp: at the largest
elements of a layer output (about six times its rms) that alone is close to
the 2e-2 * rms bar. The measure used is max(|gpu - ref| - ulp_half(ref)) /
rms(ref): the distance of the GPU value from the interval of values that
round to the same BF16 number as the exact result, i.e. the error made before
the final rounding. These tests show on real oracle outputs that it is zero
for an exact result rounded once and grows with the pre-rounding error, while
the two other forms - |gpu - ref| and |gpu - round_bf16(ref)| against the
literal bar - are dominated by a half or a whole ulp of the largest element
whatever the error is.
"""
import numpy as np
import pytest

import oracle
from combine_router_top_expert_gb300 import synth
from helpers import TOL, rel_err
from combine_router_top_expert_gb300 import mok

round_bf16 = np.vectorize(oracle.round_bf16)


@pytest.fixture(scope="module")
def layer_out():
    wl = synth.small("ragged_bf16", T=1000, H=512, I=256, E=4, k=2)
    inp = synth.make_inputs(wl)
    r = oracle.route(inp.x, inp.W_r, wl.k)
    return oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16)


def test_exact_result_rounded_once_measures_zero(layer_out):
    ref = layer_out
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.abs(ref).max() / rms > 6.0        # the heavy tail of a layer output
    perfect = round_bf16(ref)
    raw, adj = rel_err(perfect, ref)
    assert adj <= 1e-15
    # the literal |gpu - ref| <= c * rms is nearly used up by the rounding alone
    assert raw > 0.9 * TOL[mok.BF16]


@pytest.mark.parametrize("eps", [1e-5, 1e-4, 1e-3])
def test_measure_follows_the_error_before_rounding(layer_out, eps):
    ref = layer_out
    rms = np.sqrt(np.mean(ref ** 2))
    z = np.random.default_rng(0).standard_normal(ref.shape)
    gpu = round_bf16(ref + eps * rms * z)       # an error of eps * rms, then the output rounding
    raw, adj = rel_err(gpu, ref)
    assert adj <= eps * np.abs(z).max() + 1e-15
    assert adj >= 0.1 * eps
    # against round_bf16(ref), one boundary crossed at a large element costs a
    # whole ulp: the comparison reads ~0.019 even at an error 2000x below the bar
    vs_rounded = np.abs(gpu - round_bf16(ref)).max() / rms
    assert vs_rounded > 0.9 * TOL[mok.BF16]
