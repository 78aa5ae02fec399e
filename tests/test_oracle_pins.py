"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a library routine, a closed form, brute
force on a tiny input, an invariant of the method, or the hand-worked example
in ``tests/golden/worked_example.json``. None of these calls the CUDA path.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from combine_router_top_expert_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------------------------- E4M3 / E8M0

def test_e4m3_table_matches_torch_float8():
    """Decoded value of every E4M3 code equals torch's float8_e4m3fn decoding."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ref[~nan], mine[~nan])
    assert np.nanmax(mine) == 448.0


def test_e4m3_encoder_exhaustive_against_torch():
    """All 65536 BF16 patterns: the oracle's nearest-value search gives the same
    byte as torch's round-to-nearest-even conversion wherever torch's result is
    finite; beyond 448 the oracle saturates to +-448 (satfinite reading)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16_val(bits)
    finite = np.isfinite(vals)
    v32 = torch.tensor(vals[finite].astype(np.float32))
    ref = v32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_encode(v) for v in vals[finite]], dtype=np.uint8)
    inrange = np.abs(vals[finite]) <= 448.0
    assert np.array_equal(mine[inrange], ref[inrange])
    big = ~inrange
    assert big.sum() > 0
    expect = np.where(vals[finite][big] > 0, 0x7E, 0xFE).astype(np.uint8)
    assert np.array_equal(mine[big], expect)


def test_e4m3_ties_to_even_closed_form():
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (mantissa 001): even wins -> 1.
    assert oracle.e4m3_value(oracle.e4m3_encode(1.0625)) == 1.0
    # 1.1875 halfway between 1.125 (001) and 1.25 (010): even -> 1.25.
    assert oracle.e4m3_value(oracle.e4m3_encode(1.1875)) == 1.25
    # smallest subnormal 2^-9; half of it is a tie between 0 and 2^-9 -> 0.
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(-(2.0 ** -10)) == 0x80
    assert oracle.e4m3_value(oracle.e4m3_encode(3 * 2.0 ** -10)) == 2.0 ** -8


def test_e8m0_scale_closed_form():
    """X = floor(log2 amax) - 8, code = X + 127, clamped; amax=0 -> 0."""
    rng = np.random.default_rng(0)
    amax = np.exp(rng.uniform(-80, 80, 2000))
    amax = np.concatenate([amax, 2.0 ** np.arange(-140, 130).astype(np.float64)])
    for a in amax:
        X = int(np.floor(np.log2(a))) - 8
        assert oracle.e8m0_code(a) == min(max(X, -127), 127) + 127, a
    assert oracle.e8m0_code(0.0) == 0


def test_mx_roundtrip_exact_for_representable_blocks():
    """Blocks whose values are E4M3 values times 2^X with amax in [2^8, 2^9)*2^X
    survive quantisation unchanged."""
    rng = np.random.default_rng(1)
    table = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    rows = []
    for X in (-20, -3, 0, 5, 30):
        for _ in range(8):
            q = rng.choice(table, 32) * rng.choice([-1, 1], 32)
            q[rng.integers(32)] = 256.0 + 32.0 * rng.integers(0, 6)   # amax in [256, 448]
            rows.append(q * 2.0 ** X)
    v = np.array(rows)
    codes, scales = oracle.mx_quantize_rows(v)
    deq = np.vectorize(oracle.e4m3_value)(codes) * 2.0 ** (scales.astype(np.float64).repeat(32, 1) - 127)
    assert np.array_equal(deq, v)


def test_mx_saturation_and_zero_block():
    v = np.zeros((2, 32))
    v[0, 0] = 500.0  # floor(log2 500) = 8 -> X = 0; 500 > 448 saturates
    v[0, 1] = -470.0
    codes, scales = oracle.mx_quantize_rows(v)
    assert scales[0, 0] == 127
    assert codes[0, 0] == 0x7E and codes[0, 1] == 0xFE
    assert scales[1, 0] == 0 and np.all(codes[1] == 0)


def test_mx_bf16_rows_equals_generic_path():
    rng = np.random.default_rng(2)
    x = bf16_bits(rng.standard_normal((7, 96)) * 3)
    c1, s1 = oracle.mx_quantize_bf16_rows(x)
    c2, s2 = oracle.mx_quantize_rows(bf16_val(x))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


# ----------------------------------------------------------------------------- BF16 rounding

def test_round_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    mine = np.array([oracle.round_bf16(float(a)) for a in v])
    assert np.array_equal(ref, mine)


def test_round_bf16_single_rounding_from_double():
    # exactly halfway between 1 and 1+2^-7: ties to even -> 1
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # a hair above halfway must round up; rounding through binary32 first would
    # land on the halfway point and then go down to 1
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7


# ----------------------------------------------------------------------------- router

def test_router_logits_exact_on_small_integers():
    """Inputs whose every partial sum is exact in fp32: the logit equals the
    exact integer dot product (+ bias)."""
    rng = np.random.default_rng(4)
    T, H, E = 9, 1000, 12
    xi = rng.integers(-2, 3, (T, H))
    wi = rng.integers(-3, 4, (H, E))
    bias = (rng.integers(-8, 9, E) / 4.0).astype(np.float32)
    x = bf16_bits(xi)
    W_r = (wi / 16.0).astype(np.float32)
    lg = oracle.router_logits(x, W_r, bias)
    exact = (xi @ wi) / 16.0 + bias
    assert np.array_equal(lg.astype(np.float64), exact)


def test_router_logits_within_fp32_error_bound():
    rng = np.random.default_rng(5)
    T, H, E = 16, 7168, 32
    x = bf16_bits(rng.standard_normal((T, H)))
    W_r = (rng.standard_normal((H, E)) * 0.02).astype(np.float32)
    lg = oracle.router_logits(x, W_r).astype(np.float64)
    xv = bf16_val(x)
    ref = xv @ W_r.astype(np.float64)
    # each chain is <= H/32 sequential fma steps, then 5 adds: gamma_n bound
    n = H // 32 + 5
    u = 2.0 ** -24
    bound = (n * u / (1 - n * u)) * (np.abs(xv) @ np.abs(W_r.astype(np.float64)))
    assert np.all(np.abs(lg - ref) <= bound)


def test_router_logits_handle_ragged_H():
    rng = np.random.default_rng(6)
    x = bf16_bits(rng.integers(-2, 3, (3, 77)))
    W = (rng.integers(-3, 4, (77, 5)) / 8.0).astype(np.float32)
    lg = oracle.router_logits(x, W)
    assert np.array_equal(lg.astype(np.float64), bf16_val(x) @ W.astype(np.float64))


def _router_order_inputs(g):
    x = np.zeros((1, g["H"]), np.float32)
    for h, v in g["x_nonzero"]:
        x[0, h] = v
    W = np.zeros((g["H"], g["E"]), np.float32)
    for h, e, v in g["W_r_nonzero"]:
        W[h, e] = v
    return bf16_bits(x), W


def test_router_logits_follow_the_fixed_order_hand_worked():
    """Hand-worked fp32 logits (tests/golden/router_order.json) that only the
    fixed chain/butterfly order gives: sequential sums, chains over h mod 32,
    chains added in sequence, a reversed butterfly, the bias added first and
    exact arithmetic each give another value."""
    g = json.load(open(os.path.join(GOLDEN, "router_order.json")))
    x, W = _router_order_inputs(g)
    lg = oracle.router_logits(x, W)
    assert lg[0].tolist() == g["logits"]
    lgb = oracle.router_logits(x, W, np.array(g["bias"], np.float32))
    assert lgb[0].tolist() == g["logits_with_bias"]
    for name, v in g["other_readings"].items():   # the fixture tells the readings apart
        assert v != (g["logits_with_bias"] if name == "bias_added_first" else g["logits"]), name
    # the exact product sum differs from the fp32 result only by the absorbed +1
    assert (bf16_val(x).astype(np.float64) @ W.astype(np.float64))[0].tolist() == g["other_readings"]["exact"]
    r = oracle.route(x, W, 2)
    assert r["idx"][0].tolist() == g["k2"]["idx"]
    assert np.allclose(r["w"][0], g["k2"]["w"], rtol=1e-15)


# ----------------------------------------------------------------------------- top-k, weights

def _brute_topk(lg, k):
    T, E = lg.shape
    out = np.empty((T, k), np.int64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t].astype(np.float64)))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (32, 8), (5, 5), (64, 1)])
def test_topk_brute_force_and_weights(E, k):
    rng = np.random.default_rng(E * 10 + k)
    lg = (rng.standard_normal((200, E)) * 1.7).astype(np.float32)
    lg[::7, 1] = lg[::7, 0]         # exact ties: lower index must win
    idx, w = oracle.topk(lg, k)
    assert np.array_equal(idx, _brute_topk(lg, k))
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    assert np.all(w > 0)
    assert np.all(np.diff(w, axis=1) <= 0)
    # reading: softmax over all E, keep the selected, renormalise
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), 1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12, atol=0)


def test_topk_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(7)
    lg = (rng.standard_normal((50, 6)) * 2).astype(np.float32)
    idx, w = oracle.topk(lg, 6)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    assert np.allclose(np.take_along_axis(p, idx.astype(np.int64), 1), w, rtol=1e-12, atol=0)


def test_topk_tie_goes_to_lower_index_and_signed_zero():
    lg = np.array([[0.0, -0.0, 1.0, 1.0]], np.float32)
    idx, w = oracle.topk(lg, 3)
    assert idx.tolist() == [[2, 3, 0]]
    lg2 = np.array([[-0.0, 0.0]], np.float32)
    assert oracle.topk(lg2, 1)[0].tolist() == [[0]]


# ----------------------------------------------------------------------------- layout

@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (300, 32, 8), (1, 4, 4), (50, 16, 1)])
def test_layout_against_library_sort(T, E, k):
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 0] += 3.0 * (T > 10)  # one heavy expert
    idx, _ = oracle.topk(lg, k)
    counts, offsets, row_src, slot_row = oracle.layout(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert counts.sum() == T * k
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    slots = np.arange(T * k)
    order = np.lexsort((slots // k, idx.ravel()))  # by expert, then token
    assert np.array_equal(row_src, order)
    assert np.array_equal(slot_row[row_src], np.arange(T * k))
    assert np.array_equal(idx.ravel()[row_src], np.repeat(np.arange(E), counts))


# ----------------------------------------------------------------------------- forward

def _golden_routing(g, key):
    idx = np.array(g[key]["idx"], np.int32)
    w = np.array(g[key]["w"], np.float64)
    E = 2
    counts, offsets, row_src, slot_row = oracle.layout(idx, E)
    return dict(idx=idx, w=w, offsets=offsets, row_src=row_src)


def test_forward_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    x = bf16_bits(g["x"])
    Wg, Wu, Wd = (bf16_bits(g[n]) for n in ("W_gate", "W_up", "W_down"))
    W_r = np.array(g["W_r"], np.float32)
    r = oracle.route(x, W_r, 1)
    assert r["idx"].tolist() == g["k1"]["idx"]
    out = oracle.moe_forward(x, Wg, Wu, Wd, r, mode=oracle.MODE_EXACT)
    assert np.allclose(out, g["k1"]["out_exact"], rtol=1e-15, atol=1e-15)
    out = oracle.moe_forward(x, Wg, Wu, Wd, r, mode=oracle.MODE_BF16)
    assert np.array_equal(out, np.array(g["k1"]["out_bf16"]))
    r2 = oracle.route(x, W_r, 2)
    assert r2["idx"].tolist() == g["k2"]["idx"]
    assert np.allclose(r2["w"], g["k2"]["w"], rtol=1e-15)
    out = oracle.moe_forward(x, Wg, Wu, Wd, r2, mode=oracle.MODE_EXACT)
    assert np.allclose(out, g["k2"]["out_exact"], rtol=1e-14, atol=1e-15)


def _dense_reference(xv, Wg, Wu, Wd, idx, w):
    """Every token through every expert, masked by its routing weight (numpy
    fp64; the sigmoid is scipy's expit)."""
    T, H = xv.shape
    E = Wg.shape[0]
    mask = np.zeros((T, E))
    np.put_along_axis(mask, idx.astype(np.int64), w, 1)
    out = np.zeros((T, H))
    for e in range(E):
        G = xv @ Wg[e]
        U = xv @ Wu[e]
        y = (G * scipy.special.expit(G) * U) @ Wd[e]
        out += mask[:, e:e + 1] * y
    return out


def test_forward_equals_dense_brute_force():
    wl = synth.small("t", T=40, H=96, I=64, E=6, k=3)
    inp = synth.make_inputs(wl, seed=11)
    r = oracle.route(inp.x, inp.W_r, wl.k)
    out = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_EXACT)
    ref = _dense_reference(bf16_val(inp.x), bf16_val(inp.Wg), bf16_val(inp.Wu), bf16_val(inp.Wd),
                           r["idx"], r["w"])
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-14 * np.abs(ref).max())
    # BF16 operand mode differs from exact only by the rounding of h
    outb = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_BF16)
    rms = np.sqrt((ref ** 2).mean())
    assert np.abs(outb - ref).max() < 2e-2 * rms
    assert not np.array_equal(outb, out)


def test_forward_single_expert_is_dense_swiglu_torch():
    wl = synth.small("t", T=17, H=64, I=32, E=1, k=1)
    inp = synth.make_inputs(wl, seed=12)
    r = oracle.route(inp.x, inp.W_r, 1)
    assert np.all(r["w"] == 1.0)
    out = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_EXACT)
    X = torch.tensor(bf16_val(inp.x))
    Wg, Wu, Wd = (torch.tensor(bf16_val(a)[0]) for a in (inp.Wg, inp.Wu, inp.Wd))
    ref = (torch.nn.functional.silu(X @ Wg) * (X @ Wu)) @ Wd
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-16)


def test_forward_zero_input_gives_zero():
    wl = synth.small("t", T=8, H=64, I=32, E=4, k=2)
    inp = synth.make_inputs(wl, seed=13)
    x0 = np.zeros_like(inp.x)
    r = oracle.route(x0, inp.W_r, 2)
    assert r["idx"].tolist() == [[0, 1]] * 8  # all logits 0: lowest indices
    for mode in (oracle.MODE_BF16, oracle.MODE_MXFP8):
        assert np.all(oracle.moe_forward(x0, inp.Wg, inp.Wu, inp.Wd, r, mode=mode) == 0)


def test_forward_token_shuffle_invariance():
    wl = synth.small("t", T=50, H=64, I=32, E=8, k=2, zipf_s=1.2)
    inp = synth.make_inputs(wl, seed=14)
    perm = np.random.default_rng(0).permutation(wl.T)
    r = oracle.route(inp.x, inp.W_r, 2, inp.bias)
    rp = oracle.route(inp.x[perm], inp.W_r, 2, inp.bias)
    assert np.array_equal(rp["idx"], r["idx"][perm])
    assert np.array_equal(rp["w"], r["w"][perm])
    assert np.array_equal(rp["counts"], r["counts"])
    for mode in (oracle.MODE_BF16, oracle.MODE_MXFP8):
        o = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=mode)
        op = oracle.moe_forward(inp.x[perm], inp.Wg, inp.Wu, inp.Wd, rp, mode=mode)
        assert np.array_equal(op, o[perm])


def test_forward_mxfp8_equals_dense_on_dequantised_operands():
    wl = synth.small("t", T=24, H=64, I=64, E=4, k=2)
    inp = synth.make_inputs(wl, seed=15)
    r = oracle.route(inp.x, inp.W_r, 2)
    out = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_MXFP8)

    def deq_rows(v):  # blocks of 32 along the last axis
        c, s = oracle.mx_quantize_rows(v)
        return np.vectorize(oracle.e4m3_value)(c) * 2.0 ** (s.astype(np.float64).repeat(32, 1) - 127)

    xq = deq_rows(bf16_val(inp.x))
    Wg = np.stack([deq_rows(bf16_val(inp.Wg[e]).T).T for e in range(wl.E)])
    Wu = np.stack([deq_rows(bf16_val(inp.Wu[e]).T).T for e in range(wl.E)])
    Wd = np.stack([deq_rows(bf16_val(inp.Wd[e]).T).T for e in range(wl.E)])
    # reference with h quantised the same way
    mask = np.zeros((wl.T, wl.E))
    np.put_along_axis(mask, r["idx"].astype(np.int64), r["w"], 1)
    ref = np.zeros((wl.T, wl.H))
    for e in range(wl.E):
        G, U = xq @ Wg[e], xq @ Wu[e]
        h = deq_rows(G * scipy.special.expit(G) * U)
        ref += mask[:, e:e + 1] * (h @ Wd[e])
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def test_forward_sampled_tokens_and_shared_expert():
    wl = synth.small("t", T=30, H=64, I=32, E=4, k=2, shared_I=32)
    inp = synth.make_inputs(wl, seed=16)
    r = oracle.route(inp.x, inp.W_r, 2)
    full = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_EXACT)
    toks = np.array([29, 3, 17])
    part = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_EXACT, tokens=toks)
    assert np.array_equal(part, full[toks])
    withs = oracle.moe_forward(inp.x, inp.Wg, inp.Wu, inp.Wd, r, mode=oracle.MODE_EXACT, shared=inp.shared)
    X = torch.tensor(bf16_val(inp.x))
    Sg, Su, Sd = (torch.tensor(bf16_val(a)) for a in inp.shared)
    s = ((torch.nn.functional.silu(X @ Sg) * (X @ Su)) @ Sd).numpy()
    assert np.allclose(withs, full + s, rtol=1e-12, atol=1e-16)


# ----------------------------------------------------------------------------- backward

def _fd_case():
    rng = np.random.default_rng(21)
    T, H, I, E, k = 6, 16, 8, 4, 2
    x = rng.standard_normal((T, H))
    W_r = rng.standard_normal((H, E)) * 0.3
    Wg = rng.standard_normal((E, H, I)) * 0.3
    Wu = rng.standard_normal((E, H, I)) * 0.3
    Wd = rng.standard_normal((E, I, H)) * 0.3
    dY = rng.standard_normal((T, H))
    return x, W_r, Wg, Wu, Wd, dY, k


def _loss(x, W_r, Wg, Wu, Wd, dY, k, idx_fixed):
    lg = oracle.router_logits_f64(x, W_r)
    idx, w = oracle.topk(lg, k)
    assert np.array_equal(idx, idx_fixed), "finite-difference step changed the selection"
    c, off, rs, sr = oracle.layout(idx, Wg.shape[0])
    out = oracle.moe_forward(x, Wg, Wu, Wd, dict(idx=idx, w=w, offsets=off, row_src=rs),
                             mode=oracle.MODE_EXACT, f64=True)
    return float((out * dY).sum())


def test_backward_matches_central_finite_differences():
    x, W_r, Wg, Wu, Wd, dY, k = _fd_case()
    lg = oracle.router_logits_f64(x, W_r)
    srt = np.sort(lg, 1)[:, ::-1]
    assert np.all(srt[:, k - 1] - srt[:, k] > 1e-3), "inputs too close to a top-k tie"
    idx, w = oracle.topk(lg, k)
    c, off, rs, sr = oracle.layout(idx, Wg.shape[0])
    routing = dict(idx=idx, w=w, offsets=off, row_src=rs)
    dX, dWg, dWu, dWd, dWr = oracle.moe_backward(x, W_r, Wg, Wu, Wd, dY, routing,
                                                  mode=oracle.MODE_EXACT, f64=True)
    eps = 1e-6
    rng = np.random.default_rng(0)
    args = [x, W_r, Wg, Wu, Wd]
    grads = [dX, dWr, dWg, dWu, dWd]
    for ai, (a, gr) in enumerate(zip(args, grads)):
        for _ in range(12):
            pos = tuple(rng.integers(0, s) for s in a.shape)
            ap, am = a.copy(), a.copy()
            ap[pos] += eps
            am[pos] -= eps
            lp = _loss(*[ap if i == ai else args[i] for i in range(5)], dY, k, idx)
            lm = _loss(*[am if i == ai else args[i] for i in range(5)], dY, k, idx)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - gr[pos]) <= 1e-6 * max(1.0, abs(fd)), (ai, pos, fd, gr[pos])


def test_backward_matches_torch_autograd():
    x, W_r, Wg, Wu, Wd, dY, k = _fd_case()
    lg = oracle.router_logits_f64(x, W_r)
    idx, w = oracle.topk(lg, k)
    c, off, rs, sr = oracle.layout(idx, Wg.shape[0])
    routing = dict(idx=idx, w=w, offsets=off, row_src=rs)
    got = oracle.moe_backward(x, W_r, Wg, Wu, Wd, dY, routing, mode=oracle.MODE_EXACT, f64=True)
    tx, tWr, tWg, tWu, tWd = (torch.tensor(a, requires_grad=True) for a in (x, W_r, Wg, Wu, Wd))
    tidx = torch.tensor(idx, dtype=torch.int64)
    logits = tx @ tWr
    wsel = torch.softmax(torch.gather(logits, 1, tidx), dim=1)
    out = torch.zeros_like(tx)
    for j in range(k):
        e = tidx[:, j]
        G = torch.einsum("th,thi->ti", tx, tWg[e])
        U = torch.einsum("th,thi->ti", tx, tWu[e])
        y = torch.einsum("ti,tih->th", torch.nn.functional.silu(G) * U, tWd[e])
        out = out + wsel[:, j:j + 1] * y
    (out * torch.tensor(dY)).sum().backward()
    for mine, ref in zip(got, (tx.grad, tWg.grad, tWu.grad, tWd.grad, tWr.grad)):
        assert np.allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_sampled_backward_equals_full_backward():
    """The one-by-one backward gives the same numbers as the full backward."""
    wl = synth.small("t", T=40, H=64, I=32, E=4, k=2, backward=True)
    inp = synth.make_inputs(wl, seed=31)
    r = oracle.route(inp.x, inp.W_r, 2)
    dX, dWg, dWu, dWd, dWr = oracle.moe_backward(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r)
    toks = [0, 17, 39]
    cols = [(0, 3), (3, 31), (1, 0)]
    sX, sG, sU, sD = oracle.moe_backward_sampled(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, toks, cols)
    assert np.allclose(sX, dX[toks], rtol=1e-12, atol=1e-15)
    for q, (e, i) in enumerate(cols):
        assert np.allclose(sG[q], dWg[e][:, i], rtol=1e-12, atol=1e-15)
        assert np.allclose(sU[q], dWu[e][:, i], rtol=1e-12, atol=1e-15)
        assert np.allclose(sD[q], dWd[e][i, :], rtol=1e-12, atol=1e-15)
    # router-gradient columns one by one equal the full backward's
    cw = oracle.router_grad_columns(inp.x, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, [2, 0])
    assert np.allclose(cw[0], dWr[:, 2], rtol=1e-12, atol=1e-15 * np.abs(dWr).max())
    assert np.allclose(cw[1], dWr[:, 0], rtol=1e-12, atol=1e-15 * np.abs(dWr).max())


def _golden_backward_case(g):
    x = bf16_bits(g["x"])
    Wg, Wu, Wd = (bf16_bits(g[n]) for n in ("W_gate", "W_up", "W_down"))
    dY = bf16_bits(g["dY"])
    W_r = np.array(g["W_r"], np.float32)
    idx = np.array(g["idx"], np.int32)
    counts, offsets, row_src, slot_row = oracle.layout(idx, W_r.shape[1])
    routing = dict(idx=idx, w=np.array(g["w"], np.float64), offsets=offsets, row_src=row_src)
    return x, W_r, Wg, Wu, Wd, dY, routing


@pytest.mark.parametrize("mode,key", [(oracle.MODE_BF16, "bf16"), (oracle.MODE_EXACT, "exact")])
def test_backward_operand_rounding_hand_worked(mode, key):
    """Hand-worked backward (tests/golden/backward_bf16_rounding.json) whose
    values move when any one of the BF16 roundings of dy, dG or dU is dropped
    or applied to another intermediate (dh instead of dG, say); every value is
    a dyadic rational, so the comparison is exact."""
    g = json.load(open(os.path.join(GOLDEN, "backward_bf16_rounding.json")))
    x, W_r, Wg, Wu, Wd, dY, r = _golden_backward_case(g)
    dX, dWg, dWu, dWd, dWr = oracle.moe_backward(x, W_r, Wg, Wu, Wd, dY, r, mode=mode)
    exp = g[key]
    assert dX.tolist() == exp["dX"]
    assert dWg.tolist() == exp["dW_gate"]
    assert dWu.tolist() == exp["dW_up"]
    assert dWd.tolist() == exp["dW_down"]
    assert dWr.tolist() == exp["dW_r"]
    if key == "bf16":
        # the sampled form of the backward follows the same roundings
        sX, sG, sU, sD = oracle.moe_backward_sampled(x, W_r, Wg, Wu, Wd, dY, r, [0], [(0, 0), (1, 0)])
        assert sX.tolist() == exp["dX"]
        assert sG.tolist() == [[v[0] for v in exp["dW_gate"][e]] for e in (0, 1)]
        assert sU.tolist() == [[v[0] for v in exp["dW_up"][e]] for e in (0, 1)]
        assert sD.tolist() == [exp["dW_down"][e][0] for e in (0, 1)]
        cw = oracle.router_grad_columns(x, Wg, Wu, Wd, dY, r, [0, 1])
        assert cw.tolist() == [[row[0] for row in exp["dW_r"]], [row[1] for row in exp["dW_r"]]]


# ----------------------------------------------------------------------------- MXFP8 backward

def _mx_q(v, axis):
    """MXFP8 round trip along `axis` in blocks of 32 (the last block may be
    short), with torch's float8_e4m3fn conversion as the element encoder and
    the E8M0 rule X = floor(log2 amax) - 8 (clamped) as the block scale."""
    v = np.moveaxis(np.asarray(v, np.float64), axis, 0)
    out = np.empty_like(v)
    for r0 in range(0, v.shape[0], 32):
        blk = v[r0:r0 + 32]
        amax = np.abs(blk).max(axis=0)
        e = np.frexp(np.where(amax > 0, amax, 1.0))[1] - 1          # floor(log2 amax)
        X = np.clip(np.where(amax > 0, e - 8, -127), -127, 127).astype(np.float64)
        q = np.clip(blk / 2.0 ** X, -448.0, 448.0)
        f8 = torch.from_numpy(np.ascontiguousarray(q)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        out[r0:r0 + 32] = f8 * 2.0 ** X
    return np.moveaxis(out, 0, axis)


def _mx_backward_numpy(xv, W_r, Wg, Wu, Wd, dYv, r):
    """The MXFP8 backward written with numpy matmuls over explicitly
    quantised operands (fp64); BF16 roundings by the oracle's pinned rounding."""
    rb = np.vectorize(oracle.round_bf16)
    T, H = xv.shape
    E, _, I = Wg.shape
    k = r["idx"].shape[1]
    sig = lambda z: 1.0 / (1.0 + np.exp(-z))
    dWg, dWu, dWd = np.zeros((E, H, I)), np.zeros((E, H, I)), np.zeros((E, I, H))
    da = np.zeros((T * k, H))
    gw = np.zeros(T * k)
    for e in range(E):
        rows = r["row_src"][r["offsets"][e]:r["offsets"][e + 1]]
        if len(rows) == 0:
            continue
        t = rows // k
        A = xv[t]
        G = _mx_q(A, 1) @ _mx_q(Wg[e], 0)
        U = _mx_q(A, 1) @ _mx_q(Wu[e], 0)
        h = G * sig(G) * U
        y = _mx_q(h, 1) @ _mx_q(Wd[e], 0)
        gw[rows] = (dYv[t] * y).sum(1)
        dy = rb(r["w"].reshape(-1)[rows][:, None] * dYv[t])
        dh = _mx_q(dy, 1) @ _mx_q(Wd[e], 1).T
        s = sig(G)
        dG = rb(dh * U * s * (1.0 + G * (1.0 - s)))
        dU = rb(dh * G * s)
        da[rows] = _mx_q(dG, 1) @ _mx_q(Wg[e], 1).T + _mx_q(dU, 1) @ _mx_q(Wu[e], 1).T
        hb = rb(h)
        dWg[e] = _mx_q(A, 0).T @ _mx_q(dG, 0)
        dWu[e] = _mx_q(A, 0).T @ _mx_q(dU, 0)
        dWd[e] = _mx_q(hb, 0).T @ _mx_q(dy, 0)
    w = r["w"]
    gwr = gw.reshape(T, k)
    dl = w * (gwr - (w * gwr).sum(1, keepdims=True))
    dX = da.reshape(T, k, H).sum(1) + np.einsum("tj,htj->th", dl, W_r.astype(np.float64)[:, r["idx"]])
    dWr = np.zeros((H, E))
    for j in range(k):
        np.add.at(dWr.T, r["idx"][:, j], dl[:, j:j + 1] * xv)
    return dX, dWg, dWu, dWd, dWr


def test_mxfp8_backward_equals_numpy_on_explicitly_quantised_operands():
    """Random BF16 inputs: the oracle's MXFP8 backward equals the same
    formulas evaluated with numpy matmuls on operands quantised along the
    stated axes by torch's float8 conversion (dy and W_down along H for dh;
    dG, dU, W_gate, W_up along I for da; x, h, dy, dG, dU along the expert's
    rows for the weight gradients)."""
    wl = synth.small("mxb", T=70, H=64, I=96, E=4, k=2, backward=True)
    inp = synth.make_inputs(wl, seed=41)
    r = oracle.route(inp.x, inp.W_r, wl.k)
    got = oracle.moe_backward(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, mode=oracle.MODE_MXFP8)
    ref = _mx_backward_numpy(bf16_val(inp.x), inp.W_r, bf16_val(inp.Wg), bf16_val(inp.Wu), bf16_val(inp.Wd),
                             bf16_val(inp.dY), r)
    for n, a, b in zip(("dX", "dW_gate", "dW_up", "dW_down", "dW_r"), got, ref):
        assert np.allclose(a, b, rtol=1e-9, atol=1e-12 * np.abs(b).max()), n
    # and the quantisation matters: the BF16-mode backward differs
    b16 = oracle.moe_backward(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, mode=oracle.MODE_BF16)
    assert not np.allclose(b16[1], got[1], rtol=1e-3)


def test_mxfp8_backward_exact_operands_equal_bf16_backward():
    """Inputs on which every MXFP8 quantisation of the backward is exact
    (powers of two; G = 64 or 0, where silu and silu' are exact; one nonzero
    per weight column or row): the MXFP8 backward equals the BF16 one bit for
    bit, so the quantised mode adds nothing but the quantisations."""
    T, H, I, E, k = 40, 64, 32, 4, 2
    rng = np.random.default_rng(3)
    x = rng.choice([0.0, 1.0, -1.0, 0.5, -0.5], (T, H))
    x[:, 0] = 1.0
    Wg = np.zeros((E, H, I)); Wu = np.zeros((E, H, I)); Wd = np.zeros((E, I, H))
    for e in range(E):
        Wg[e, 0] = rng.choice([0.0, 64.0], I)
        Wu[e, 0] = rng.choice([1.0, -1.0, 0.5, -0.5], I)
        for i in range(I):
            Wd[e, i, rng.integers(H)] = rng.choice([1.0, -1.0, 0.5])
    dY = rng.choice([1.0, -1.0, 2.0, -2.0], (T, H))
    W_r = (rng.standard_normal((H, E)) * 0.1).astype(np.float32)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, row_src, slot_row = oracle.layout(idx, E)
    r = dict(idx=idx, w=np.full((T, k), 0.5), offsets=offsets, row_src=row_src)
    args = [bf16_bits(a) for a in (x, Wg, Wu, Wd, dY)]
    mx = oracle.moe_backward(args[0], W_r, args[1], args[2], args[3], args[4], r, mode=oracle.MODE_MXFP8)
    bf = oracle.moe_backward(args[0], W_r, args[1], args[2], args[3], args[4], r, mode=oracle.MODE_BF16)
    for a, b in zip(mx, bf):
        assert np.array_equal(a, b)
    assert np.abs(mx[1]).max() > 0 and np.abs(mx[3]).max() > 0


def test_sampled_mxfp8_backward_equals_full_mxfp8_backward():
    """The one-by-one MXFP8 backward (dX rows, weight-gradient columns) gives
    the full MXFP8 backward's numbers."""
    wl = synth.small("t", T=70, H=64, I=64, E=4, k=2, backward=True)
    inp = synth.make_inputs(wl, seed=43)
    r = oracle.route(inp.x, inp.W_r, 2)
    dX, dWg, dWu, dWd, dWr = oracle.moe_backward(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r,
                                                  mode=oracle.MODE_MXFP8)
    toks = [0, 33, 69]
    cols = [(0, 3), (3, 63), (1, 0)]
    sX, sG, sU, sD = oracle.moe_backward_sampled(inp.x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.dY, r, toks, cols,
                                                 mode=oracle.MODE_MXFP8)
    assert np.allclose(sX, dX[toks], rtol=1e-12, atol=1e-14 * np.abs(dX).max())
    for q, (e, i) in enumerate(cols):
        assert np.allclose(sG[q], dWg[e][:, i], rtol=1e-12, atol=1e-14 * np.abs(dWg).max())
        assert np.allclose(sU[q], dWu[e][:, i], rtol=1e-12, atol=1e-14 * np.abs(dWu).max())
        assert np.allclose(sD[q], dWd[e][i, :], rtol=1e-12, atol=1e-14 * np.abs(dWd).max())
