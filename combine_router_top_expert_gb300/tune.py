"""Per-shape choice of the forward's execution knobs by timing them.

The pages say the right minibatch size, the split of SMs between token
movers and compute, and the ring capacity change with the hidden size, the
top-k and the expert size (KuCoin article on MoK, section 03, limits
paragraph). This module picks them per problem shape: it enumerates candidate
configurations of the library (the stage kernels with each GEMM tiling, and
the persistent megakernel with several mover counts, minibatch sizes and ring
capacities), times each on the device through the C ABI (CUDA events, after
warm-up, device status checked), and keeps the fastest per shape key. Every
candidate computes the same layer; only the schedule differs.
"""
from __future__ import annotations

import statistics
from dataclasses import dataclass

from . import mok


@dataclass(frozen=True)
class Candidate:
    """One execution configuration (the knobs of mok_config)."""
    name: str
    flags: int = 0
    mover_ctas: int = 0
    minibatch_tokens: int = 0
    ring_rows: int = 0

    @property
    def megakernel(self) -> bool:
        return bool(self.flags & mok.FLAG_MEGAKERNEL)

    def config(self) -> mok.Config:
        return mok.make_config(flags=self.flags, mover_ctas=self.mover_ctas,
                               minibatch_tokens=self.minibatch_tokens, ring_rows=self.ring_rows)


def shape_key(p: mok.Problem, batches: int = 1, ring_rows: int = 0) -> tuple:
    return (p.T, p.H, p.I, p.E, p.k, p.dtype, p.I_shared, batches, ring_rows)


def megakernel_supported(p: mok.Problem) -> bool:
    """The megakernel's tiles: gate/up 256 wide, down as wide as H allows."""
    down = 256 if p.H % 256 == 0 else (224 if (p.dtype == mok.MXFP8 and p.H % 224 == 0) else 128)
    return (2 * p.I) % 256 == 0 and p.H % down == 0


def candidates(p: mok.Problem, batches: int = 1, ring_rows: int = 0, num_sms: int = 152) -> list[Candidate]:
    """Candidate configurations for one layer shape. With several macro-batches
    the stage kernels run batch by batch and the megakernel streams all of
    them through one ring of `ring_rows` rows (0: the library's default)."""
    # the stage kernels' default: BF16 token tiles as 2-SM pairs, MXFP8 on single CTAs
    out = [Candidate("staged")]
    if p.dtype == mok.BF16:
        out += [Candidate("staged, 128-row token tiles on single CTAs", mok.FLAG_ROW_TILES),
                Candidate("staged, swapped-operand pair tiles", mok.FLAG_SWAPPED_TILES),
                Candidate("staged, swapped-operand pair tiles, balanced token tiles",
                          mok.FLAG_SWAPPED_TILES | mok.FLAG_TOKEN_TILES_BALANCED)]
    elif p.dtype == mok.MXFP8:
        out += [Candidate("staged, 2-SM pairs", mok.FLAG_GEMM_PAIRS)]
    if megakernel_supported(p) and p.T > 0:
        for movers in (4, 8, 16):
            if movers >= num_sms // 2:
                continue
            for mb in sorted({0, max(16, p.T // 2)}):
                out.append(Candidate(f"megakernel, {movers} mover SMs, minibatch {mb or 'ring-limited'} tokens",
                                     mok.FLAG_MEGAKERNEL, movers, mb, ring_rows))
    return out


def pick(times: dict) -> Candidate:
    """The fastest candidate (the first listed among equal times)."""
    best, best_t = None, None
    for c, t in times.items():
        if t is not None and (best_t is None or t < best_t):
            best, best_t = c, t
    if best is None:
        raise RuntimeError("no candidate ran")
    return best


class Tuner:
    """Keeps the fastest candidate per shape key."""

    def __init__(self):
        self.cache: dict = {}
        self.tables: dict = {}

    def choose(self, key, cands, time_fn) -> Candidate:
        """time_fn(candidate) -> ms per step, or None if the candidate cannot
        run this shape (a library error or a bad device status)."""
        if key in self.cache:
            return self.cache[key]
        times = {}
        for c in cands:
            try:
                times[c] = time_fn(c)
            except mok.MokError:
                times[c] = None
        best = pick(times)
        self.cache[key] = best
        self.tables[key] = {c.name: t for c, t in times.items()}
        return best


def time_forward(layer, xs, cand: Candidate, steps: int = 5, warmup: int = 2, stream=None) -> float | None:
    """Median ms per step of routing + forward of the macro-batches `xs` with
    candidate `cand` on `layer` (inference). The stage kernels run batch by
    batch; a megakernel candidate with several batches streams them through
    one launch."""
    import torch
    T = xs[0].shape[0]
    p = layer.problem(T)
    cfg = cand.config()
    stream = stream or torch.cuda.current_stream()
    if cand.megakernel and len(xs) > 1:
        n = mok.workspace_size_batches(p, len(xs), cfg)
        if n == 0:
            return None
        ws = mok.alloc_bytes(n)
        b = layer.buffers(T)
        routings = [{k2: v.clone() for k2, v in b["routing"].items()} for _ in xs]
        outs = [torch.empty_like(x) for x in xs]

        def step():
            for x, r in zip(xs, routings):
                mok.route_layout(x, layer.W_r, layer.k, layer.bias, out=r, workspace=b["route_ws"], stream=stream)
            mok.moe_forward_batches(p, xs, layer.packed, routings, outs, ws, packed_shared=layer.packed_shared,
                                    cfg=cfg, stream=stream)
    else:
        ws = mok.alloc_bytes(mok.workspace_size(p, cfg))
        b = layer.buffers(T)
        out = torch.empty_like(xs[0])

        def step():
            for x in xs:
                layer.route(x, stream=stream)
                mok.moe_forward(p, x, layer.packed, b["routing"], out, ws, packed_shared=layer.packed_shared,
                                cfg=cfg, stream=stream)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if mok.device_status(ws)[0] != mok.OK:
        return None
    ms = []
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    if mok.device_status(ws)[0] != mok.OK:
        return None
    return statistics.median(ms)


_default = Tuner()


def tune_forward(layer, xs, ring_rows: int = 0, steps: int = 5, warmup: int = 2, tuner: Tuner | None = None):
    """The fastest candidate for routing + forward of the macro-batches `xs`
    (a list of [T, H] bf16 device tensors) on `layer`, and its timing table
    {candidate name: ms per step (None: could not run)}."""
    import torch
    tuner = tuner or _default
    T = xs[0].shape[0]
    p = layer.problem(T)
    sms = torch.cuda.get_device_properties(xs[0].device).multi_processor_count
    key = shape_key(p, len(xs), ring_rows)
    best = tuner.choose(key, candidates(p, len(xs), ring_rows, sms),
                        lambda c: time_forward(layer, xs, c, steps, warmup))
    return best, tuner.tables[key]
