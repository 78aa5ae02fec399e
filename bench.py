"""Benchmark of the routed MoE layer on GB300 (one JSON line on stdout).

Default workload: BF16 forward, T=2560 tokens, H=7168, I=2048, E=32 experts,
top-k=8 (Kimi-2.5-shaped experts), uniform routing. One step = one whole
layer: route + top-k + layout, pull-dispatch, grouped gate/up GEMM with fused
SwiGLU, grouped down GEMM with push-combine, fixed-order weighted sum.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl mok|reference]

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; L2 is flushed (a 256 MiB write) before every timed
step. Multi-GPU (torchrun, N > 1): every rank runs an independent replica of
the layer on its own token shard with the same weights (data parallel; no
collective on the data path, since expert parallelism needs peer GPUs in one
NVLink domain); rank 0 reports all ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_router_top_expert_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s (fwd, fwd+bwd) at H7168/I2048; grouped-GEMM % TC peak"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d.get("hbm_gbs", 6800.0), bf16=d.get("bf16_tflops", 1900.0),
                    bf16_sus=d.get("bf16_tflops_sustained", 1700.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the steps run; the SM clock is
    the median over samples taken under load (GPU utilisation >= 50%)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.window = None   # host wall-clock (start, end) of the timed region
        self.path = os.path.join("/tmp", f"mok_clocks_{os.getpid()}.csv")

    def mark(self, t_start, t_end):
        """The timed region, as host wall-clock times taken right after the
        synchronisations that bracket it."""
        self.window = (t_start, t_end)

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def wait_first(self, timeout_s=3.0):
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < timeout_s:
            self.f.flush()
            if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        lines = open(self.path).read().splitlines()
        os.unlink(self.path)
        return self.summarise(lines, self.window)

    @staticmethod
    def summarise(lines, window=None):
        """Clock record from nvidia-smi CSV lines (the fields of Q). The
        samples taken inside `window` (host wall-clock seconds) are the ones
        summarised when there are any; else those at >= 50 % utilisation;
        else all."""
        import datetime
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 11:
                rows.append(parts)
        if not rows:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        def stamp(v):
            try:
                return datetime.datetime.strptime(v, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        timed = []
        if window is not None:
            timed = [r for r in rows if stamp(r[0]) is not None and window[0] <= stamp(r[0]) <= window[1]]
        loaded = [r for r in rows if (num(r[5]) or 0.0) >= 50.0]
        use = timed or loaded or rows
        sm = [num(r[2]) for r in use if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        pw = [num(r[4]) for r in use if num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[7:11]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded), "samples_in_timed_region": len(timed),
                "summarised": "timed region" if timed else "under load" if loaded else "all samples"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# DRAM bytes per step of the grouped GEMM pair (dram__bytes_read.sum +
# dram__bytes_write.sum of both launches) from one ncu capture, with the
# hash of the GEMM kernel sources it was captured on; the 32-expert figure is
# the 8-expert profiling case's traffic x 4 (experts and routed rows both
# 4x). A capture whose sources no longer match the built kernels is stale and
# reported as null.
GEMM_SOURCES = ["gemm.cuh", "tc.cuh", "gemm.cu", "gemm_swap.cuh"]
GEMM_PAIR_TRAFFIC = {"bf16_fwd_T2560": {"bytes": 3.7829e+09, "gemm_sources_sha1": "e26ec62c46cfe7ad"}}


def gemm_sources_sha1():
    import hashlib
    h = hashlib.sha1()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "combine_router_top_expert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(name):
    """(bytes, note) of the GEMM pair's captured DRAM traffic for workload
    `name`, or (None, why) when there is none for the kernels as built."""
    c = GEMM_PAIR_TRAFFIC.get(name)
    if c is None:
        return None, "not captured for this workload"
    if c["gemm_sources_sha1"] != gemm_sources_sha1():
        return None, "stale: captured on GEMM sources " + c["gemm_sources_sha1"]
    return c["bytes"], "ncu capture on GEMM sources " + c["gemm_sources_sha1"]


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over all ranks (identity on
    one rank): the slowest rank's timings set the whole job's rate."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world_size, units_per_rank_step, steps, slowest_ms):
    """Units processed by all ranks per second of the slowest rank's time."""
    return world_size * units_per_rank_step * steps / (slowest_ms / 1000.0)


def oracle_layer_seconds(inp, wl, t0, n):
    """Wall time of the oracle as it stands running the layer on tokens
    [t0, t0+n) of the workload's input, as a layer of n tokens: routing,
    layout and the expert FFNs (fp64), plus for backward workloads the
    oracle's backward of those tokens (dX rows and two weight columns)."""
    import oracle
    dt = oracle.MODE_MXFP8 if wl.dtype == "mxfp8" else oracle.MODE_BF16
    x = np.ascontiguousarray(inp.x[t0:t0 + n])
    t_start = time.perf_counter()
    r = oracle.route(x, inp.W_r, wl.k, inp.bias)
    oracle.moe_forward(x, inp.Wg, inp.Wu, inp.Wd, r, mode=dt, shared=inp.shared)
    if wl.backward:
        dY = np.ascontiguousarray(inp.dY[t0:t0 + n])
        oracle.moe_backward_sampled(x, inp.W_r, inp.Wg, inp.Wu, inp.Wd, dY, r, np.arange(n, dtype=np.int32),
                                    [(0, 0), (wl.E - 1, wl.I - 1)], mode=dt)
    return time.perf_counter() - t_start


def oracle_sample_text(wl, n, steps):
    what = "forward" + (" + backward (dX rows, 2 weight columns)" if wl.backward else "")
    return (f"{steps} x {n} tokens of the workload's input, each run as a layer of {n} tokens "
            f"(routing, layout, {what}; fp64 oracle)")


def cpu_baseline(inp, wl, n_tokens=32):
    """The oracle as it stands on a bounded sample of the workload's tokens."""
    import oracle
    n = min(n_tokens, wl.T)
    dt_s = oracle_layer_seconds(inp, wl, 0, n)
    return {"value": n / dt_s, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": oracle_sample_text(wl, n, 1) + f", {dt_s:.1f} s"}


def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    inp = synth.make_inputs(wl)
    import oracle
    oracle.build()
    # size each step's sample so all K steps take about two minutes
    per_token = oracle_layer_seconds(inp, wl, 0, 1)
    n_tok = int(max(1, min(32, 120.0 / max(1, args.steps) / max(per_token, 1e-6))))
    times = []
    for i in range(args.steps):
        t0 = (i * n_tok) % max(1, wl.T - n_tok + 1)
        times.append(oracle_layer_seconds(inp, wl, t0, n_tok))
    v = n_tok * len(times) / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                                            "k": wl.k, "operands": wl.dtype},
            "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "value": v, "unit": "tokens/s",
                             "sample": oracle_sample_text(wl, n_tok, args.steps)},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def trace_step(args, mok, layer, x, xs, p, cfg, b, wl, stream, routings, ws_b):
    """One megakernel step with per-CTA trace records; fractions of the kernel
    window each role spends working on tiles / moves, waiting on GPU-local
    counters, in the weighted sums, and idle (before its first unit of work
    and after it exits). A mover's weighted-sum chunks taken while it waits
    for a ring region count as weighted sums, not as waiting."""
    import torch
    cfg2 = mok.make_config(num_sms=cfg.num_sms, timeout_ms=cfg.timeout_ms, flags=cfg.flags | mok.FLAG_TRACE,
                           mover_ctas=cfg.mover_ctas, minibatch_tokens=cfg.minibatch_tokens, ring_rows=cfg.ring_rows)
    if len(xs) > 1:
        mok.moe_forward_batches(p, xs, layer.packed, routings, [torch.empty_like(xb) for xb in xs], ws_b,
                                packed_shared=layer.packed_shared, cfg=cfg2, stream=stream)
        ws = ws_b
    else:
        layer.route(x, stream=stream)
        layer.forward(x, cfg=cfg2, stream=stream, route=False)
        ws = b["ws"]
    torch.cuda.synchronize()
    dev = torch.cuda.current_device()
    n = torch.cuda.get_device_properties(dev).multi_processor_count
    if cfg.num_sms:
        n = min(n, cfg.num_sms)
    rec = mok.megakernel_trace(ws, n).astype(np.float64)
    t0, t1 = rec[:, 1].min(), rec[:, 4].max()
    dur = t1 - t0
    out = {"kernel_us": dur / 1e3, "ctas": int(n)}
    for role, name in ((0, "movers"), (1, "compute")):
        r = rec[rec[:, 0] == role]
        if len(r) == 0:
            continue
        comb_final = r[:, 4] - r[:, 3]                      # the pass after the tile/move work
        comb_in_window = np.maximum(r[:, 7] - comb_final, 0.0)
        work = (r[:, 3] - r[:, 2] - r[:, 5] - comb_in_window) / dur
        out[name] = {"ctas": int(len(r)),
                     "first_work_us": float(np.mean(r[:, 2] - t0) / 1e3),
                     "work_frac": float(np.mean(work)),
                     "counter_wait_frac": float(np.mean(r[:, 5] / dur)),
                     "combine_frac": float(np.mean(r[:, 7] / dur)),
                     "idle_frac": float(np.mean(1.0 - work - r[:, 5] / dur - r[:, 7] / dur)),
                     "units_mean": float(np.mean(r[:, 6]))}
    return out


def build_layer(wl, dev, rank, inp=None):
    """Host inputs and the layer (packed weights on `dev`). Workloads of one
    expert shape draw the same weights (seed 0), so `inp` of one can be
    reused for another: only its tokens (and the logit bias) are redrawn."""
    from combine_router_top_expert_gb300 import mok
    from combine_router_top_expert_gb300.layer import MoELayer
    dtype = mok.MXFP8 if wl.dtype == "mxfp8" else mok.BF16
    if inp is None:
        # data-parallel replicas: every rank holds the same weights and its own tokens
        inp = synth.make_inputs(wl, shard=rank)
    else:
        inp = synth.LayerInputs(wl, inp.W_r, synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None,
                                inp.Wg, inp.Wu, inp.Wd, inp.shared)
        inp.xs = [synth.make_x(wl, b, 0, rank) for b in range(wl.batches)]
        if wl.backward:
            inp.dY = synth.make_dY(wl, 0, rank)
    layer = MoELayer(inp.W_r, inp.Wg, inp.Wu, inp.Wd, wl.k, dtype=dtype, bias=inp.bias, shared=inp.shared,
                     device=dev, keep_unpacked=wl.backward)
    return inp, layer


def measure(args, wl, inp, layer, dev, steps, warmup, trace=False, with_e2e=True):
    """Time `steps` layer steps of workload `wl` after `warmup` untimed ones
    (CUDA events per step, L2 flushed before each), then, with `with_e2e`,
    the same steps end to end through the public API with host buffers.
    Every rank calls this; returns the per-step record (timings already the
    maximum over ranks) that line() turns into JSON."""
    import torch
    from combine_router_top_expert_gb300 import mok
    from combine_router_top_expert_gb300.layer import to_dev_bf16
    ws, rank, local = dist_env()

    dtype = mok.MXFP8 if wl.dtype == "mxfp8" else mok.BF16
    T, H = wl.T, wl.H
    xs = [to_dev_bf16(xb, dev) for xb in inp.xs]
    x = xs[0]
    p = layer.problem(T)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    staged = not args.megakernel or wl.backward
    flags = ((0 if staged else mok.FLAG_MEGAKERNEL) | (mok.FLAG_GEMM_PAIRS if args.gemm_pairs else 0) |
             (mok.FLAG_SWAPPED_TILES if args.swapped_tiles else 0) |
             (mok.FLAG_ROW_TILES if args.single_cta else 0) |
             (mok.FLAG_MB_TOKEN_RANGES if args.mb_token_ranges else 0))
    cfg = mok.make_config(flags=flags, ring_rows=wl.ring_rows, mover_ctas=args.movers,
                          minibatch_tokens=args.minibatch)
    b = layer.buffers(T, training=wl.backward, cfg=cfg)
    rt = b["routing"]
    routings = ws_b = None
    mode = ("fwd+bwd (staged)" if wl.backward else
            f"{len(xs)} macro-batches, megakernel" if len(xs) > 1 and not staged else
            f"{len(xs)} macro-batches, staged kernels batch by batch" if len(xs) > 1 else
            "staged kernels" if staged else "megakernel")

    if wl.backward:
        dY = to_dev_bf16(inp.dY, dev)

        def step(ev=None):
            # route + training forward (saves activations) + backward
            layer.route(x, training=True, stream=stream)
            if ev is not None:
                ev[0].record(stream)
            layer.forward(x, training=True, cfg=cfg, stream=stream, route=False)
            layer.backward(x, dY, cfg=cfg, stream=stream)
            if ev is not None:
                ev[1].record(stream)
        # route 3; BF16: training forward 4 (dispatch, 2 GEMMs, combine), backward
        # 12; MXFP8: forward 6 (BF16 rows, E4M3 rows, pad zeroing, 2 GEMMs,
        # combine), backward 16 (5 quantisation passes into 3, 4 GEMMs as in BF16)
        launches_per_step = 3 + (6 + 16 if dtype == mok.MXFP8 else 4 + 12)
        status_ws = b["ws"]
        flops = 18.0 * H * wl.I * T * wl.k
        kern = ("layer GEMMs fwd+bwd (staged; 2 fwd + 4 bwd grouped GEMM launches" +
                (", MXFP8 operands and quantisation passes)" if dtype == mok.MXFP8 else ")"))
    elif len(xs) > 1 and staged:
        outs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in xs]
        status_ws = b["ws"]

        def step(ev=None):
            # batch by batch: route/layout, dispatch, grouped GEMMs, shared
            # expert, weighted sum
            if ev is not None:
                ev[0].record(stream)
            for xb, ob in zip(xs, outs):
                layer.route(xb, stream=stream)
                layer.forward(xb, cfg=cfg, stream=stream, route=False, out=ob)
            if ev is not None:
                ev[1].record(stream)
        # per batch: route 3, dispatch 1, grouped GEMMs 2, shared expert 2, weighted sum 1
        launches_per_step = len(xs) * (3 + 1 + 2 + (2 if wl.shared_I else 0) + 1)
        flops = wl.fwd_flops()
        kern = "every launch of the batch-by-batch stage kernels (routing, dispatch, GEMMs, shared expert, sum)"
    elif len(xs) > 1:
        routings = [{n: v.clone() for n, v in rt.items()} for _ in xs]
        outs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in xs]
        ws_b = mok.alloc_bytes(mok.workspace_size_batches(p, len(xs), cfg), dev)
        route_ws = b["route_ws"]

        def step(ev=None):
            for xb, rb in zip(xs, routings):
                mok.route_layout(xb, layer.W_r, wl.k, layer.bias, out=rb, workspace=route_ws, stream=stream)
            if ev is not None:
                ev[0].record(stream)
            mok.moe_forward_batches(p, xs, layer.packed, routings, outs, ws_b, packed_shared=layer.packed_shared,
                                    cfg=cfg, stream=stream)
            if ev is not None:
                ev[1].record(stream)
        # per batch: route 3 (+ 2 shared-expert GEMMs); then plan 2 + megakernel 1
        launches_per_step = 3 * len(xs) + (2 * len(xs) if wl.shared_I else 0) + 3
        status_ws = ws_b
        flops = wl.fwd_flops()
        kern = "shared-expert GEMMs + forward megakernel (one launch for all macro-batches)"
    elif staged:
        rows = mok.padded_rows_max(T, wl.E, wl.k)
        eb = 1 if dtype == mok.MXFP8 else 2
        A = mok.alloc_bytes(rows * H * eb, dev)
        A_sf = mok.alloc_bytes(rows * H // 32, dev) if dtype == mok.MXFP8 else None
        h = mok.alloc_bytes(rows * wl.I * eb, dev)
        h_sf = mok.alloc_bytes(rows * wl.I // 32, dev) if dtype == mok.MXFP8 else None
        part = torch.empty((T * wl.k, H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        status_ws = b["ws"]
        mx_once = dtype == mok.MXFP8   # MXFP8: one token-major pass quantises each token once

        def step(ev=None):
            # route/layout, dispatch, grouped GEMMs, combine (7 launches)
            layer.route(x, stream=stream)
            if ev is not None:
                ev[2].record(stream)
            if mx_once:
                mok.dispatch_tokens(p, x, rt, A, A_sf, stream=stream)
            else:
                mok.dispatch(p, x, rt, A, A_sf, stream=stream)
            if ev is not None:
                ev[0].record(stream)
            mok.expert_ffn(p, A, A_sf, layer.packed, rt, h, h_sf, part, status_ws, cfg=cfg, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            mok.combine(p, part, rt["topk_w"], out, stream=stream)
        launches_per_step = 7
        flops = 6.0 * H * wl.I * T * wl.k
        kern = "grouped expert GEMMs (gate/up+SwiGLU, down+push; 2 launches)"
    else:
        status_ws = b["ws"]

        def step(ev=None):
            # route/layout (3 launches), plan (2), megakernel (1)
            layer.route(x, stream=stream)
            if ev is not None:
                ev[0].record(stream)
            layer.forward(x, cfg=cfg, stream=stream, route=False)
            if ev is not None:
                ev[1].record(stream)
        launches_per_step = 6
        flops = 6.0 * H * wl.I * T * wl.k
        kern = "forward megakernel (dispatch + grouped GEMMs + combine, one launch; plus 2 plan launches)"

    # clocks are sampled from before the warm-up steps to the end of the timed
    # steps (nvidia-smi needs a moment before its first sample)
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    st = mok.device_status(status_ws)
    if st[0] != mok.OK:
        raise SystemExit(f"{wl.name}: device status after warm-up: {st}")

    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(5)) for _ in range(steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_timed0 = time.time()
    for i in range(steps):
        flush.zero_()
        s0, s1, g0, g1, x0 = evs[i]
        s0.record(stream)
        step((g0, g1, x0))
        s1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(t_timed0, time.time())
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    gemm_ms = [e[2].elapsed_time(e[3]) for e in evs]
    stage_lines = None
    if staged and not wl.backward and len(xs) == 1:
        # the other stages of the staged step, each against its own bound
        peaks0 = load_peaks()
        R = T * wl.k
        eb = 1 if dtype == mok.MXFP8 else 2
        route_ms = statistics.median(e[0].elapsed_time(e[4]) for e in evs)
        disp_ms = statistics.median(e[4].elapsed_time(e[2]) for e in evs)
        comb_ms = statistics.median(e[3].elapsed_time(e[1]) for e in evs)
        disp_b = T * H * 2 + R * H * eb + (R * H // 32 if dtype == mok.MXFP8 else 0)
        comb_b = R * H * 2 + R * 4 + T * H * 2
        fma_peak = 152 * 128 * 2 * 2.07e9 / 1e12   # fp32 FMA: SMs x lanes x 2 FLOP x max SM clock
        stage_lines = {
            "route_topk_layout": {"ms": route_ms, "bound": "alu", "unit": "TFLOP/s",
                                  "achieved": 2.0 * T * wl.E * H / (route_ms / 1e3) / 1e12, "peak": fma_peak,
                                  "frac": 2.0 * T * wl.E * H / (route_ms / 1e3) / 1e12 / fma_peak,
                                  "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2070 MHz",
                                  "note": "3 launches (weight re-layout, logits + top-k, layout)"},
            "dispatch": {"ms": disp_ms, "bound": "hbm", "unit": "GB/s", "bytes": disp_b,
                         "achieved": disp_b / (disp_ms / 1e3) / 1e9, "peak": peaks0["hbm"],
                         "frac": disp_b / (disp_ms / 1e3) / 1e9 / peaks0["hbm"]},
            "combine": {"ms": comb_ms, "bound": "hbm", "unit": "GB/s", "bytes": comb_b,
                        "achieved": comb_b / (comb_ms / 1e3) / 1e9, "peak": peaks0["hbm"],
                        "frac": comb_b / (comb_ms / 1e3) / 1e9 / peaks0["hbm"]},
        }
    total_ms = sum(step_ms)
    st = mok.device_status(status_ws)
    if st[0] != mok.OK:
        raise SystemExit(f"{wl.name}: device status after timed steps: {st}")

    sm_partition = None
    if trace and not staged:
        sm_partition = trace_step(args, mok, layer, x, xs, p, cfg, b, wl, stream, routings, ws_b)

    e2e = None
    if with_e2e:
        e2e = measure_e2e(wl, inp, layer, dev, stream, cfg, b, p, xs, routings, ws_b, status_ws, steps, staged)

    # aggregate over ranks: the slowest rank's times
    t_max, e2e_max = max_over_ranks([total_ms, e2e["ms"] if e2e else 0.0], dev)
    return dict(wl=wl, dtype=dtype, steps=steps, warmup=warmup, total_ms=t_max, rank_total_ms=total_ms,
                step_ms=step_ms, gemm_ms=gemm_ms, stage_lines=stage_lines, sm_partition=sm_partition, clocks=clk,
                e2e=e2e, e2e_ms=e2e_max, launches_per_step=launches_per_step, flops=flops, kern=kern, mode=mode,
                staged=staged, tokens_per_step=T * len(xs), batches=len(xs))


def measure_e2e(wl, inp, layer, dev, stream, cfg, b, p, xs, routings, ws_b, status_ws, steps, staged):
    """End to end through the public API with host buffers: every step copies
    its inputs in from pinned host memory and its result back out; steps are
    pipelined the way a serving loop would run them (copy streams in and out
    beside the compute stream, two buffer slots), so the copies of steps i+1
    and i-1 overlap the kernels of step i."""
    import torch
    from combine_router_top_expert_gb300 import mok
    T, H = wl.T, wl.H
    x_host = [torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory() for xb in inp.xs]
    dY_host = (torch.from_numpy(inp.dY.view(np.int16)).view(torch.bfloat16).pin_memory() if wl.backward else None)
    out_host = [[torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in xs] for _ in range(2)]
    x_slot = [[torch.empty_like(xb) for xb in xs] for _ in range(2)]
    dY_slot = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)] if wl.backward else None
    out_slot = [[torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in xs] for _ in range(2)]
    grads_slot = None
    if wl.backward:
        grads_slot = [dict(dX=out_slot[i][0], dW_gate=torch.empty_like(layer.Wg), dW_up=torch.empty_like(layer.Wu),
                           dW_down=torch.empty_like(layer.Wd),
                           dW_r=torch.empty((H, wl.E), dtype=torch.float32, device=dev)) for i in range(2)]
    batched = len(xs) > 1 and not staged   # one megakernel launch over all macro-batches
    route_e2e = routings if batched else [layer.buffers(T, wl.backward)["routing"]]
    c_in, c_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_step(sl):
        c_in.wait_event(ev_done[sl])            # step i-2 finished reading this slot
        with torch.cuda.stream(c_in):
            for xh, xd in zip(x_host, x_slot[sl]):
                xd.copy_(xh, non_blocking=True)
            if wl.backward:
                dY_slot[sl].copy_(dY_host, non_blocking=True)
        ev_in[sl].record(c_in)
        stream.wait_event(ev_in[sl])
        stream.wait_event(ev_out[sl])           # step i-2's result has left this slot
        with torch.cuda.stream(stream):
            xsl = x_slot[sl]
            if wl.backward:
                layer.forward(xsl[0], training=True, cfg=cfg, stream=stream)
                layer.backward(xsl[0], dY_slot[sl], cfg=cfg, stream=stream, grads=grads_slot[sl])
            elif batched:
                for xd, rb in zip(xsl, route_e2e):
                    mok.route_layout(xd, layer.W_r, wl.k, layer.bias, out=rb, workspace=b["route_ws"],
                                     stream=stream)
                mok.moe_forward_batches(p, xsl, layer.packed, route_e2e, out_slot[sl], ws_b,
                                        packed_shared=layer.packed_shared, cfg=cfg, stream=stream)
            else:
                # batch by batch (one batch: the single-step path)
                for xd, od in zip(xsl, out_slot[sl]):
                    mok.route_layout(xd, layer.W_r, wl.k, layer.bias, out=route_e2e[0], workspace=b["route_ws"],
                                     stream=stream)
                    mok.moe_forward(p, xd, layer.packed, route_e2e[0], od, b["ws"],
                                    packed_shared=layer.packed_shared, cfg=cfg, stream=stream)
        ev_done[sl].record(stream)
        c_out.wait_event(ev_done[sl])
        with torch.cuda.stream(c_out):
            for o, oh in zip(out_slot[sl], out_host[sl]):
                oh.copy_(o, non_blocking=True)
        ev_out[sl].record(c_out)

    for i in range(4):
        e2e_step(i % 2)
    torch.cuda.synchronize(dev)
    n_e2e = max(8, steps)   # pipelined: amortise the first copy-in and last copy-out
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(c_in)
    for i in range(n_e2e):
        e2e_step(i % 2)
    c_out.wait_event(ev_done[(n_e2e - 1) % 2])
    a1.record(c_out)
    torch.cuda.synchronize(dev)
    if mok.device_status(status_ws)[0] != mok.OK:
        raise SystemExit(f"{wl.name}: device status after end-to-end steps: {mok.device_status(status_ws)}")
    return dict(ms=a0.elapsed_time(a1), steps=n_e2e,
                h2d=len(xs) * T * H * 2 * (2 if wl.backward else 1), d2h=len(xs) * T * H * 2,
                api="mok_route_layout + " + ("mok_moe_forward(training) + mok_moe_backward" if wl.backward else
                                             "mok_moe_forward_batches" if batched else "mok_moe_forward"))


def roofline(m, args):
    """The dominant kernels' roofline object of measurement `m`."""
    from combine_router_top_expert_gb300 import mok
    wl, dtype = m["wl"], m["dtype"]
    peaks = load_peaks()
    H = wl.H
    # captured traffic belongs to the default stage kernels (BF16: 2-SM pairs) only
    traffic, traffic_note = (captured_traffic(wl.name) if (m["staged"] and m["batches"] == 1 and not args.gemm_pairs
                                                           and not args.swapped_tiles and not args.single_cta)
                             else (None, "not captured for this path"))
    fl = m["flops"]
    g_ms = statistics.mean(m["gemm_ms"])
    achieved = fl / (g_ms / 1000.0) / 1e12
    long_region = m["rank_total_ms"] > 1000.0
    peak = (peaks["bf16_sus"] if long_region else peaks["bf16"]) * (2.0 if dtype == mok.MXFP8 else 1.0)
    # the GEMM pair's algorithmic HBM bytes: expert weights (+ MXFP8 scales),
    # the gathered rows read, h written and read back, the partials written
    R_rows = wl.T * wl.k * m["batches"]
    ebw = (1.0 + 1.0 / 32) if dtype == mok.MXFP8 else 2.0
    gemm_bytes = (3.0 * wl.E * H * wl.I * ebw + R_rows * H * ebw + 2.0 * R_rows * wl.I * ebw + R_rows * H * 2.0)
    if wl.backward:
        gemm_bytes = None   # the fwd+bwd step is tensor-bound at every size measured here
    hbm_achieved = gemm_bytes / (g_ms / 1000.0) / 1e9 if gemm_bytes else None
    # the bound of the workload: whichever of FLOP / peak and bytes / HBM peak is longer
    hbm_bound = bool(gemm_bytes) and gemm_bytes / (peaks["hbm"] * 1e9) > fl / (peak * 1e12)
    kern = m["kern"]
    if hbm_bound:
        return {"kernel": kern, "bound": "hbm", "achieved": hbm_achieved, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": hbm_achieved / peaks["hbm"], "peak_source": f"{peaks['source']} hbm copy",
                "bytes_per_step": gemm_bytes, "ms_per_step": g_ms, "traffic": traffic, "traffic_note": traffic_note,
                "tensor": {"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak}}
    return {"kernel": kern, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_source": f"{peaks['source']} bf16 {'sustained' if long_region else 'burst'}" +
                           (" x2 (fp8 nominal ratio)" if dtype == mok.MXFP8 else ""),
            "flops_per_step": fl, "ms_per_step": g_ms, "traffic": traffic, "traffic_note": traffic_note,
            "hbm": ({"achieved": hbm_achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": hbm_achieved / peaks["hbm"], "bytes_per_step": gemm_bytes} if gemm_bytes else None)}


def config_of(m, args, ws):
    wl = m["wl"]
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
            "operands": wl.dtype, "routing": "zipf s=1.2 bias" if wl.zipf_s else "uniform",
            "macro_batches": m["batches"], "shared_expert_I": wl.shared_I, "ring_rows": wl.ring_rows or "default",
            "mover_ctas": args.movers or 8, "path": m["mode"],
            "minibatches": (("token ranges" if args.mb_token_ranges else "expert-tile runs")
                            if (not m["staged"] or m["batches"] > 1) else None),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "l2": "flushed before every timed step (256 MiB write); per-step CUDA events"}


def e2e_of(m, ws):
    e = m["e2e"]
    return {"value": whole_job_rate(ws, m["tokens_per_step"], e["steps"], m["e2e_ms"]), "unit": "tokens/s",
            "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"], "api": e["api"], "steps": e["steps"],
            "pipelining": "H2D of step i+1 and D2H of step i-1 on two copy streams overlap step i's kernels; "
                          "no L2 flush (each step's working set, the expert weights, is larger than L2)"}


def torch_composed_forward(x, W_r, bias, Wg, Wu, Wd, k):
    """The same layer written with stock PyTorch ops on the GPU, the way an
    MoE layer is commonly composed in PyTorch: router matmul (fp32), top-k,
    softmax over the selected logits, a stable sort of the routed rows by
    expert, index_select gather, one cuBLAS matmul per expert and projection
    (SwiGLU between), then the weighted index_add_ back into token order.
    Context arm only (a stand-in for the "PyTorch" baseline class the pages
    compare against); the routing of exact ties may differ from the fixed
    order of the library's router."""
    import torch
    import torch.nn.functional as F
    T, H = x.shape
    E = W_r.shape[1]
    logits = x.float() @ W_r
    if bias is not None:
        logits = logits + bias
    val, idx = torch.topk(logits, k, dim=1)
    w = torch.softmax(val, dim=1)
    flat = idx.reshape(-1)
    order = torch.argsort(flat, stable=True)
    tok = order // k
    counts = torch.bincount(flat, minlength=E).tolist()      # host sync, as in the usual loop form
    xs = x.index_select(0, tok)
    ys = torch.empty_like(xs)
    s0 = 0
    for e in range(E):
        s1 = s0 + counts[e]
        if s1 > s0:
            a = xs[s0:s1]
            h = F.silu(a @ Wg[e]) * (a @ Wu[e])
            ys[s0:s1] = h @ Wd[e]
        s0 = s1
    out = torch.zeros((T, H), dtype=torch.float32, device=x.device)
    out.index_add_(0, tok, ys.float() * w.reshape(-1)[order, None])
    return out.to(torch.bfloat16)


def measure_torch_composed(wl, inp, dev, steps, warmup):
    """tokens/s of torch_composed_forward on the workload (BF16, CUDA events
    per step, L2 flushed before each)."""
    import torch
    from combine_router_top_expert_gb300.layer import to_dev_bf16
    x = to_dev_bf16(inp.x, dev)
    W_r = torch.from_numpy(np.ascontiguousarray(inp.W_r)).to(dev)
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).to(dev)
    Wg, Wu, Wd = (to_dev_bf16(a, dev) for a in (inp.Wg, inp.Wu, inp.Wd))
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        torch_composed_forward(x, W_r, bias, Wg, Wu, Wd, wl.k)
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch_composed_forward(x, W_r, bias, Wg, Wu, Wd, wl.k)
        e1.record()
        torch.cuda.synchronize(dev)
        ms.append(e0.elapsed_time(e1))
    del Wg, Wu, Wd
    torch.cuda.empty_cache()
    med = statistics.median(ms)
    return {"what": "the same layer composed of stock PyTorch ops (index_select gather, one cuBLAS matmul per "
                    "expert and projection, index_add_ combine), BF16, same inputs; context only",
            "value": wl.T / (med / 1e3), "unit": "tokens/s", "ms_per_step": med, "steps": steps,
            "torch": torch.__version__}


# Sub-measurements of the default line: the metric's other halves ("fwd+bwd"
# and MXFP8, forward and training), on the same GPU in the same run.
EXTRA_WORKLOADS = ("bf16_bwd_T4096", "mxfp8_zipf_T2560", "mxfp8_bwd_T4096")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="bf16_fwd_T2560", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="mok", choices=["mok", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the fwd+bwd and MXFP8 sub-measurements of the default workload")
    ap.add_argument("--megakernel", action="store_true", help="time the persistent megakernel forward")
    ap.add_argument("--gemm-pairs", action="store_true", help="BF16 grouped GEMMs as 2-SM CTA pairs (tcgen05 cta_group::2)")
    ap.add_argument("--single-cta", action="store_true",
                    help="BF16 grouped GEMMs on single CTAs (128-row token tiles) instead of 2-SM pairs")
    ap.add_argument("--swapped-tiles", action="store_true",
                    help="BF16 inference GEMMs with swapped operands (weight rows as M of 2-SM pair tiles)")
    ap.add_argument("--movers", type=int, default=0, help="megakernel mover CTAs (0 = library default)")
    ap.add_argument("--minibatch", type=int, default=0, help="megakernel minibatch tokens (0 = ring-limited)")
    ap.add_argument("--mb-token-ranges", action="store_true",
                    help="megakernel minibatches as token ranges (default: runs of expert tiles)")
    ap.add_argument("--trace", action="store_true",
                    help="megakernel: after the timed steps, one traced step; report the SM partition's busy/idle time")
    args = ap.parse_args()
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from combine_router_top_expert_gb300 import mok

    inp, layer = build_layer(wl, dev, rank)
    m = measure(args, wl, inp, layer, dev, args.steps, args.warmup, trace=args.trace)
    extras = []
    if (args.workload == "bf16_fwd_T2560" and not args.no_extra and not args.megakernel and not args.gemm_pairs
            and not args.swapped_tiles and not args.single_cta and ws == 1):
        # the same experts (same weight draw): BF16 fwd+bwd at T=4096, the
        # MXFP8 forward with Zipf-skewed routing at T=2560, MXFP8 fwd+bwd at T=4096
        del layer
        torch.cuda.empty_cache()
        for name in EXTRA_WORKLOADS:
            wx = synth.WORKLOADS[name]
            ix, lx = build_layer(wx, dev, rank, inp=inp)
            mx = measure(args, wx, ix, lx, dev, max(20, args.steps // 4), max(3, args.warmup), with_e2e=True)
            extras.append(mx)
            del lx
            torch.cuda.empty_cache()
    torch_arm = None
    if args.workload == "bf16_fwd_T2560" and not args.no_extra and ws == 1:
        torch_arm = measure_torch_composed(wl, inp, dev, 20, 3)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    value = whole_job_rate(ws, m["tokens_per_step"], m["steps"], m["total_ms"])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": m["steps"],
        "warmup": m["warmup"], "ms_per_step": m["total_ms"] / m["steps"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if m["dtype"] == mok.BF16 else "mxfp8",
        "data": "synthetic",
        "config": config_of(m, args, ws),
        "gemm_cta_pairs": bool(args.gemm_pairs),
        "gemm_swapped_tiles": bool(args.swapped_tiles),
        "gemm_single_cta": bool(args.single_cta),
        "roofline": roofline(m, args),
        "e2e": e2e_of(m, ws),
        "stage_rooflines": m["stage_lines"],
        "sm_partition": m["sm_partition"],
        "gpu_launches": m["launches_per_step"] * m["steps"] + sum(x["launches_per_step"] * x["steps"]
                                                                  for x in extras),
        "clocks": m["clocks"],
        "stage_ms": {"step_median": statistics.median(m["step_ms"]),
                     "timed_kernels_median": statistics.median(m["gemm_ms"])},
    }
    if extras:
        line["also"] = [{"workload": x["wl"].name, "what": ("forward + backward" if x["wl"].backward else "forward"),
                         "value": whole_job_rate(ws, x["tokens_per_step"], x["steps"], x["total_ms"]),
                         "unit": "tokens/s", "ms_per_step": x["total_ms"] / x["steps"], "steps": x["steps"],
                         "warmup": x["warmup"], "dtype": "bf16" if x["dtype"] == mok.BF16 else "mxfp8",
                         "config": config_of(x, args, ws), "roofline": roofline(x, args), "e2e": e2e_of(x, ws),
                         "stage_rooflines": x["stage_lines"], "clocks": x["clocks"],
                         "gpu_launches": x["launches_per_step"] * x["steps"]} for x in extras]
    if torch_arm is not None:
        line["context_torch_composed"] = torch_arm
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, wl)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
