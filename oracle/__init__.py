"""CPU oracle of the routed MoE layer (ctypes loader for ``mok_oracle.c``).

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg import this module. The CUDA library and its
Python binding never import it; the two share no code.

Every function here marshals numpy arrays into the C oracle and back; the
arithmetic lives in ``mok_oracle.c`` (fp64, plain loops, OpenMP across rows),
whose comments cite the passages of the pages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mok_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmok_oracle.so")
_lock = threading.Lock()
_lib = None

MODE_BF16, MODE_MXFP8, MODE_EXACT = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmok_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.orc_router_logits.argtypes = [P, P, P, I, I, I, P]
            L.orc_router_logits_f64.argtypes = [P, P, P, I, I, I, P]
            L.orc_topk_f32.argtypes = [P, I, I, I, P, P]
            L.orc_topk_f64.argtypes = [P, I, I, I, P, P]
            L.orc_layout.argtypes = [P, I, I, I, P, P, P, P]
            L.orc_moe_forward.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, P, I, P, I,
                                          P, P, P, I, P, P]
            L.orc_moe_backward.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, I,
                                           P, P, P, P, P]
            L.orc_moe_backward_sampled.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, I, P, I, P, P, I,
                                                   P, P, P, P]
            L.orc_moe_backward_sampled_mx.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, I, P, P, I,
                                                      P, P, P, P]
            L.orc_router_grad_columns.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, P, P, I, P, I, P]
            L.orc_mx_quantize_rows.argtypes = [P, I64, I64, P, P]
            L.orc_mx_quantize_bf16_rows.argtypes = [P, I64, I64, P, P]
            L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_value.restype = ctypes.c_double
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e8m0_code.argtypes = [ctypes.c_double]
            L.orc_round_bf16.argtypes = [ctypes.c_double]
            L.orc_round_bf16.restype = ctypes.c_double
            L.orc_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bf16(a: np.ndarray) -> np.ndarray:
    """BF16 bit patterns as a contiguous uint16 array."""
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "BF16 inputs travel as uint16 bit patterns"
    return a


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed (rc={rc})")


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ----------------------------------------------------------------------------- routing

def router_logits(x_bf16, W_r, bias=None):
    """fp32 logits [T, E] in the canonical summation order."""
    x = _bf16(x_bf16)
    T, H = x.shape
    W_r = np.ascontiguousarray(W_r, dtype=np.float32)
    E = W_r.shape[1]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), np.float32)
    _check(lib().orc_router_logits(_p(x), _p(W_r), _p(b), T, H, E, _p(out)), "router_logits")
    return out


def router_logits_f64(x, W_r, bias=None):
    x = np.ascontiguousarray(x, dtype=np.float64)
    W_r = np.ascontiguousarray(W_r, dtype=np.float64)
    T, H = x.shape
    E = W_r.shape[1]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    out = np.empty((T, E), np.float64)
    _check(lib().orc_router_logits_f64(_p(x), _p(W_r), _p(b), T, H, E, _p(out)), "router_logits_f64")
    return out


def topk(logits, k):
    """(idx int32 [T,k], w fp64 [T,k]) from fp32 or fp64 logits."""
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if logits.dtype == np.float32:
        rc = lib().orc_topk_f32(_p(np.ascontiguousarray(logits)), T, E, k, _p(idx), _p(w))
    else:
        rc = lib().orc_topk_f64(_p(np.ascontiguousarray(logits, dtype=np.float64)), T, E, k, _p(idx), _p(w))
    _check(rc, "topk")
    return idx, w


def layout(idx, E):
    """(counts [E], offsets [E+1], row_src [T*k], slot_row [T*k]), all int32."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_src = np.empty(T * k, np.int32)
    slot_row = np.empty(T * k, np.int32)
    _check(lib().orc_layout(_p(idx), T, E, k, _p(counts), _p(offsets), _p(row_src), _p(slot_row)), "layout")
    return counts, offsets, row_src, slot_row


def route(x_bf16, W_r, k, bias=None):
    """Router + top-k + layout, as one dict."""
    lg = router_logits(x_bf16, W_r, bias)
    idx, w = topk(lg, k)
    counts, offsets, row_src, slot_row = layout(idx, W_r.shape[1])
    return dict(logits=lg, idx=idx, w=w, counts=counts, offsets=offsets,
                row_src=row_src, slot_row=slot_row)


# ----------------------------------------------------------------------------- MXFP8

def mx_quantize_rows(v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, cols = v.shape
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty((rows, cols // 32), np.uint8)
    _check(lib().orc_mx_quantize_rows(_p(v), rows, cols, _p(codes), _p(scales)), "mx_quantize_rows")
    return codes, scales


def mx_quantize_bf16_rows(x_bf16):
    x = _bf16(x_bf16)
    rows, cols = x.shape
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty((rows, cols // 32), np.uint8)
    _check(lib().orc_mx_quantize_bf16_rows(_p(x), rows, cols, _p(codes), _p(scales)), "mx_quantize_bf16_rows")
    return codes, scales


def e4m3_value(code: int) -> float:
    return float(lib().orc_e4m3_value(code))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e8m0_code(amax: float) -> int:
    return int(lib().orc_e8m0_code(float(amax)))


def round_bf16(v: float) -> float:
    return float(lib().orc_round_bf16(float(v)))


# ----------------------------------------------------------------------------- layer

def _inputs(arrs, f64):
    out = []
    for a in arrs:
        if a is None:
            out.append(None)
        elif f64:
            out.append(np.ascontiguousarray(a, dtype=np.float64))
        else:
            out.append(_bf16(a))
    return out


def moe_forward(x, Wg, Wu, Wd, routing, mode=MODE_BF16, tokens=None, shared=None,
                return_y=False, f64=False):
    """Layer output in fp64 for all tokens ([T, H]) or the listed ones ([n, H]).

    x [T,H], Wg/Wu [E,H,I], Wd [E,I,H]: BF16 bit patterns (uint16), or float64
    arrays when ``f64``. ``routing`` is the dict from :func:`route` (or any
    dict with idx, w, offsets, row_src). ``shared`` = (Wsg [H,Is], Wsu [H,Is],
    Wsd [Is,H]) adds the BF16 shared expert.
    """
    x, Wg, Wu, Wd = _inputs([x, Wg, Wu, Wd], f64)
    T, H = x.shape
    E, _, I = Wg.shape
    k = routing["idx"].shape[1]
    idx = np.ascontiguousarray(routing["idx"], dtype=np.int32)
    w = np.ascontiguousarray(routing["w"], dtype=np.float64)
    offsets = np.ascontiguousarray(routing["offsets"], dtype=np.int32)
    row_src = np.ascontiguousarray(routing["row_src"], dtype=np.int32)
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = T if tok is None else len(tok)
    out = np.empty((n, H), np.float64)
    y = np.empty((n, k, H), np.float64) if return_y else None
    Wsg = Wsu = Wsd = None
    Is = 0
    if shared is not None:
        Wsg, Wsu, Wsd = _inputs(shared, f64)
        Is = Wsg.shape[1]
    rc = lib().orc_moe_forward(_p(x), _p(Wg), _p(Wu), _p(Wd), int(f64), T, H, I, E, k,
                               _p(idx), _p(w), _p(offsets), _p(row_src), mode,
                               _p(tok), n, _p(Wsg), _p(Wsu), _p(Wsd), Is, _p(out), _p(y))
    _check(rc, "moe_forward")
    return (out, y) if return_y else out


def moe_backward(x, W_r, Wg, Wu, Wd, dY, routing, mode=MODE_BF16, f64=False):
    """(dX [T,H], dWg [E,H,I], dWu [E,H,I], dWd [E,I,H], dWr [H,E]) in fp64."""
    x, Wg, Wu, Wd, dY = _inputs([x, Wg, Wu, Wd, dY], f64)
    W_r = np.ascontiguousarray(W_r, dtype=np.float64 if f64 else np.float32)
    T, H = x.shape
    E, _, I = Wg.shape
    k = routing["idx"].shape[1]
    idx = np.ascontiguousarray(routing["idx"], dtype=np.int32)
    w = np.ascontiguousarray(routing["w"], dtype=np.float64)
    offsets = np.ascontiguousarray(routing["offsets"], dtype=np.int32)
    row_src = np.ascontiguousarray(routing["row_src"], dtype=np.int32)
    dX = np.empty((T, H), np.float64)
    dWg = np.empty((E, H, I), np.float64)
    dWu = np.empty((E, H, I), np.float64)
    dWd = np.empty((E, I, H), np.float64)
    dWr = np.empty((H, E), np.float64)
    rc = lib().orc_moe_backward(_p(x), _p(W_r), _p(Wg), _p(Wu), _p(Wd), _p(dY), int(f64),
                                T, H, I, E, k, _p(idx), _p(w), _p(offsets), _p(row_src), mode,
                                _p(dX), _p(dWg), _p(dWu), _p(dWd), _p(dWr))
    _check(rc, "moe_backward")
    return dX, dWg, dWu, dWd, dWr


def moe_backward_sampled(x, W_r, Wg, Wu, Wd, dY, routing, tokens, cols, mode=MODE_BF16):
    """Selected backward outputs: dX rows of `tokens` [n, H]; for each (e, i)
    in `cols`: dW_gate[e][:, i], dW_up[e][:, i], dW_down[e][i, :] (each [n_col, H])."""
    x, Wg, Wu, Wd, dY = _inputs([x, Wg, Wu, Wd, dY], False)
    W_r = np.ascontiguousarray(W_r, dtype=np.float32)
    T, H = x.shape
    E, _, I = Wg.shape
    k = routing["idx"].shape[1]
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    ce = np.ascontiguousarray([c[0] for c in cols], dtype=np.int32)
    ci = np.ascontiguousarray([c[1] for c in cols], dtype=np.int32)
    dX = np.empty((len(tok), H))
    dWg = np.empty((len(cols), H))
    dWu = np.empty((len(cols), H))
    dWd = np.empty((len(cols), H))
    if mode == MODE_MXFP8:
        rc = lib().orc_moe_backward_sampled_mx(
            _p(x), _p(W_r), _p(Wg), _p(Wu), _p(Wd), _p(dY), T, H, I, E, k,
            _p(np.ascontiguousarray(routing["idx"], dtype=np.int32)),
            _p(np.ascontiguousarray(routing["w"], dtype=np.float64)),
            _p(np.ascontiguousarray(routing["offsets"], dtype=np.int32)),
            _p(np.ascontiguousarray(routing["row_src"], dtype=np.int32)),
            _p(tok), len(tok), _p(ce), _p(ci), len(cols), _p(dX), _p(dWg), _p(dWu), _p(dWd))
        _check(rc, "moe_backward_sampled_mx")
        return dX, dWg, dWu, dWd
    rc = lib().orc_moe_backward_sampled(
        _p(x), _p(W_r), _p(Wg), _p(Wu), _p(Wd), _p(dY), T, H, I, E, k,
        _p(np.ascontiguousarray(routing["idx"], dtype=np.int32)),
        _p(np.ascontiguousarray(routing["w"], dtype=np.float64)),
        _p(np.ascontiguousarray(routing["offsets"], dtype=np.int32)),
        _p(np.ascontiguousarray(routing["row_src"], dtype=np.int32)), mode,
        _p(tok), len(tok), _p(ce), _p(ci), len(cols), _p(dX), _p(dWg), _p(dWu), _p(dWd))
    _check(rc, "moe_backward_sampled")
    return dX, dWg, dWu, dWd


def router_grad_columns(x, Wg, Wu, Wd, dY, routing, experts, mode=MODE_BF16):
    """dW_r[:, e] for each expert e in `experts` ([n, H] fp64), for inputs too
    large for the full backward (runs every routed row of the tokens that
    chose a listed expert)."""
    x, Wg, Wu, Wd, dY = _inputs([x, Wg, Wu, Wd, dY], False)
    T, H = x.shape
    E, _, I = Wg.shape
    k = routing["idx"].shape[1]
    ce = np.ascontiguousarray(experts, dtype=np.int32)
    out = np.empty((len(ce), H), np.float64)
    rc = lib().orc_router_grad_columns(
        _p(x), _p(Wg), _p(Wu), _p(Wd), _p(dY), T, H, I, E, k,
        _p(np.ascontiguousarray(routing["idx"], dtype=np.int32)),
        _p(np.ascontiguousarray(routing["w"], dtype=np.float64)),
        _p(np.ascontiguousarray(routing["offsets"], dtype=np.int32)),
        _p(np.ascontiguousarray(routing["row_src"], dtype=np.int32)), mode, _p(ce), len(ce), _p(out))
    _check(rc, "router_grad_columns")
    return out
