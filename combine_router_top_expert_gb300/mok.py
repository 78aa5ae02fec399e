"""Python binding of libmok.so (the C ABI in include/mok.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
Tensors are torch CUDA tensors; PyTorch supplies device memory and streams.
If the library or a CUDA device is missing, calls raise - there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmok.so")

BF16, MXFP8 = 0, 1
OK, ERR_INVALID, ERR_CUDA, ERR_TIMEOUT, ERR_CAPACITY, ERR_UNSUPPORTED = range(6)
STATUS_NAMES = {0: "MOK_OK", 1: "MOK_ERR_INVALID", 2: "MOK_ERR_CUDA", 3: "MOK_ERR_TIMEOUT",
                4: "MOK_ERR_CAPACITY", 5: "MOK_ERR_UNSUPPORTED"}

# every function declared in include/mok.h
EXPORTS = ["mok_route_workspace_size", "mok_route_layout", "mok_packed_weights_size", "mok_pack_weights",
           "mok_workspace_size", "mok_saved_size", "mok_moe_forward", "mok_padded_rows_max", "mok_dispatch",
           "mok_expert_ffn", "mok_combine", "mok_moe_backward", "mok_device_status", "mok_status_string",
           "mok_version", "mok_route_layout_static", "mok_workspace_size_batches", "mok_moe_forward_batches",
           "mok_quantize_rows", "mok_dispatch_quantized", "mok_route_test_hook", "mok_ep_workspace_size",
           "mok_ep_dispatch", "mok_ep_push", "mok_packed_weights_bwd_size", "mok_pack_weights_bwd",
           "mok_dispatch_tokens"]

FLAG_MEGAKERNEL = 1
FLAG_GEMM_PAIRS = 2
FLAG_TRACE = 4
FLAG_MB_TOKEN_RANGES = 8
FLAG_ROW_TILES = 16
FLAG_TOKEN_TILES_BALANCED = 32
FLAG_NO_L2_PREFETCH = 64
FLAG_SWAPPED_TILES = 128
FLAG_TEST_WITHHOLD_PUBLISH = 256


class MokError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("dtype", ctypes.c_int32), ("I_shared", ctypes.c_int32)]


class Config(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("timeout_ms", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("mover_ctas", ctypes.c_int32), ("minibatch_tokens", ctypes.c_int32), ("ring_rows", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


class Routing(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("row_src", ctypes.c_void_p), ("slot_row", ctypes.c_void_p)]


class FwdArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("packed", ctypes.c_void_p), ("packed_shared", ctypes.c_void_p),
                ("routing", Routing), ("out", ctypes.c_void_p), ("saved", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("W_r", ctypes.c_void_p), ("W_gate", ctypes.c_void_p),
                ("W_up", ctypes.c_void_p), ("W_down", ctypes.c_void_p), ("packed", ctypes.c_void_p),
                ("dY", ctypes.c_void_p), ("routing", Routing), ("saved", ctypes.c_void_p),
                ("dX", ctypes.c_void_p), ("dW_gate", ctypes.c_void_p), ("dW_up", ctypes.c_void_p),
                ("dW_down", ctypes.c_void_p), ("dW_r", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t), ("packed_bwd", ctypes.c_void_p)]


class EpPeer(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("offsets", ctypes.c_void_p), ("row_src", ctypes.c_void_p),
                ("partials", ctypes.c_void_p), ("T", ctypes.c_int32)]


EP_MAX_RANKS = 8
_lock = threading.Lock()
_lib = None


def lib():
    """Load libmok.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libmok.so not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            PP = ctypes.POINTER(Problem)
            PC = ctypes.POINTER(Config)
            PR = ctypes.POINTER(Routing)
            L.mok_route_workspace_size.argtypes = [I32] * 4
            L.mok_route_workspace_size.restype = SZ
            L.mok_route_layout.argtypes = [P, P, P, I32, I32, I32, I32, P, P, P, P, P, P, P, SZ, P]
            L.mok_route_layout_static.argtypes = [P, P, P, I32, I32, I32, I32, P, P, P, P, P, P, P]
            L.mok_packed_weights_size.argtypes = [I32] * 4
            L.mok_packed_weights_size.restype = SZ
            L.mok_pack_weights.argtypes = [I32, I32, I32, I32, P, P, P, P, SZ, P]
            L.mok_packed_weights_bwd_size.argtypes = [I32] * 4
            L.mok_packed_weights_bwd_size.restype = SZ
            L.mok_pack_weights_bwd.argtypes = [I32, I32, I32, I32, P, P, P, P, SZ, P]
            L.mok_workspace_size.argtypes = [PP, PC]
            L.mok_workspace_size.restype = SZ
            L.mok_saved_size.argtypes = [PP]
            L.mok_saved_size.restype = SZ
            L.mok_moe_forward.argtypes = [PP, ctypes.POINTER(FwdArgs), PC, P]
            L.mok_moe_forward_batches.argtypes = [PP, I32, ctypes.POINTER(FwdArgs), PC, P]
            L.mok_workspace_size_batches.argtypes = [PP, I32, PC]
            L.mok_workspace_size_batches.restype = SZ
            L.mok_padded_rows_max.argtypes = [I32, I32, I32]
            L.mok_padded_rows_max.restype = ctypes.c_int64
            L.mok_dispatch.argtypes = [PP, P, PR, P, P, P]
            L.mok_quantize_rows.argtypes = [P, I32, I32, P, P, P]
            L.mok_dispatch_tokens.argtypes = [PP, P, PR, P, P, P]
            L.mok_dispatch_quantized.argtypes = [PP, P, P, PR, P, P, P]
            L.mok_expert_ffn.argtypes = [PP, P, P, P, PR, P, P, P, PC, P, P]
            L.mok_combine.argtypes = [PP, P, P, P, P, P]
            L.mok_moe_backward.argtypes = [PP, ctypes.POINTER(BwdArgs), PC, P]
            L.mok_device_status.argtypes = [P, P, ctypes.POINTER(I32), I32]
            L.mok_route_test_hook.argtypes = [I32, I32]
            L.mok_ep_workspace_size.argtypes = [I32, I32]
            L.mok_ep_workspace_size.restype = SZ
            L.mok_ep_dispatch.argtypes = [I32, I32, I32, I32, I32, ctypes.POINTER(EpPeer), P, P, ctypes.c_int64, P, P,
                                          P, P, P, P, SZ, P]
            L.mok_ep_push.argtypes = [I32, I32, I32, I32, ctypes.POINTER(EpPeer), P, ctypes.c_int64, P, P, P, P]
            L.mok_status_string.argtypes = [I32]
            L.mok_status_string.restype = ctypes.c_char_p
            L.mok_version.restype = ctypes.c_char_p
            for name in ("mok_route_layout", "mok_route_layout_static", "mok_pack_weights", "mok_moe_forward",
                         "mok_moe_forward_batches", "mok_dispatch", "mok_quantize_rows", "mok_dispatch_quantized",
                         "mok_expert_ffn", "mok_combine", "mok_moe_backward", "mok_device_status", "mok_route_test_hook",
                         "mok_ep_dispatch", "mok_ep_push", "mok_pack_weights_bwd", "mok_dispatch_tokens"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc, what):
    if rc != OK:
        raise MokError(rc, what)


def _bf16(t):
    assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(), "bf16 contiguous CUDA tensor expected"
    return t


def make_problem(T, H, I, E, k, dtype=BF16, I_shared=0) -> Problem:
    return Problem(T, H, I, E, k, dtype, I_shared)


def make_config(num_sms=0, timeout_ms=0, flags=0, mover_ctas=0, minibatch_tokens=0, ring_rows=0) -> Config:
    return Config(num_sms, timeout_ms, flags, mover_ctas, minibatch_tokens, ring_rows)


# --------------------------------------------------------------------------- sizes

def route_workspace_size(T, H, E, k) -> int:
    return int(lib().mok_route_workspace_size(T, H, E, k))


def packed_weights_size(E, H, I, dtype) -> int:
    return int(lib().mok_packed_weights_size(E, H, I, dtype))


def workspace_size(p: Problem, cfg: Config | None = None) -> int:
    return int(lib().mok_workspace_size(ctypes.byref(p), ctypes.byref(cfg) if cfg else None))


def workspace_size_batches(p: Problem, nbatch: int, cfg: Config | None = None) -> int:
    return int(lib().mok_workspace_size_batches(ctypes.byref(p), nbatch, ctypes.byref(cfg) if cfg else None))


def saved_size(p: Problem) -> int:
    return int(lib().mok_saved_size(ctypes.byref(p)))


def padded_rows_max(T, E, k) -> int:
    return int(lib().mok_padded_rows_max(T, E, k))


def version() -> str:
    return lib().mok_version().decode()


# --------------------------------------------------------------------------- calls

def alloc_bytes(n, device="cuda"):
    """Device buffer of n bytes, 1024-byte aligned (torch's caching allocator
    returns 512-byte aligned blocks; one extra KiB is sliced off the front)."""
    raw = torch.empty(max(int(n), 1) + 1024, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % 1024
    return raw[off:off + max(int(n), 1)]


def route_layout(x, W_r, k, bias=None, out=None, workspace=None, stream=None):
    """Router + top-k + layout. Returns a dict of device tensors."""
    _bf16(x)
    T, H = x.shape
    E = W_r.shape[1]
    dev = x.device
    if out is None:
        out = dict(topk_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                   topk_w=torch.empty((T, k), dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   row_src=torch.empty(T * k, dtype=torch.int32, device=dev),
                   slot_row=torch.empty(T * k, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = alloc_bytes(route_workspace_size(T, H, E, k), dev)
    rc = lib().mok_route_layout(_ptr(x), _ptr(W_r), _ptr(bias), T, H, E, k, _ptr(out["topk_idx"]),
                                _ptr(out["topk_w"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                                _ptr(out["row_src"]), _ptr(out["slot_row"]), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "mok_route_layout")
    return out


ROUTE_STATIC_SCRATCH_BYTES = 8 << 20  # MOK_ROUTE_STATIC_SCRATCH_BYTES


def route_layout_static(x, W_r, k, bias=None, out=None, stream=None):
    """Routing with the library's own scratch array: no workspace argument,
    nothing allocated by the library (the outputs are still the caller's)."""
    _bf16(x)
    T, H = x.shape
    E = W_r.shape[1]
    dev = x.device
    if out is None:
        out = dict(topk_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                   topk_w=torch.empty((T, k), dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   row_src=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
                   slot_row=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev))
    rc = lib().mok_route_layout_static(_ptr(x), _ptr(W_r), _ptr(bias), T, H, E, k, _ptr(out["topk_idx"]),
                                       _ptr(out["topk_w"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                                       _ptr(out["row_src"]), _ptr(out["slot_row"]), _stream(stream))
    _check(rc, "mok_route_layout_static")
    return out


def routing_struct(r) -> Routing:
    return Routing(r["topk_idx"].data_ptr(), r["topk_w"].data_ptr(), r["counts"].data_ptr(),
                   r["offsets"].data_ptr(), r["row_src"].data_ptr(), r["slot_row"].data_ptr())


def pack_weights(Wg, Wu, Wd, dtype, packed=None, stream=None):
    E, H, I = Wg.shape
    n = packed_weights_size(E, H, I, dtype)
    if n == 0:
        raise MokError(ERR_INVALID, "mok_packed_weights_size")
    if packed is None:
        packed = alloc_bytes(n, Wg.device)
    rc = lib().mok_pack_weights(E, H, I, dtype, _ptr(_bf16(Wg)), _ptr(_bf16(Wu)), _ptr(_bf16(Wd)), _ptr(packed),
                                packed.numel(), _stream(stream))
    _check(rc, "mok_pack_weights")
    return packed


def pack_weights_bwd(Wg, Wu, Wd, dtype, packed_bwd=None, stream=None):
    """The MXFP8 backward's weight copies (None for BF16)."""
    E, H, I = Wg.shape
    n = int(lib().mok_packed_weights_bwd_size(E, H, I, dtype))
    if n == 0:
        return None
    if packed_bwd is None:
        packed_bwd = alloc_bytes(n, Wg.device)
    rc = lib().mok_pack_weights_bwd(E, H, I, dtype, _ptr(_bf16(Wg)), _ptr(_bf16(Wu)), _ptr(_bf16(Wd)),
                                    _ptr(packed_bwd), packed_bwd.numel(), _stream(stream))
    _check(rc, "mok_pack_weights_bwd")
    return packed_bwd


def moe_forward(p: Problem, x, packed, routing, out, workspace, saved=None, packed_shared=None,
                cfg: Config | None = None, stream=None):
    a = FwdArgs(x.data_ptr(), packed.data_ptr(), packed_shared.data_ptr() if packed_shared is not None else None,
                routing_struct(routing), out.data_ptr(), saved.data_ptr() if saved is not None else None,
                workspace.data_ptr(), workspace.numel())
    rc = lib().mok_moe_forward(ctypes.byref(p), ctypes.byref(a), ctypes.byref(cfg) if cfg else None, _stream(stream))
    _check(rc, "mok_moe_forward")
    return out


def moe_forward_batches(p: Problem, xs, packed, routings, outs, workspace, packed_shared=None,
                        cfg: Config | None = None, stream=None):
    """One megakernel launch over len(xs) macro-batches (same weights)."""
    n = len(xs)
    arr = (FwdArgs * n)()
    for b in range(n):
        arr[b] = FwdArgs(xs[b].data_ptr(), packed.data_ptr(),
                         packed_shared.data_ptr() if packed_shared is not None else None,
                         routing_struct(routings[b]), outs[b].data_ptr(), None, workspace.data_ptr(),
                         workspace.numel())
    rc = lib().mok_moe_forward_batches(ctypes.byref(p), n, arr, ctypes.byref(cfg) if cfg else None, _stream(stream))
    _check(rc, "mok_moe_forward_batches")
    return outs


def moe_backward(p: Problem, x, W_r, Wg, Wu, Wd, packed, dY, routing, saved, grads, workspace,
                 cfg: Config | None = None, stream=None, packed_bwd=None):
    """grads: dict with dX, dW_gate, dW_up, dW_down, dW_r (preallocated)."""
    a = BwdArgs(x.data_ptr(), W_r.data_ptr(), Wg.data_ptr(), Wu.data_ptr(), Wd.data_ptr(), packed.data_ptr(),
                dY.data_ptr(), routing_struct(routing), saved.data_ptr(), grads["dX"].data_ptr(),
                grads["dW_gate"].data_ptr(), grads["dW_up"].data_ptr(), grads["dW_down"].data_ptr(),
                grads["dW_r"].data_ptr(), workspace.data_ptr(), workspace.numel(),
                packed_bwd.data_ptr() if packed_bwd is not None else None)
    rc = lib().mok_moe_backward(ctypes.byref(p), ctypes.byref(a), ctypes.byref(cfg) if cfg else None,
                                _stream(stream))
    _check(rc, "mok_moe_backward")
    return grads


def dispatch(p: Problem, x, routing, A, A_sf=None, stream=None):
    rs = routing_struct(routing)
    rc = lib().mok_dispatch(ctypes.byref(p), _ptr(x), ctypes.byref(rs), _ptr(A), _ptr(A_sf), _stream(stream))
    _check(rc, "mok_dispatch")


def dispatch_tokens(p: Problem, x, routing, A, A_sf, stream=None):
    rs = routing_struct(routing)
    rc = lib().mok_dispatch_tokens(ctypes.byref(p), _ptr(x), ctypes.byref(rs), _ptr(A), _ptr(A_sf), _stream(stream))
    _check(rc, "mok_dispatch_tokens")


def quantize_rows(x, x_q, x_sf, stream=None):
    T, H = x.shape
    rc = lib().mok_quantize_rows(_ptr(x), T, H, _ptr(x_q), _ptr(x_sf), _stream(stream))
    _check(rc, "mok_quantize_rows")


def dispatch_quantized(p: Problem, x_q, x_sf, routing, A, A_sf, stream=None):
    rs = routing_struct(routing)
    rc = lib().mok_dispatch_quantized(ctypes.byref(p), _ptr(x_q), _ptr(x_sf), ctypes.byref(rs), _ptr(A), _ptr(A_sf),
                                      _stream(stream))
    _check(rc, "mok_dispatch_quantized")


def expert_ffn(p: Problem, A, A_sf, packed, routing, h, h_sf, partials, workspace, cfg: Config | None = None,
               stream=None):
    rs = routing_struct(routing)
    rc = lib().mok_expert_ffn(ctypes.byref(p), _ptr(A), _ptr(A_sf), _ptr(packed), ctypes.byref(rs), _ptr(h),
                              _ptr(h_sf), _ptr(partials), ctypes.byref(cfg) if cfg else None, _ptr(workspace),
                              _stream(stream))
    _check(rc, "mok_expert_ffn")


def combine(p: Problem, partials, topk_w, out, shared=None, stream=None):
    rc = lib().mok_combine(ctypes.byref(p), _ptr(partials), _ptr(topk_w), _ptr(shared), _ptr(out), _stream(stream))
    _check(rc, "mok_combine")


def megakernel_trace(workspace, n_ctas):
    """Per-CTA megakernel records written under FLAG_TRACE: int64 [n_ctas, 8]
    (role, t_begin, t_first, t_work_end, t_exit, wait_ns, units, combine_ns)."""
    return workspace[256:256 + 64 * n_ctas].view(torch.int64).view(n_ctas, 8).cpu().numpy()


def route_test_hook(withhold_copy, timeout_ms=0):
    """Test hook of the routing kernels' bounded waits (see mok.h)."""
    _check(lib().mok_route_test_hook(int(withhold_copy), int(timeout_ms)), "mok_route_test_hook")


def device_status(workspace, reset=False, stream=None):
    """(status code, detail) recorded on the device by the last call; with
    workspace None, the last mok_route_layout_static call on this device."""
    d = ctypes.c_int32(0)
    rc = lib().mok_device_status(_ptr(workspace), _stream(stream), ctypes.byref(d), int(reset))
    return int(rc), int(d.value)


def check_device_status(workspace, what="device", stream=None):
    rc, d = device_status(workspace, stream=stream)
    if rc != OK:
        raise MokError(rc, f"{what} (detail {d})")


# --------------------------------------------------------------------------- expert parallelism

def ep_workspace_size(G, E) -> int:
    return int(lib().mok_ep_workspace_size(G, E))


def _peers(peers):
    arr = (EpPeer * len(peers))()
    for i, q in enumerate(peers):
        arr[i] = EpPeer(q["x"].data_ptr() if q.get("x") is not None else None, q["offsets"].data_ptr(),
                        q["row_src"].data_ptr() if q.get("row_src") is not None else None,
                        q["partials"].data_ptr() if q.get("partials") is not None else None, int(q["T"]))
    return arr


def ep_dispatch(G, rank, H, E, k, peers, counts_all, A, rows_cap, counts_local, offsets_local, src_rank, src_slot,
                ident, workspace, stream=None):
    """peers: list of G dicts {x, offsets, row_src, partials, T} (device tensors)."""
    rc = lib().mok_ep_dispatch(G, rank, H, E, k, _peers(peers), _ptr(counts_all), _ptr(A), int(rows_cap),
                               _ptr(counts_local), _ptr(offsets_local), _ptr(src_rank), _ptr(src_slot), _ptr(ident),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mok_ep_dispatch")


def ep_push(G, H, E, k, peers, ys, rows_cap, offsets_local, src_rank, src_slot, stream=None):
    rc = lib().mok_ep_push(G, H, E, k, _peers(peers), _ptr(ys), int(rows_cap), _ptr(offsets_local), _ptr(src_rank),
                           _ptr(src_slot), _stream(stream))
    _check(rc, "mok_ep_push")
