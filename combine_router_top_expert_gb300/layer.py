"""A routed MoE layer on one GPU, driven through the C ABI.

PyTorch allocates the device buffers and supplies the stream; every step of
the layer (routing, dispatch, grouped expert GEMMs, combine, backward) runs
in libmok.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mok


def to_dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """BF16 bit patterns (uint16) -> bf16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


class MoELayer:
    def __init__(self, W_r, Wg, Wu, Wd, k, dtype=mok.BF16, bias=None, shared=None, device="cuda",
                 keep_unpacked=True):
        """Weights as host numpy arrays (BF16 as uint16 bit patterns, W_r/bias fp32)."""
        self.device = device
        self.k = k
        self.dtype = dtype
        self.H, self.E = W_r.shape
        self.I = Wg.shape[2]
        self.W_r = torch.from_numpy(np.ascontiguousarray(W_r, dtype=np.float32)).to(device)
        self.bias = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, dtype=np.float32)).to(device)
        Wg_d, Wu_d, Wd_d = (to_dev_bf16(a, device) for a in (Wg, Wu, Wd))
        self.packed = mok.pack_weights(Wg_d, Wu_d, Wd_d, dtype)
        # MXFP8 training: the backward's weight copies, packed once like the forward's
        self.packed_bwd = mok.pack_weights_bwd(Wg_d, Wu_d, Wd_d, dtype) if keep_unpacked else None
        self.Wg, self.Wu, self.Wd = (Wg_d, Wu_d, Wd_d) if keep_unpacked else (None, None, None)
        self.I_shared = 0
        self.packed_shared = None
        if shared is not None:
            Sg, Su, Sd = (to_dev_bf16(a, device) for a in shared)
            self.I_shared = Sg.shape[1]
            self.packed_shared = mok.pack_weights(Sg[None], Su[None], Sd[None], mok.BF16)
        torch.cuda.synchronize()
        self._bufs = {}

    def problem(self, T) -> mok.Problem:
        return mok.make_problem(T, self.H, self.I, self.E, self.k, self.dtype, self.I_shared)

    def buffers(self, T, training=False, cfg=None):
        key = (T, training)
        if key not in self._bufs:
            p = self.problem(T)
            b = dict(
                route_ws=mok.alloc_bytes(mok.route_workspace_size(T, self.H, self.E, self.k), self.device),
                routing=dict(topk_idx=torch.empty((T, self.k), dtype=torch.int32, device=self.device),
                             topk_w=torch.empty((T, self.k), dtype=torch.float32, device=self.device),
                             counts=torch.empty(self.E, dtype=torch.int32, device=self.device),
                             offsets=torch.empty(self.E + 1, dtype=torch.int32, device=self.device),
                             row_src=torch.empty(max(T * self.k, 1), dtype=torch.int32, device=self.device),
                             slot_row=torch.empty(max(T * self.k, 1), dtype=torch.int32, device=self.device)),
                ws=mok.alloc_bytes(mok.workspace_size(p, cfg), self.device),
                out=torch.empty((max(T, 1), self.H), dtype=torch.bfloat16, device=self.device),
            )
            if training:
                b["saved"] = mok.alloc_bytes(mok.saved_size(p), self.device)
            self._bufs[key] = b
        return self._bufs[key]

    def route(self, x, training=False, stream=None):
        b = self.buffers(x.shape[0], training)
        return mok.route_layout(x, self.W_r, self.k, self.bias, out=b["routing"], workspace=b["route_ws"],
                                stream=stream)

    def forward(self, x, training=False, cfg=None, stream=None, route=True, out=None):
        """out [T, H] bf16 (a view of a reused buffer unless `out` is given).
        The stage kernels run unless cfg has FLAG_MEGAKERNEL (inference only);
        training keeps the activations the backward needs."""
        T = x.shape[0]
        b = self.buffers(T, training, cfg)
        if route:
            self.route(x, training, stream)
        dst = b["out"] if out is None else out
        mok.moe_forward(self.problem(T), x, self.packed, b["routing"], dst, b["ws"],
                        saved=b.get("saved") if training else None, packed_shared=self.packed_shared, cfg=cfg,
                        stream=stream)
        return dst[:T]

    def backward(self, x, dY, cfg=None, stream=None, grads=None):
        T = x.shape[0]
        b = self.buffers(T, True)
        if grads is None:
            grads = dict(dX=torch.empty_like(x), dW_gate=torch.empty_like(self.Wg), dW_up=torch.empty_like(self.Wu),
                         dW_down=torch.empty_like(self.Wd),
                         dW_r=torch.empty((self.H, self.E), dtype=torch.float32, device=self.device))
        mok.moe_backward(self.problem(T), x, self.W_r, self.Wg, self.Wu, self.Wd, self.packed, dY, b["routing"],
                         b["saved"], grads, b["ws"], cfg=cfg, stream=stream, packed_bwd=self.packed_bwd)
        return grads

    def status(self, T, training=False):
        return mok.device_status(self.buffers(T, training)["ws"])
