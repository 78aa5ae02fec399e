"""Shared test helpers: device transfer and the tolerance metric.

Tolerance metric (per output tensor): max_i |gpu_i - ref_i| <= c * rms(ref),
c = 2e-2 for BF16 operands and 5e-2 for MXFP8 operands.
"""
import numpy as np
import torch

from combine_router_top_expert_gb300 import mok, synth
from combine_router_top_expert_gb300.layer import MoELayer, to_dev_bf16

TOL = {mok.BF16: 2e-2, mok.MXFP8: 5e-2}


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    return float(np.max(np.abs(gpu.astype(np.float64) - ref))) / max(rms, 1e-300)


def assert_close(gpu, ref, c, what=""):
    e = rel_err(gpu, ref)
    assert e <= c, f"{what}: max|d|/rms = {e:.3e} > {c:.1e}"
    return e


def layer_for(inp, dtype):
    return MoELayer(inp.W_r, inp.Wg, inp.Wu, inp.Wd, inp.wl.k, dtype=dtype, bias=inp.bias, shared=inp.shared)


def dtype_of(wl):
    return mok.MXFP8 if wl.dtype == "mxfp8" else mok.BF16


def untile_sf(sf_tiled: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Scales from the tensor-core chunk order back to [rows, cols/32]:
    chunk (rt, kc) at (rt * (cols/128) + kc) * 512, byte (r%32)*16 + (r//32)*4 + j."""
    nkc = cols // 128
    out = np.empty((rows, cols // 32), np.uint8)
    r = np.arange(rows)
    for b in range(cols // 32):
        kc, j = b // 4, b % 4
        off = ((r // 128) * nkc + kc) * 512 + (r % 128 % 32) * 16 + ((r % 128) // 32) * 4 + j
        out[:, b] = sf_tiled[off]
    return out
