"""Shared test helpers: device transfer and the tolerance metric.

Tolerance metric (per output tensor): c = 2e-2 for BF16 operands and 5e-2 for
MXFP8 operands, and
    max_i ( |gpu_i - ref_i| - ulp_half_i ) <= c * rms(ref)
where ref is the oracle's fp64 value and ulp_half_i is half a BF16 ulp of
ref_i when the GPU output is BF16 (0 for fp32 outputs). The rounding of the
result to the BF16 output format is part of the format, not an error of the
computation: a perfect computation rounded once to BF16 already differs from
the fp64 value by up to half an ulp, which at a 6-sigma element alone is
~2.3% of rms. The raw max|d|/rms is reported as well.
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


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Half the spacing of BF16 values at |ref| (8 significant bits)."""
    a = np.abs(ref.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def rel_err(gpu: np.ndarray, ref: np.ndarray, bf16_out: bool = True):
    """(raw max|d|/rms, max(|d| - half BF16 ulp)/rms)."""
    ref = ref.astype(np.float64)
    rms = max(float(np.sqrt(np.mean(ref ** 2))), 1e-300)
    d = np.abs(gpu.astype(np.float64) - ref)
    raw = float(d.max()) / rms
    adj = float(np.max(d - (half_ulp_bf16(ref) if bf16_out else 0.0))) / rms
    return raw, adj


def assert_close(gpu, ref, c, what="", bf16_out=True):
    raw, adj = rel_err(gpu, ref, bf16_out)
    print(f"[parity] {what}: max|d|/rms={raw:.3e}, beyond output rounding={adj:.3e} (tol {c:.0e})")
    assert adj <= c, f"{what}: max(|d| - ulp/2)/rms = {adj:.3e} > {c:.1e} (raw {raw:.3e})"
    return adj


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
