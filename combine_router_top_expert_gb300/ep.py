"""Expert parallelism across ranks, driven through the C ABI.

Rank g of G owns experts [g*E/G, (g+1)*E/G) (the pages' "E local experts"
per GPU, KuCoin article on MoK, section 02). Each step: every rank routes its
own tokens over all E experts; the per-rank expert counts are all-gathered
(a [G, E] int32 collective, the only host-side collective of the step);
every rank pulls the rows of its local experts from their source ranks
(mok_ep_dispatch), runs its grouped expert GEMMs (mok_expert_ffn), pushes
each result row to its source rank's slot buffer (mok_ep_push); after a
barrier every rank sums its own slots in fixed order (mok_combine).

`EPRank` holds one rank's local expert weights and buffers. On one GPU,
`forward_logical` runs G ranks as separate allocations of the same device,
stream-ordered (every rank's routing before any pull, every push before any
combine), which is how the path is tested here. Across GPUs the peer table
must hold pointers that map the peers' allocations and the barriers are the
process group's; that path is unmeasured on hardware.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mok


def local_experts(rank: int, G: int, E: int) -> range:
    if E % G:
        raise ValueError("E must be a multiple of the rank count")
    El = E // G
    return range(rank * El, (rank + 1) * El)


def plan_host(counts_all: np.ndarray, rank: int):
    """The plan mok_ep_dispatch builds on the device, in numpy: for local
    expert l, counts_local[l] = sum_s counts_all[s, e]; offsets_local
    (unpadded, E/G + 1); seg_off[l*G + s] = first local row of source s's
    rows of local expert l (rows ordered by expert, then source rank)."""
    counts_all = np.asarray(counts_all, np.int64)
    G, E = counts_all.shape
    el = list(local_experts(rank, G, E))
    counts_l = counts_all[:, el].sum(0)
    offsets_l = np.concatenate([[0], np.cumsum(counts_l)])
    seg = [0]
    for l in range(len(el)):
        for s in range(G):
            seg.append(seg[-1] + counts_all[s, el[l]])
    return counts_l.astype(np.int32), offsets_l.astype(np.int32), np.array(seg, np.int32)


def pulled_slots_host(counts_all, rank, offsets_all, row_src_all):
    """(source rank, slot) of every local row of `rank` in local row order,
    from the sources' layouts (host reference of the pull's bookkeeping)."""
    G, E = np.asarray(counts_all).shape
    out = []
    for e in local_experts(rank, G, E):
        for s in range(G):
            o = offsets_all[s]
            for r in range(int(o[e + 1] - o[e])):
                out.append((s, int(row_src_all[s][o[e] + r])))
    return out


def gather_counts(counts: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of this rank's expert counts [E] into [G, E] (rank-major)
    over the process group (gloo on CPU tensors, NCCL on device tensors)."""
    import torch.distributed as dist
    G = dist.get_world_size(group)
    out = torch.empty(G * counts.numel(), dtype=counts.dtype, device=counts.device)
    dist.all_gather_into_tensor(out, counts.contiguous().view(-1), group=group)
    return out.view(G, counts.numel())


class EPRank:
    """One rank: its slice of the experts (packed), its routing and buffers."""

    def __init__(self, rank, G, W_r, Wg, Wu, Wd, k, T_cap, bias=None, device="cuda"):
        from .layer import to_dev_bf16
        self.rank, self.G, self.k = rank, G, k
        self.H, self.E = W_r.shape
        self.I = Wg.shape[2]
        self.El = self.E // G
        el = local_experts(rank, G, self.E)
        self.W_r = torch.from_numpy(np.ascontiguousarray(W_r, dtype=np.float32)).to(device)
        self.bias = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).to(device)
        sl = slice(el.start, el.stop)
        self.packed = mok.pack_weights(*(to_dev_bf16(np.ascontiguousarray(a[sl]), device) for a in (Wg, Wu, Wd)),
                                       mok.BF16)
        self.T_cap = T_cap
        self.device = device
        self.rows_cap = G * T_cap * k + 128 * self.El
        dev = device
        self.route_ws = mok.alloc_bytes(mok.route_workspace_size(T_cap, self.H, self.E, k), dev)
        self.ep_ws = mok.alloc_bytes(mok.ep_workspace_size(G, self.E), dev)
        self.A = mok.alloc_bytes(self.rows_cap * self.H * 2, dev)
        self.counts_local = torch.empty(self.El, dtype=torch.int32, device=dev)
        self.offsets_local = torch.empty(self.El + 1, dtype=torch.int32, device=dev)
        self.src_rank = torch.empty(self.rows_cap, dtype=torch.int32, device=dev)
        self.src_slot = torch.empty(self.rows_cap, dtype=torch.int32, device=dev)
        self.ident = torch.empty(self.rows_cap, dtype=torch.int32, device=dev)
        self.p_local = mok.make_problem(self.rows_cap - 128 * self.El, self.H, self.I, self.El, 1, mok.BF16)
        self.rows_pad = mok.padded_rows_max(self.p_local.T, self.El, 1)
        self.h = mok.alloc_bytes(self.rows_pad * self.I * 2, dev)
        self.ys = mok.alloc_bytes(self.p_local.T * self.H * 2, dev)
        self.ffn_ws = mok.alloc_bytes(mok.workspace_size(self.p_local), dev)
        self.partials = mok.alloc_bytes(T_cap * k * self.H * 2, dev)
        self.routing = None

    def route(self, x):
        self.T = x.shape[0]
        self.x = x
        self.routing = mok.route_layout(x, self.W_r, self.k, self.bias, workspace=self.route_ws)
        return self.routing["counts"]

    def peer(self):
        return {"x": self.x, "offsets": self.routing["offsets"], "row_src": self.routing["row_src"],
                "partials": self.partials, "T": self.T}

    def expert_step(self, peers, counts_all, cfg=None):
        """Pull, grouped expert GEMMs on the local experts, push."""
        mok.ep_dispatch(self.G, self.rank, self.H, self.E, self.k, peers, counts_all, self.A, self.rows_cap,
                        self.counts_local, self.offsets_local, self.src_rank, self.src_slot, self.ident, self.ep_ws)
        r = {"topk_idx": self.ident, "topk_w": self.ident, "counts": self.counts_local,
             "offsets": self.offsets_local, "row_src": self.ident, "slot_row": self.ident}
        mok.expert_ffn(self.p_local, self.A, None, self.packed, r, self.h, None, self.ys, self.ffn_ws, cfg=cfg)
        mok.ep_push(self.G, self.H, self.E, self.k, peers, self.ys, self.rows_cap, self.offsets_local,
                    self.src_rank, self.src_slot)

    def combine(self, out):
        p = mok.make_problem(self.T, self.H, self.I, self.E, self.k, mok.BF16)
        mok.combine(p, self.partials, self.routing["topk_w"], out)
        return out


def forward_logical(ranks, xs, cfg=None):
    """G ranks as separate allocations of one GPU, stream-ordered: route all,
    gather the counts, every rank's pull / GEMMs / push, then every rank's
    fixed-order sum. Returns each rank's output [T_r, H] bf16."""
    counts_all = torch.stack([rk.route(x) for rk, x in zip(ranks, xs)])
    peers = [rk.peer() for rk in ranks]
    for rk in ranks:
        rk.expert_step(peers, counts_all, cfg)
    return [rk.combine(torch.empty((x.shape[0], rk.H), dtype=torch.bfloat16, device=x.device))
            for rk, x in zip(ranks, xs)]
