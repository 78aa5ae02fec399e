// ep.cu - expert parallelism across ranks: pull-dispatch from the ranks that
// own the tokens, push-combine back to them.
//
// The pages' layer spans many GPUs: experts are partitioned across GPUs,
// the expert side pulls the token rows it needs from the GPUs that hold them
// ("pull dispatch"), and each result row is pushed back to the slot of the
// token it belongs to ("push combine"), over NVLink with GPU-local signalling
// instead of a collective library (KuCoin article on MoK, section 02;
// RuntimeWire, "Rebuilding the MoE layer around communication"). Here rank g
// of G owns experts [g*E/G, (g+1)*E/G). Every rank routes its own tokens
// over all E experts; the per-rank expert counts are all-gathered by the
// caller; then each rank
//   1. lays out the rows of its local experts (mok_ep_dispatch, plan step):
//      local expert l's rows ordered by source rank, then by the source's
//      own layout order (ascending token);
//   2. pulls each row from its source rank's x through a table of per-rank
//      base pointers (plain 16-byte loads; on one node the pointers map the
//      peers' memory);
//   3. runs the grouped expert GEMMs on them (mok_expert_ffn, unchanged);
//   4. pushes each result row to its source rank's slot buffer (mok_ep_push,
//      plain 16-byte stores);
// and, once every rank's pushes are done, sums its own slots in fixed order
// (mok_combine). No TMA and no multicast touch peer memory.
#include <algorithm>

#include "common.cuh"
#include "moves.cuh"

namespace mok {

struct EpPeers {
    const __nv_bfloat16* x[MOK_EP_MAX_RANKS];
    const int32_t* offsets[MOK_EP_MAX_RANKS];
    const int32_t* row_src[MOK_EP_MAX_RANKS];
    __nv_bfloat16* partials[MOK_EP_MAX_RANKS];
    int T[MOK_EP_MAX_RANKS];
};

// Workspace of the plan: seg_off [E_l * G + 1] (first local row of each
// (local expert, source rank) segment), poff [E_l + 1] (padded offsets of
// the local experts' segments in A).
size_t ep_workspace_ints(int G, int El) { return (size_t)El * G + 1 + El + 1; }

__global__ void ep_plan_kernel(int G, int e0, int El, int E, const int32_t* __restrict__ counts_all,
                               int32_t* __restrict__ counts_l, int32_t* __restrict__ offsets_l,
                               int32_t* __restrict__ seg_off, int32_t* __restrict__ poff) {
    if (threadIdx.x != 0) return;
    int row = 0, prow = 0;
    for (int l = 0; l < El; ++l) {
        offsets_l[l] = row;
        poff[l] = prow;
        int n = 0;
        for (int s = 0; s < G; ++s) {
            seg_off[l * G + s] = row + n;
            n += counts_all[(int64_t)s * E + e0 + l];
        }
        counts_l[l] = n;
        row += n;
        prow += ceil_div(n, kTileM) * kTileM;
    }
    offsets_l[El] = row;
    seg_off[El * G] = row;
    poff[El] = prow;
}

// Pull: one warp per local row. Row -> (local expert, source rank) segment by
// binary search on seg_off; the source's layout names the slot t*k + j, the
// row copies x_s[t] into the padded expert-contiguous A.
__global__ void __launch_bounds__(256)
ep_pull_kernel(EpPeers peers, int G, int e0, int El, int H, int k, const int32_t* __restrict__ seg_off,
               const int32_t* __restrict__ offsets_l, const int32_t* __restrict__ poff,
               __nv_bfloat16* __restrict__ A, int32_t* __restrict__ src_rank, int32_t* __restrict__ src_slot,
               int32_t* __restrict__ ident, int64_t rows_cap) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = (int)min((int64_t)offsets_l[El], rows_cap);
    const int nseg = El * G;
    for (int row = blockIdx.x * 8 + warp; row < total; row += gridDim.x * 8) {
        int lo = 0, hi = nseg - 1;   // last segment with seg_off <= row (empty segments skipped)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seg_off[mid] <= row) lo = mid; else hi = mid - 1;
        }
        const int l = lo / G, s = lo % G;
        const int r = row - seg_off[lo];
        // the gathered counts must agree with the source's layout and slots:
        // a row that does not is skipped (marked rank -1, never pushed)
        const int base = peers.offsets[s][e0 + l];
        const int32_t slot = r < peers.offsets[s][e0 + l + 1] - base ? peers.row_src[s][base + r] : -1;
        const int64_t arow = (int64_t)poff[l] + row - offsets_l[l];
        if (slot < 0 || slot >= peers.T[s] * k || arow >= rows_cap) {
            if (lane == 0) {
                src_rank[row] = -1;
                src_slot[row] = 0;
                ident[row] = row;
            }
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(peers.x[s] + (int64_t)(slot / k) * H);
        uint4* dst = reinterpret_cast<uint4*>(A + arow * H);
        const int n = H / 8;
        for (int c = lane; c < n; c += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + 32 * u < n) v[u] = src[c + 32 * u];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + 32 * u < n) dst[c + 32 * u] = v[u];
        }
        if (lane == 0) {
            src_rank[row] = s;
            src_slot[row] = slot;
            ident[row] = row;
        }
    }
}

// Push: one warp per local row: ys[row] -> partials of its source rank at the
// row's slot.
__global__ void __launch_bounds__(256)
ep_push_kernel(EpPeers peers, int G, int El, int H, int k, const int32_t* __restrict__ offsets_l,
               const __nv_bfloat16* __restrict__ ys, const int32_t* __restrict__ src_rank,
               const int32_t* __restrict__ src_slot, int64_t rows_cap) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = (int)min((int64_t)offsets_l[El], rows_cap);
    for (int row = blockIdx.x * 8 + warp; row < total; row += gridDim.x * 8) {
        const int s = src_rank[row], slot = src_slot[row];
        if (s < 0 || s >= G || slot < 0 || slot >= peers.T[s] * k) continue;   // skipped by the pull
        const uint4* src = reinterpret_cast<const uint4*>(ys + (int64_t)row * H);
        uint4* dst = reinterpret_cast<uint4*>(peers.partials[s] + (int64_t)slot * H);
        const int n = H / 8;
        for (int c = lane; c < n; c += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + 32 * u < n) v[u] = src[c + 32 * u];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + 32 * u < n) dst[c + 32 * u] = v[u];
        }
    }
}

namespace {

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool peers_ok(const mok_ep_peer* peers, int G, bool need_partials) {
    if (!peers) return false;
    for (int s = 0; s < G; ++s) {
        if (peers[s].T < 0) return false;
        if (peers[s].T > 0 && (!peers[s].x || !a16(peers[s].x) || !peers[s].row_src)) return false;
        if (!peers[s].offsets) return false;
        if (need_partials && peers[s].T > 0 && (!peers[s].partials || !a16(peers[s].partials))) return false;
    }
    return true;
}

EpPeers to_kernel(const mok_ep_peer* peers, int G) {
    EpPeers k{};
    for (int s = 0; s < G; ++s) {
        k.x[s] = static_cast<const __nv_bfloat16*>(peers[s].x);
        k.offsets[s] = peers[s].offsets;
        k.row_src[s] = peers[s].row_src;
        k.partials[s] = static_cast<__nv_bfloat16*>(peers[s].partials);
        k.T[s] = peers[s].T;
    }
    return k;
}

int blocks_for(int64_t rows) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (rows + 7) / 8;
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 8));
}

}  // namespace
}  // namespace mok

using namespace mok;

extern "C" size_t mok_ep_workspace_size(int32_t G, int32_t E) {
    if (G < 1 || G > MOK_EP_MAX_RANKS || E < G || E % G) return 0;
    return align_up((int64_t)ep_workspace_ints(G, E / G) * 4, 256);
}

extern "C" mok_status mok_ep_dispatch(int32_t G, int32_t rank, int32_t H, int32_t E, int32_t k,
                                      const mok_ep_peer* peers, const int32_t* counts_all, void* A,
                                      int64_t rows_cap, int32_t* counts_local, int32_t* offsets_local,
                                      int32_t* src_rank, int32_t* src_slot, int32_t* ident, void* workspace,
                                      size_t ws_bytes, mok_stream_t stream) {
    if (G < 1 || G > MOK_EP_MAX_RANKS || rank < 0 || rank >= G || E < G || E % G || E > kMaxE) return MOK_ERR_INVALID;
    if (H <= 0 || H % 8 || k < 1 || k > E) return MOK_ERR_INVALID;
    if (!peers_ok(peers, G, false) || !counts_all || !A || !a16(A) || !counts_local || !offsets_local || !src_rank ||
        !src_slot || !ident || !workspace || ws_bytes < mok_ep_workspace_size(G, E))
        return MOK_ERR_INVALID;
    const int El = E / G;
    int64_t rows_all = 0;   // every routed row of every rank could land here
    for (int s = 0; s < G; ++s) rows_all += (int64_t)peers[s].T * k;
    if (rows_cap < rows_all + (int64_t)kTileM * El) return MOK_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t* w = static_cast<int32_t*>(workspace);
    int32_t* seg_off = w;
    int32_t* poff = w + El * G + 1;
    ep_plan_kernel<<<1, 32, 0, s>>>(G, rank * El, El, E, counts_all, counts_local, offsets_local, seg_off, poff);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return MOK_ERR_CUDA;
    if (rows_all == 0) return MOK_OK;
    ep_pull_kernel<<<blocks_for(rows_all), 256, 0, s>>>(to_kernel(peers, G), G, rank * El, El, H, k, seg_off,
                                                        offsets_local, poff, static_cast<__nv_bfloat16*>(A),
                                                        src_rank, src_slot, ident, rows_cap);
    return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

extern "C" mok_status mok_ep_push(int32_t G, int32_t H, int32_t E, int32_t k, const mok_ep_peer* peers,
                                  const void* ys, int64_t rows_cap, const int32_t* offsets_local,
                                  const int32_t* src_rank, const int32_t* src_slot, mok_stream_t stream) {
    if (G < 1 || G > MOK_EP_MAX_RANKS || E < G || E % G || H <= 0 || H % 8 || k < 1) return MOK_ERR_INVALID;
    if (!peers_ok(peers, G, true) || !ys || !a16(ys) || !offsets_local || !src_rank || !src_slot || rows_cap < 0)
        return MOK_ERR_INVALID;
    int64_t rows_all = 0;
    for (int s = 0; s < G; ++s) rows_all += (int64_t)peers[s].T * k;
    if (rows_all == 0) return MOK_OK;
    ep_push_kernel<<<blocks_for(rows_all), 256, 0, (cudaStream_t)stream>>>(
        to_kernel(peers, G), G, E / G, H, k, offsets_local, static_cast<const __nv_bfloat16*>(ys), src_rank, src_slot,
        rows_cap);
    return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
