// route.cu - router logits, top-k, routing weights, per-expert counts and
// the expert-contiguous layout.
//
// The pages (KuCoin article on Cursor's MoK, section 01) say the router
// re-decides every step which experts each token goes to, and that before
// any data moves the system must count each expert's tokens, decide where
// each token lands, and keep the same expert's tokens adjacent so the grouped
// GEMM receives ordered input. These kernels do exactly that on one GPU, with
// no host round trip:
//   route_topk_kernel   logits (fixed fp32 order) + top-k + weights +
//                       per-block expert histogram
//   route_layout_kernel counts, offsets, and the stable (expert, token)
//                       permutation row_src / slot_row
#include "common.cuh"
#include "moves.cuh"
#include "tc.cuh"

namespace mok {

constexpr int kRouteTTMax = 32;    // tokens per CTA, at most
constexpr int kRouteTTMin = 4;     // tokens per CTA, at least (sizes the histogram)
constexpr int kRouteThreads = 256; // layout kernel
constexpr int kTopkThreads = 512;  // top-k kernel: 16 warps, two summation chains each
constexpr int kRouteChunk = 256;   // h values per pipeline chunk (32 chains x 8)
constexpr int kRouteRow = kRouteChunk + 4;   // padded shared-memory row (weights and fp32 x), in floats
constexpr uint64_t kRouteTimeoutNs = 4000000000ull;   // bound on every wait of the top-k kernel

// Router weights in the order the top-k kernel streams them: per 256-wide h
// chunk c and 32-expert group g one contiguous block [32 experts][kRouteRow]
// (zero past H and E, four pad floats per row so that rows of consecutive
// experts start four banks apart). Inside a row, h and h + 128 are adjacent
// (h < 128 at 2h, h + 128 at 2h + 1): summation chains L and L + 16 then
// advance together in one packed fp32x2 FMA. One bulk copy moves a whole
// chunk into shared memory.
__host__ __device__ inline int64_t router_chunk_floats() { return 32 * (int64_t)kRouteRow; }
__host__ __device__ inline int64_t router_copy_floats(int E, int H) {
    return (int64_t)ceil_div(H, kRouteChunk) * ceil_div(E, 32) * router_chunk_floats();
}

// Identical copies of that layout (at most 16, at most 4 MB in all): every
// CTA streams the same chunks at about the same time, and reading one of
// several copies spreads those reads over more L2 slices.
int route_wr_copies(int E, int H) {
    const int64_t one = router_copy_floats(E, H) * 4;
    int64_t r = one > 0 ? ((int64_t)4 << 20) / one : 1;
    return (int)(r < 1 ? 1 : r > 16 ? 16 : r);
}

// W_r [H, E] -> the chunk layout above, copy blockIdx.z. Grid: (8 * chunks,
// expert groups, copies), block (32, 8).
__global__ void router_weight_layout_kernel(const float* __restrict__ W_r, float* __restrict__ dst_copies, int H,
                                            int E) {
    __shared__ float tile[32][33];
    const int EG = ceil_div(E, 32);
    float* __restrict__ dst = dst_copies + (int64_t)blockIdx.z * router_copy_floats(E, H);
    const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int h = h0 + i, e = e0 + threadIdx.x;
        tile[i][threadIdx.x] = (h < H && e < E) ? W_r[(int64_t)h * E + e] : 0.f;
    }
    __syncthreads();
    const int c = h0 / kRouteChunk, hl0 = h0 % kRouteChunk;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        // expert e0 + i: row i of group blockIdx.y
        float* row = dst + ((int64_t)c * EG + blockIdx.y) * router_chunk_floats() + (int64_t)i * kRouteRow;
        const int hl = hl0 + threadIdx.x;
        row[2 * (hl & 127) + (hl >> 7)] = tile[threadIdx.x][i];
        if (hl0 + 32 == kRouteChunk && threadIdx.x < kRouteRow - kRouteChunk) row[kRouteChunk + threadIdx.x] = 0.f;
    }
}

// W_r [H, E] -> `copies` identical copies of WrT [E, H] (the backward's
// layout), back to back.
__global__ void transpose_wr_kernel(const float* __restrict__ W_r, float* __restrict__ WrT_copies, int H, int E) {
    __shared__ float tile[32][33];
    float* __restrict__ WrT = WrT_copies + (int64_t)blockIdx.z * E * H;   // copy blockIdx.z
    int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        int h = h0 + i, e = e0 + threadIdx.x;
        tile[i][threadIdx.x] = (h < H && e < E) ? W_r[(int64_t)h * E + e] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        int e = e0 + i, h = h0 + threadIdx.x;
        if (e < E && h < H) WrT[(int64_t)e * H + h] = tile[threadIdx.x][i];
    }
}

// Ranking key: larger logit first, lower expert index on ties (+0 == -0).
__device__ __forceinline__ bool ranks_before(float va, int ea, float vb, int eb) {
    return va > vb || (va == vb && ea < eb);
}

// One CTA = TT tokens x all experts, 16 warps.
//
// Work split. Warp w owns summation chains w and w + 16 (chain L: h = 256*i
// + 8*L + m) for every token and expert of the CTA. Each lane is one (token
// slot tl < 4, expert slot el < 8) and accumulates tokens tl + 4u (u < TT/4)
// x experts el + 8v (v < 4) of the current 32-expert group on both of its
// warp's chains, as the two halves of a float2 advanced by packed fp32x2
// FMAs: h of chain w and h + 128 of chain w + 16 sit side by side in shared
// memory, and each half is an ordinary fp32 FMA, so every chain keeps its
// order and its bits. One 16-byte load (two h of both chains) feeds 4 or
// TT/4 tokens' FMAs.
//
// Shared-memory reads. The lanes of a warp read only 4 (x) or 8 (weights)
// distinct rows, 16 B each, four banks apart. A 128-bit shared load costs as
// many wavefronts as the most distinct addresses among any four aligned
// lanes, and at least two (measured on this GPU), so lane bits 0 and 1 pick
// one bit of tl and one of el: every quad reads two x and two weight rows
// and both loads take the minimum of two wavefronts.
//
// Data flow. The chunks (c, g) of the router weights (one bulk copy each,
// from the layout above) and the matching [TT tokens x 256 h] box of raw x
// (one tensor copy; tokens past T and h past H read 0) stream through a
// STAGES-deep ring, one mbarrier per slot; thread 0 issues the copies. x is
// widened to fp32 (in the paired h order) once per CTA, one chunk ahead,
// into a double buffer. After a group's last chunk the 32 chains of every
// (token, expert) are added in the butterfly's tree: chain w + 16 into
// chain w in registers, then warp w + d into warp w for d = 8, 4, 2, 1
// through shared memory (the fp32 x buffer just consumed), then the bias.
//
// Every wait is bounded: after a timeout the status block records it, no
// thread waits again, and the CTA runs to its end (its results are then
// garbage; the caller sees MOK_ERR_TIMEOUT).
//
// Dynamic shared memory:
//   bars [STAGES] u64 (128 B) | ws [STAGES][32][kRouteRow] f32 | xr [STAGES][TT][256] bf16 |
//   xf [2][TT][kRouteRow] f32 | lg [TT][E] f32 | slog [TT][k] f32 | cnt [E] i32
template <int TT, int STAGES>
__global__ void __launch_bounds__(kTopkThreads, 1)
route_topk_kernel(const __grid_constant__ CUtensorMap tmx, const float* __restrict__ Wr_copies, int wr_copies,
                  const float* __restrict__ bias, int T, int H, int E, int k, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w, int32_t* __restrict__ hist, StatusBlock* st, uint64_t tmo,
                  int withhold) {
    constexpr int TU = TT / 4;   // token slots per thread
    constexpr int NT = kTopkThreads;
    static_assert(TT % 4 == 0 && TT <= kRouteTTMax && TT >= kRouteTTMin && STAGES >= 3 && STAGES <= 16,
                  "router tile");
    static_assert(8 * 32 <= kRouteRow, "the chain sums of 8 warps fit one fp32 x buffer");
    extern __shared__ __align__(128) unsigned char route_smem[];
    const uint32_t bar0 = tc::smem_u32(route_smem);
    float* ws = reinterpret_cast<float*>(route_smem + 128);
    __nv_bfloat16* xr = reinterpret_cast<__nv_bfloat16*>(ws + STAGES * router_chunk_floats());
    float* xf = reinterpret_cast<float*>(xr + STAGES * TT * kRouteChunk);
    float* lg = xf + 2 * TT * kRouteRow;
    float* slog = lg + TT * E;
    int32_t* cnt = reinterpret_cast<int32_t*>(slog + TT * k);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // lane bits b4..b0: tl = b0 + 2*b2, el = b1 + 2*b3 + 4*b4
    const int tl = (lane & 1) | ((lane >> 1) & 2), el = ((lane >> 1) & 1) | ((lane >> 2) & 6);
    const int t0 = blockIdx.x * TT;
    const int ntok = min(TT, T - t0);
    const int nchunks = ceil_div(H, kRouteChunk);
    const int EG = ceil_div(E, 32);
    const int total = nchunks * EG;   // chunk sequence n = g * nchunks + c
    const float* __restrict__ Wr = Wr_copies + (int64_t)(blockIdx.x % wr_copies) * total * router_chunk_floats();

    for (int e = tid; e < E; e += NT) cnt[e] = 0;
    if (tid == 0) {
        tc::prefetch_tmap(&tmx);
        for (int s = 0; s < STAGES; ++s) tc::mbar_init(bar0 + 8u * s, 1);
        tc::fence_mbar_init();
    }
    pdl_wait();   // the re-laid router weights are written by the kernel before
    pdl_allow_next();
    __syncthreads();

    bool ok = true;
    int issued = 0, seen = 0;   // thread 0: chunks issued / chunks it has seen land
    // thread 0: the copies of chunk n into slot n % STAGES (nothing more
    // once one of its waits gave up)
    // withhold (test hook): CTA 0 never issues chunk 1, so its wait runs out
    const bool hold = withhold != 0 && blockIdx.x == 0;
    auto issue = [&](int n) {
        if (!ok || n >= total) return;
        issued = n + 1;
        if (hold && n == 1) return;
        const int g = n / nchunks, c = n % nchunks, slot = n % STAGES;
        const uint32_t bar = bar0 + 8u * slot;
        tc::mbar_expect_tx(bar, (uint32_t)(router_chunk_floats() * 4 + TT * kRouteChunk * 2));
        tc::bulk_load(tc::smem_u32(ws + slot * router_chunk_floats()),
                      Wr + ((int64_t)c * EG + g) * router_chunk_floats(), (uint32_t)(router_chunk_floats() * 4), bar);
        tc::tma_load_2d(tc::smem_u32(xr + slot * TT * kRouteChunk), &tmx, bar, c * kRouteChunk, t0);
    };
    auto wait = [&](int n) {
        if (ok && n < total) {
            ok = tc::mbar_wait(bar0 + 8u * (n % STAGES), (uint32_t)((n / STAGES) & 1), st, tmo, kSiteRouterChunk);
            if (ok) seen = n + 1;
        }
    };
    // raw x of slot b -> fp32 buffer d (h and h + 128 side by side, padded rows)
    auto convert_x = [&](int b, int d) {
        const __nv_bfloat16* xb = xr + b * TT * kRouteChunk;
        for (int v = tid; v < TT * 32; v += NT) {
            const int t = v >> 5, h0 = 4 * (v & 31);
            const uint2 lo = *reinterpret_cast<const uint2*>(xb + t * kRouteChunk + h0);
            const uint2 hi = *reinterpret_cast<const uint2*>(xb + t * kRouteChunk + h0 + 128);
            float* o = xf + (d * TT + t) * kRouteRow + 2 * h0;
            *reinterpret_cast<float4*>(o) = make_float4(bf16_lo(lo.x), bf16_lo(hi.x), bf16_hi(lo.x), bf16_hi(hi.x));
            *reinterpret_cast<float4*>(o + 4) = make_float4(bf16_lo(lo.y), bf16_lo(hi.y), bf16_hi(lo.y), bf16_hi(hi.y));
        }
    };

    if (tid == 0)
        for (int n = 0; n < STAGES - 1; ++n) issue(n);
    wait(0);
    convert_x(0, 0);
    float2 acc[TU][4];   // .x: chain warp, .y: chain warp + 16
    for (int n = 0; n < total; ++n) {
        wait(n + 1);       // its x is converted below
        __syncthreads();   // x(n) converted by every thread; chunk n - 1 consumed
        if (tid == 0) issue(n + STAGES - 1);   // into slot (n - 1) % STAGES
        if (n + 1 < total) convert_x((n + 1) % STAGES, (n + 1) & 1);
        const int g = n / nchunks, c = n % nchunks;
        if (c == 0) {
#pragma unroll
            for (int u = 0; u < TU; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = make_float2(0.f, 0.f);
        }
        const float* wb = ws + (n % STAGES) * router_chunk_floats() + el * kRouteRow;
        const float* xb = xf + ((n & 1) * TT + tl) * kRouteRow;
        // chain warp: h = hl .. hl + 7 of the chunk; chain warp + 16: the same
        // + 128. Past H both read zeros (a chain never holds -0, so adding
        // 0 * 0 leaves it unchanged); a step whose first chain starts past H
        // is skipped.
        const int hl = 8 * warp;
        if (c * kRouteChunk + hl < H) {
#pragma unroll(TT >= 28 ? 1 : 2)   // 28 tokens: no spills with one step in flight
            for (int s2 = 0; s2 < 8; s2 += 2) {
                // h = hl + s2 and hl + s2 + 1 of both chains
                float4 wv[4], xv[TU];
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    wv[v] = *reinterpret_cast<const float4*>(wb + 8 * v * kRouteRow + 2 * (hl + s2));
#pragma unroll
                for (int u = 0; u < TU; ++u)
                    xv[u] = *reinterpret_cast<const float4*>(xb + 4 * u * kRouteRow + 2 * (hl + s2));
                // every (token, expert, chain) accumulator takes its h in
                // ascending order; the TU x 4 float2 accumulators are independent
#pragma unroll
                for (int u = 0; u < TU; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        acc[u][v] = __ffma2_rn(make_float2(xv[u].x, xv[u].y), make_float2(wv[v].x, wv[v].y), acc[u][v]);
#pragma unroll
                for (int u = 0; u < TU; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        acc[u][v] = __ffma2_rn(make_float2(xv[u].z, xv[u].w), make_float2(wv[v].z, wv[v].w), acc[u][v]);
            }
        }
        if (c == nchunks - 1) {
            // the butterfly's tree over the 32 chains: chain L + 16 into chain
            // L (this thread's two chains), then chains L + 8, + 4, + 2, + 1
            // (warp w + d into warp w), then the bias. fp32 addition is
            // commutative, so which operand comes first does not matter.
            float p[TU][4];
#pragma unroll
            for (int u = 0; u < TU; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) p[u][v] = acc[u][v].x + acc[u][v].y;
            float* red = xf + (n & 1) * TT * kRouteRow;   // free until chunk n + 2 is converted into it
#pragma unroll
            for (int d = 8; d >= 1; d >>= 1) {
                __syncthreads();   // red's previous readers (chunk n's x, or the level before) are done
                if (warp >= d && warp < 2 * d) {
#pragma unroll
                    for (int u = 0; u < TU; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v) red[((warp - d) * TT + tl + 4 * u) * 32 + el + 8 * v] = p[u][v];
                }
                __syncthreads();
                if (warp < d) {
#pragma unroll
                    for (int u = 0; u < TU; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v) p[u][v] = p[u][v] + red[(warp * TT + tl + 4 * u) * 32 + el + 8 * v];
                }
            }
            if (warp == 0) {
#pragma unroll
                for (int u = 0; u < TU; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int e = 32 * g + el + 8 * v, tt = tl + 4 * u;
                        if (e < E && tt < ntok) lg[tt * E + e] = bias ? p[u][v] + bias[e] : p[u][v];
                    }
            }
        }
    }
    if (tid == 0 && seen < issued) {
        // a wait gave up: let the copies still in flight (at most one per
        // slot) land before the CTA exits, within the same time bound
        const uint64_t start = globaltimer_ns();
        for (int n = seen; n < issued; ++n)
            while (!(hold && n == 1) && !tc::mbar_try_wait(bar0 + 8u * (n % STAGES), (uint32_t)((n / STAGES) & 1)) &&
                   globaltimer_ns() - start < tmo) {
            }
    }
    // after a give-up the logits of this CTA's tokens are incomplete: rank
    // zeros instead, so the outputs stay valid routing (the lowest-index
    // experts, distinct, equal weights) for whatever reads them before the
    // caller sees the status
    if (__syncthreads_or(!ok)) {
        for (int i = tid; i < TT * E; i += NT) lg[i] = 0.f;
        __syncthreads();
    }

    // top-k per token: warp w takes tokens w, w + 8, ...
    const int nq = (E + 31) / 32;
    for (int t = warp; t < ntok; t += NT / 32) {
        float v[kMaxE / 32];
#pragma unroll
        for (int q = 0; q < kMaxE / 32; ++q) {
            int e = lane + 32 * q;
            v[q] = (q < nq && e < E) ? lg[t * E + e] : 0.f;
        }
        uint32_t taken = 0;
        float l0 = 0.f, den = 0.f;
        for (int j = 0; j < k; ++j) {
            float bv = 0.f;
            int be = -1;
#pragma unroll
            for (int q = 0; q < kMaxE / 32; ++q) {
                int e = lane + 32 * q;
                if (q < nq && e < E && !((taken >> q) & 1u) && (be < 0 || ranks_before(v[q], e, bv, be))) {
                    bv = v[q];
                    be = e;
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (oe >= 0 && (be < 0 || ranks_before(ov, oe, bv, be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (j == 0) l0 = bv;
            den += expf(bv - l0);   // j ascending; identical in every lane
            if (lane == 0) {
                slog[t * k + j] = bv;
                topk_idx[(int64_t)(t0 + t) * k + j] = be;
                atomicAdd(&cnt[be], 1);
            }
        }
        __syncwarp();
        for (int j = lane; j < k; j += 32) topk_w[(int64_t)(t0 + t) * k + j] = expf(slog[t * k + j] - l0) / den;
    }
    __syncthreads();
    for (int e = tid; e < E; e += NT) hist[(int64_t)blockIdx.x * E + e] = cnt[e];
}

size_t route_topk_smem_bytes(int TT, int STAGES, int E, int k) {
    return (size_t)128 + (size_t)STAGES * router_chunk_floats() * 4 + (size_t)STAGES * TT * kRouteChunk * 2 +
           (size_t)2 * TT * kRouteRow * 4 + (size_t)TT * E * 4 + (size_t)TT * k * 4 + (size_t)E * 4;
}

// Counts, offsets and the stable (expert, token) permutation. CTA b handles
// the same tt tokens as route_topk_kernel's CTA b: its rows for expert e
// start at offsets[e] + (rows of e in CTAs < b).
__global__ void __launch_bounds__(kRouteThreads)
route_layout_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ hist, int T, int E,
                    int k, int tt, int nblocks, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ row_src, int32_t* __restrict__ slot_row) {
    __shared__ int32_t pre[kMaxE], tot[kMaxE], off[kMaxE + 1];
    __shared__ int32_t part[kRouteThreads];
    __shared__ int32_t part2[kRouteThreads];
    __shared__ unsigned char sel[kRouteTTMax][kMaxE];
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const int t0 = b * tt;
    const int ntok = min(tt, T - t0);
    pdl_wait();
    pdl_allow_next();

    // per-expert sums over blocks (before b, and over all): `per` threads
    // share one expert, then combine their partial sums
    {
        int per = kRouteThreads / E > 0 ? kRouteThreads / E : 1;  // threads per expert
        for (int ebase = 0; ebase < E; ebase += kRouteThreads / per) {
            int e = ebase + tid / per, lane = tid % per;
            int s_pre = 0, s_tot = 0;
            if (tid / per < kRouteThreads / per && e < E) {
                for (int bb = lane; bb < nblocks; bb += per) {
                    int v = hist[(int64_t)bb * E + e];
                    s_tot += v;
                    if (bb < b) s_pre += v;
                }
            }
            part[tid] = s_pre;
            part2[tid] = s_tot;
            __syncthreads();
            if (lane == 0 && tid / per < kRouteThreads / per && e < E) {
                int a = 0, c = 0;
                for (int i = 0; i < per; ++i) { a += part[tid + i]; c += part2[tid + i]; }
                pre[e] = a;
                tot[e] = c;
            }
            __syncthreads();
        }
    }
    if (tid == 0) {
        int s = 0;
        for (int e = 0; e < E; ++e) { off[e] = s; s += tot[e]; }
        off[E] = s;
    }
    for (int i = tid; i < kRouteTTMax * E; i += kRouteThreads) sel[i / E][i % E] = 0;
    __syncthreads();
    if (b == 0) {
        for (int e = tid; e < E; e += kRouteThreads) counts[e] = tot[e];
        for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = off[e];
    }
    for (int i = tid; i < ntok * k; i += kRouteThreads) {
        int t = i / k;
        const int e = topk_idx[(int64_t)t0 * k + i];
        if ((unsigned)e < (unsigned)E) sel[t][e] = 1;
    }
    __syncthreads();
    for (int i = tid; i < ntok * k; i += kRouteThreads) {
        int t = i / k;
        int e = topk_idx[(int64_t)t0 * k + i];
        if ((unsigned)e >= (unsigned)E) continue;   // never produced by the top-k kernel
        int rank = 0;
        for (int tt = 0; tt < t; ++tt) rank += sel[tt][e];
        int row = off[e] + pre[e] + rank;
        int slot = t0 * k + i;
        row_src[row] = slot;
        slot_row[slot] = row;
    }
}

cudaError_t launch_transpose_wr(const float* W_r, float* WrT, int H, int E, int copies, cudaStream_t s) {
    transpose_wr_kernel<<<dim3(ceil_div(H, 32), ceil_div(E, 32), copies), dim3(32, 8), 0, s>>>(W_r, WrT, H, E);
    return cudaGetLastError();
}

// status | router weight copies | per-CTA expert histogram
size_t route_workspace_bytes(int T, int H, int E, int k) {
    (void)k;
    int nblocks = ceil_div(T, kRouteTTMin);
    return (size_t)kStatusBytes + align_up((int64_t)route_wr_copies(E, H) * router_copy_floats(E, H) * 4, 256) +
           align_up((int64_t)nblocks * E * 4, 256);
}

cudaError_t launch_router_weight_layout(const float* W_r, float* dst, int H, int E, int copies, cudaStream_t s) {
    router_weight_layout_kernel<<<dim3(8 * ceil_div(H, kRouteChunk), ceil_div(E, 32), copies), dim3(32, 8), 0, s>>>(
        W_r, dst, H, E);
    return cudaGetLastError();
}

// Launch the top-k kernel with TT tokens per CTA and a STAGES-deep ring.
template <int TT, int STAGES>
cudaError_t launch_topk_variant(const CUtensorMap& tmx, const float* Wr, int wr_copies, const float* bias, int T,
                                int H, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* hist,
                                StatusBlock* st, uint64_t timeout_ns, int withhold, cudaStream_t s) {
    const size_t smem = route_topk_smem_bytes(TT, STAGES, E, k);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    auto kern = route_topk_kernel<TT, STAGES>;
    if (smem > 48 * 1024) ensure_smem_attr(reinterpret_cast<const void*>(kern), (int)smem);
    cudaError_t e = launch_after(kern, dim3(ceil_div(T, TT)), dim3(kTopkThreads), smem, s, tmx, Wr, wr_copies, bias, T,
                                 H, E, k, topk_idx, topk_w, hist, st, timeout_ns, withhold);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Tokens per CTA: TT in {28, 20, 12, 8, 4}. One CTA per SM; a CTA's time is
// about (a fixed cost of streaming every weight chunk, worth about one token
// slot per thread) + TT/4, so the kernel takes about rounds x (TT/4 + 1),
// rounds = CTAs over SMs. Pick the cheapest that fits shared memory, larger
// tiles on ties.
constexpr int kRouteStages(int tt) { return tt >= 20 ? 3 : 4; }
int route_tokens_per_cta(int T, int num_sms, int E, int k) {
    const int tts[5] = {28, 20, 12, 8, 4};
    int best = 4;
    int64_t best_cost = -1;
    for (int tt : tts) {
        if (route_topk_smem_bytes(tt, kRouteStages(tt), E, k) > 227 * 1024) continue;
        const int64_t rounds = ceil_div(ceil_div(T, tt), num_sms > 0 ? num_sms : 1);
        const int64_t cost = rounds * (tt / 4 + 1);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = tt; }
    }
    return best;
}

cudaError_t launch_route_topk(const __nv_bfloat16* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                              int tt, int32_t* topk_idx, float* topk_w, int32_t* hist, StatusBlock* st,
                              uint64_t tmo, int hold, cudaStream_t s) {
    const int r = route_wr_copies(E, H);
    // x [T, H] BF16 in boxes of 256 h x tt tokens (H % 8 == 0: 16-byte row pitch)
    CUtensorMap tmx;
    if (!make_tmap_rows(&tmx, x, T, H, 2, kRouteChunk, tt)) return cudaErrorInvalidValue;
    switch (tt) {
    case 28: return launch_topk_variant<28, kRouteStages(28)>(tmx, Wr, r, bias, T, H, E, k, topk_idx, topk_w, hist, st,
                                                              tmo, hold, s);
    case 20: return launch_topk_variant<20, kRouteStages(20)>(tmx, Wr, r, bias, T, H, E, k, topk_idx, topk_w, hist, st,
                                                              tmo, hold, s);
    case 12: return launch_topk_variant<12, kRouteStages(12)>(tmx, Wr, r, bias, T, H, E, k, topk_idx, topk_w, hist, st,
                                                              tmo, hold, s);
    case 8: return launch_topk_variant<8, kRouteStages(8)>(tmx, Wr, r, bias, T, H, E, k, topk_idx, topk_w, hist, st,
                                                           tmo, hold, s);
    case 4: return launch_topk_variant<4, kRouteStages(4)>(tmx, Wr, r, bias, T, H, E, k, topk_idx, topk_w, hist, st,
                                                           tmo, hold, s);
    default: return cudaErrorInvalidValue;
    }
}

namespace {
RouteTestHook g_route_hook{};
}  // namespace

RouteTestHook route_test_hook() { return g_route_hook; }
void set_route_test_hook(int withhold, uint64_t timeout_ns) { g_route_hook = RouteTestHook{withhold, timeout_ns}; }

cudaError_t launch_route_layout(const void* x, const float* W_r, const float* bias, int T, int H, int E, int k,
                                int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                int32_t* row_src, int32_t* slot_row, void* ws, cudaStream_t s) {
    char* base = static_cast<char*>(ws) + kStatusBytes;
    float* Wr = reinterpret_cast<float*>(base);
    const int copies = route_wr_copies(E, H);
    int32_t* hist = reinterpret_cast<int32_t*>(base + align_up((int64_t)copies * router_copy_floats(E, H) * 4, 256));
    cudaError_t err = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (err != cudaSuccess) return err;
    if (T == 0) {
        cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tt = route_tokens_per_cta(T, sms, E, k);
    const int nblocks = ceil_div(T, tt);
    err = launch_router_weight_layout(W_r, Wr, H, E, copies, s);
    if (err != cudaSuccess) return err;
    const RouteTestHook hook = route_test_hook();
    err = launch_route_topk(static_cast<const __nv_bfloat16*>(x), Wr, bias, T, H, E, k, tt, topk_idx, topk_w, hist,
                            static_cast<StatusBlock*>(ws), hook.timeout_ns ? hook.timeout_ns : kRouteTimeoutNs,
                            hook.withhold, s);
    // the layout kernel must never run on top-k results that were not produced
    if (err != cudaSuccess) return err;
    err = launch_after(route_layout_kernel, dim3(nblocks), dim3(kRouteThreads), 0, s, topk_idx, hist, T, E, k, tt,
                       nblocks, counts, offsets, row_src, slot_row);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace mok
