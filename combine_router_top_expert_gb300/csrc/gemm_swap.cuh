// gemm_swap.cuh - grouped expert GEMM with the operands swapped: the expert's
// weight rows are the M side of 2-SM tcgen05 tiles, its tokens the N side.
//
// The grouped GEMM of the layer ("grouped GEMM" over each expert's contiguous
// token segment, KuCoin article on MoK, section 01) computes, per expert e,
// out[t, f] = sum_k act[t, k] * W_e[f, k]. Here each tile computes the
// transposed product D[f, t] = sum_k W_e[f, k] * act[t, k]: a CTA pair
// (tcgen05 cta_group::2) holds 256 weight rows (128 per CTA) as the A operand
// and N tokens (N/2 per CTA) as the B operand, with N any multiple of 32 up
// to 256 (the M=256 pair shape is used with N in steps of 32 only). An
// expert's tokens are cut into tiles of 256 and one remainder tile, so at most
// 31 rows of tensor work per expert are spent on padding (not a whole 128-row
// tile) and no CTA of a pair is idle; the accumulator holds one weight row per TMEM lane and one token
// per column.
//
// CTA layout (clusters of two CTAs, persistent over pair tiles):
//   warp 0     TMA producer (both CTAs): this CTA's 128 weight rows and its
//              N/2 token rows of each 64-element K block, signalling the
//              leader's full barrier; it also prefetches the weight box
//              l2_prefetch K blocks ahead into L2 (beyond the shared-memory
//              ring, into the next tile at a tile's end)
//   warp 1     allocates tensor memory; in the leader, one lane issues the
//              M=256 MMAs into a double-buffered fp32 accumulator
//   warps 2-5  epilogue (both CTAs): tcgen05.ld of this CTA's 128 lanes,
//              32 token columns at a time, staged through shared memory so
//              each token's row segment leaves in one 32-byte store
// Epilogues:
//   kSwapSwiGLU   gate/up GEMM. BF16 packed weights interleave gate and up
//                 rows per 16, so TMEM lanes 32q..32q+15 hold the gate and
//                 lanes 32q+16..32q+31 the up pre-activations of the same 16
//                 features: one shuffle pairs them; h = silu(G) * U (BF16)
//                 goes to h[row, feature].
//   kSwapScatter  down GEMM: y (BF16) of each token goes to its (token,
//                 slot) partial row, row_src[offset_e + local token].
// Every wait is bounded (StatusBlock); nothing traps.
#pragma once

#include "gemm.cuh"

namespace mok {

enum SwapEpi : int { kSwapSwiGLU = 0, kSwapScatter = 1 };

// Token tiles of an expert: 256 rows plus a remainder (default), or ceil(n/256)
// tiles of about equal size, each a multiple of 32. Measured: a pair tile's
// time follows the bytes its stages load (128 weight rows and up to 128 token
// rows per CTA and K block), not its N, so tiles narrower than 256 tokens
// cost nearly a full tile; the remainder cut loads fewer token rows.
enum SwapTilePolicy : int { kTiles256 = 0, kTilesBalanced = 1 };

struct SwapParams {
    int E;
    int num_kb;             // 64-element K blocks
    int m_tiles;            // 256-row weight tiles per expert
    int w_rows_per_expert;  // packed weight rows per expert
    const int32_t* counts;  // [E] routed rows per expert
    const int32_t* offsets; // scatter: unpadded offsets [E+1]
    const int32_t* row_src; // scatter: expert-ordered row -> slot
    void* out;              // SwiGLU: h [rows, ldo] bf16; scatter: partials [T*k, ldo] bf16
    int ldo;
    int tile_policy;
    int l2_prefetch;        // K blocks ahead of the load at which the weight box is prefetched into L2 (0: off)
    StatusBlock* status;
    unsigned long long timeout_ns;
};

struct SwapSched {
    int poff[kMaxE + 1];   // padded row offset of each expert segment (128-row padding of the layout)
    int toff[kMaxE + 1];   // first pair tile of each expert
    int nt[kMaxE];         // token-tile stride (multiple of 32)
    int nnt[kMaxE];        // token tiles
};

struct SwapTile {
    int e, m;
    int row0;    // first token row of the tile in the padded layout
    int tok0;    // first expert-local token of the tile
    int valid;   // tokens of the tile
    int N;       // MMA N: valid rounded up to 32
};

template <int STAGES>
struct SwapCfg {
    static constexpr int kThreads = 192;
    static constexpr int kBytesA = 128 * 128;       // 128 weight rows x 64 BF16
    static constexpr int kBytesB = 128 * 128;       // up to 128 token rows x 64 BF16
    static constexpr int kStageBytes = kBytesA + kBytesB;
    static constexpr int kBarOffset = STAGES * kStageBytes;
    static constexpr int kEpiOffset = kBarOffset + 256;
    static constexpr int kEpiBytes = 4 * 2048;      // per epilogue warp: 32 tokens x 64 bytes
    static constexpr int kSmemBytes = 1024 + kEpiOffset + kEpiBytes;
    static constexpr int kTmemCols = 512;           // two 256-column accumulators
    static_assert(kSmemBytes <= 227 * 1024 - (int)sizeof(SwapSched) - 64, "shared memory budget");
};

__device__ __forceinline__ void swap_build_sched(const SwapParams& p, SwapSched& s) {
    if (threadIdx.x == 0) {
        int rows = 0, tiles = 0;
        for (int e = 0; e < p.E; ++e) {
            const int cnt = p.counts[e];
            int nt = 256, nnt = 0;
            if (cnt > 0) {
                if (p.tile_policy == kTilesBalanced) {
                    const int parts = ceil_div(cnt, 256);
                    nt = min(256, ceil_div(ceil_div(cnt, parts), 32) * 32);
                }
                nnt = ceil_div(cnt, nt);
            }
            s.poff[e] = rows;
            s.toff[e] = tiles;
            s.nt[e] = nt;
            s.nnt[e] = nnt;
            rows += ceil_div(cnt, kTileM) * kTileM;
            tiles += nnt * p.m_tiles;
        }
        s.poff[p.E] = rows;
        s.toff[p.E] = tiles;
    }
}

// Pair tile g: expert e, weight tile m, token tile n (n fastest, so the pairs
// running at once share weight tiles in L2).
__device__ __forceinline__ SwapTile swap_decode(const SwapParams& p, const SwapSched& s, int g) {
    int lo = 0, hi = p.E - 1;   // last e with toff[e] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.toff[mid] <= g) lo = mid; else hi = mid - 1;
    }
    SwapTile t;
    t.e = lo;
    const int local = g - s.toff[lo];
    const int nnt = s.nnt[lo], nt = s.nt[lo];
    t.m = local / nnt;
    const int n = local % nnt;
    t.tok0 = n * nt;
    t.row0 = s.poff[lo] + t.tok0;
    t.valid = min(nt, p.counts[lo] - t.tok0);
    t.N = ceil_div(t.valid, 32) * 32;
    return t;
}

template <int EPI, int STAGES>
__global__ void __launch_bounds__(SwapCfg<STAGES>::kThreads, 1)
grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX64,
                         const __grid_constant__ CUtensorMap tmX32, const __grid_constant__ CUtensorMap tmX16,
                         const SwapParams p) {
    // tmW: packed weights [E * w_rows_per_expert, K], boxes of 64 x 128 rows;
    // tmX64/32/16: token rows [rows, K] in boxes of 64 x 64, 32 and 16 rows, so
    // a CTA loads exactly its N/2 token rows (a multiple of 16) in at most
    // four copies; all 128-byte swizzled
    using C = SwapCfg<STAGES>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ SwapSched sched;
    __shared__ uint32_t s_tmem_base;

    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = tc::smem_u32(smem);
    const uint32_t bar_base = smem_base + C::kBarOffset;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto accf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto acce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
    auto a_tile = [&](int s) { return smem_base + s * C::kStageBytes; };
    auto b_tile = [&](int s) { return smem_base + s * C::kStageBytes + C::kBytesA; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    StatusBlock* st = p.status;
    const uint64_t tmo = p.timeout_ns;

    swap_build_sched(p, sched);
    if (threadIdx.x == 32) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full_bar(s), 1);
            tc::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(accf_bar(a), 1);
            tc::mbar_init(acce_bar(a), 2 * 128);   // both CTAs' epilogue threads
        }
        tc::mbar_init(drain_bar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmW);
        tc::prefetch_tmap(&tmX64);
        tc::prefetch_tmap(&tmX32);
        tc::prefetch_tmap(&tmX16);
    }
    if (warp == 1) {
        tc::tmem_alloc_2sm(tc::smem_u32(&s_tmem_base), C::kTmemCols);
        tc::tmem_relinquish_2sm();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    tc::cluster_sync();   // the peer's barriers and tensor memory exist
    const uint32_t tmem = s_tmem_base;
    const int rank = (int)tc::cluster_ctarank();
    const int gstart = (int)blockIdx.x / 2;
    const int gstep = (int)gridDim.x / 2;
    const int gtotal = sched.toff[p.E];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int last_par[STAGES];
            for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
            bool ok = true;
            const int pf = p.l2_prefetch;
            for (int gi = gstart; gi < gtotal && ok; gi += gstep) {
                const SwapTile t = swap_decode(p, sched, gi);
                const int half = t.N / 2;                 // token rows of this CTA (multiple of 16)
                const int wrow = t.e * p.w_rows_per_expert + t.m * 256 + rank * 128;
                const int xrow = t.row0 + rank * half;
                // weight rows of this CTA's next tile, for the prefetches that run past this one
                int wnext = -1;
                if (pf > 0 && gi + gstep < gtotal) {
                    const SwapTile tn = swap_decode(p, sched, gi + gstep);
                    wnext = tn.e * p.w_rows_per_expert + tn.m * 256 + rank * 128;
                }
                if (pf > 0 && gi == gstart)
                    for (int kb = 0; kb < pf && kb < p.num_kb; ++kb) tc::tma_prefetch_2d(&tmW, kb * 64, wrow);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (pf > 0) {
                        // the weight box pf K blocks ahead: this tile's, or the next tile's first ones
                        if (kb + pf < p.num_kb) tc::tma_prefetch_2d(&tmW, (kb + pf) * 64, wrow);
                        else if (wnext >= 0 && wnext != wrow && kb + pf - p.num_kb < p.num_kb)
                            tc::tma_prefetch_2d(&tmW, (kb + pf - p.num_kb) * 64, wnext);
                    }
                    if (!tc::mbar_wait(empty_bar(stage), ph ^ 1u, st, tmo, kSiteProducerEmpty)) { ok = false; break; }
                    const uint32_t lead_full = tc::mapa_shared(full_bar(stage), 0);
                    if (rank == 0) tc::mbar_expect_tx(full_bar(stage), 2u * (C::kBytesA + (uint32_t)half * 128u));
                    tc::tma_load_2d_2sm(a_tile(stage), &tmW, lead_full, kb * 64, wrow);
                    // this CTA's half token rows as 64-, 32- and 16-row boxes
                    int r0 = 0;
                    for (; r0 + 64 <= half; r0 += 64)
                        tc::tma_load_2d_2sm(b_tile(stage) + r0 * 128, &tmX64, lead_full, kb * 64, xrow + r0);
                    if (r0 + 32 <= half) {
                        tc::tma_load_2d_2sm(b_tile(stage) + r0 * 128, &tmX32, lead_full, kb * 64, xrow + r0);
                        r0 += 32;
                    }
                    if (r0 < half) tc::tma_load_2d_2sm(b_tile(stage) + r0 * 128, &tmX16, lead_full, kb * 64, xrow + r0);
                    last_par[stage] = (int)ph;
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // the copies already issued land before the CTA exits; the
                // leader's barrier collects them
                for (int s = 0; s < STAGES; ++s)
                    if (last_par[s] >= 0 && rank == 0) tc::mbar_wait(full_bar(s), (uint32_t)last_par[s], st, tmo, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            bool ok = true, issued = false;
            for (int gi = gstart; gi < gtotal && ok; gi += gstep) {
                const SwapTile t = swap_decode(p, sched, gi);
                if (!tc::mbar_wait(acce_bar(acc), acc_ph ^ 1u, st, tmo, kSiteMmaAccEmpty)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(acc * 256);
                const uint32_t idesc = tc::idesc_bf16(256, t.N, false, false);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!tc::mbar_wait(full_bar(stage), ph, st, tmo, kSiteMmaFull)) { ok = false; break; }
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::make_sdesc(a_tile(stage) + kk * 32, 16, 1024, tc::kLayoutSW128);
                        const uint64_t bd = tc::make_sdesc(b_tile(stage) + kk * 32, 16, 1024, tc::kLayoutSW128);
                        tc::mma_bf16_2sm(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    issued = true;
                    tc::mma_commit_2sm_multicast(empty_bar(stage), (uint16_t)0x3);
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc::mma_commit_2sm_multicast(accf_bar(acc), (uint16_t)0x3);
                if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
            }
            if (!ok && issued) {
                // every MMA issued so far must finish before tensor memory is freed
                tc::mma_commit_2sm(drain_bar);
                tc::mbar_wait(drain_bar, 0, st, tmo, kSiteDrain);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;   // TMEM lane quadrant of this warp
        const uint32_t stg = smem_base + C::kEpiOffset + (uint32_t)(warp - 2) * 2048u;
        unsigned char* stg_p = smem + C::kEpiOffset + (warp - 2) * 2048;
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int gi = gstart; gi < gtotal; gi += gstep) {
            const SwapTile t = swap_decode(p, sched, gi);
            if (!tc::mbar_wait(accf_bar(acc), acc_ph, st, tmo, kSiteEpiAccFull)) break;
            tc::fence_after_sync();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
#pragma unroll 1
            for (int c0 = 0; c0 < t.N; c0 += 32) {
                uint32_t v[32];
                tc::tmem_ld_32x32b_x32(tbase + c0, v);
                tc::tmem_ld_wait();
                if constexpr (EPI == kSwapSwiGLU) {
                    // lanes 0-15: gate of features f0 + lane, lanes 16-31: up
                    // of the same features; the lower half forms h for tokens
                    // c0 .. c0+15, the upper half for c0+16 .. c0+31
                    const bool lower = lane < 16;
                    __nv_bfloat16* sp = reinterpret_cast<__nv_bfloat16*>(stg_p);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t send = lower ? v[16 + i] : v[i];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const float g = __uint_as_float(lower ? v[i] : recv);
                        const float u = __uint_as_float(lower ? recv : v[16 + i]);
                        const int tok = lower ? i : 16 + i;
                        sp[tok * 16 + (lane & 15)] = __float2bfloat16_rn(silu_f(g) * u);
                    }
                    __syncwarp();
                    // lane j: token c0 + j, 16 features = 32 bytes
                    const int tok = c0 + lane;
                    if (tok < t.valid) {
                        uint32_t w[8];
                        const uint4 a = *reinterpret_cast<const uint4*>(stg_p + lane * 32);
                        const uint4 b = *reinterpret_cast<const uint4*>(stg_p + lane * 32 + 16);
                        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
                        const int f0 = t.m * 128 + rank * 64 + q * 16;
                        tc::stg_v8(static_cast<__nv_bfloat16*>(p.out) + (int64_t)(t.row0 + tok) * p.ldo + f0, w);
                    }
                    __syncwarp();
                } else {
                    // lane = feature f0 + lane; the 32 token columns to rows
                    // of 32 features (64 bytes) in shared memory
                    __nv_bfloat16* sp = reinterpret_cast<__nv_bfloat16*>(stg_p);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sp[i * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[i]));
                    __syncwarp();
                    const int f0 = t.m * 256 + rank * 128 + q * 32;
#pragma unroll
                    for (int rd = 0; rd < 2; ++rd) {
                        const int tt = (lane >> 1) + 16 * rd, hf = lane & 1;
                        const int tok = c0 + tt;
                        if (tok < t.valid) {
                            const int64_t dest = p.row_src[p.offsets[t.e] + t.tok0 + tok];
                            uint32_t w[8];
                            const unsigned char* src = stg_p + tt * 64 + hf * 32;
                            const uint4 a = *reinterpret_cast<const uint4*>(src);
                            const uint4 b = *reinterpret_cast<const uint4*>(src + 16);
                            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
                            tc::stg_v8(static_cast<__nv_bfloat16*>(p.out) + dest * p.ldo + f0 + hf * 16, w);
                        }
                    }
                    __syncwarp();
                }
            }
            (void)stg;
            tc::fence_before_sync();
            tc::mbar_arrive_cluster(tc::mapa_shared(acce_bar(acc), 0));
            if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    tc::cluster_sync();   // no CTA frees or leaves while its peer may still use the pair's resources
    if (warp == 1) tc::tmem_dealloc_2sm(tmem, C::kTmemCols);
}

}  // namespace mok
