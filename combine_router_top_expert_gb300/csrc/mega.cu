// mega.cu - the persistent forward megakernel and its device-side plan.
//
// Pages (KuCoin article on Cursor's MoK, section 02): one kernel whose SMs are
// split in two - one part moves tokens in and results out and keeps the
// state, the other runs the expert FFN - talking through GPU-local counters
// (the movers tell the compute side when a complete set of tokens has
// arrived; the compute side tells the movers when results can go back), with
// tokens handed over in minibatches of at least two full waves, staged in a
// fixed-size ring token buffer that is reused as soon as its tokens were
// consumed, and no CPU decision inside the loop.
//
// On one GB300 this is:
//   mover CTAs    pull-gather (and MXFP8-quantise) each minibatch's rows into
//                 one of two ring regions, expert by expert; after every
//                 8-row chunk they publish the rows with a release-increment
//                 of ready[mb][e]; a region is refilled only once every
//                 gate/up tile that read it has finished (g1_mb[mb-2]).
//   compute CTAs  tcgen05 tiles in the plan's phase order G1(0), G1(1),
//                 G2(0), G1(2), G2(1), ...: the TMA producer acquires the
//                 tile's dependency counter (ready rows for a gate/up tile,
//                 finished gate/up tiles of the expert for a down tile)
//                 before its first load; the epilogue publishes each tile
//                 with release increments (g1_e, g1_mb, g2_mb).
//   everyone      once a minibatch's down tiles are all done, CTAs that have
//                 nothing else to do take 4-token chunks of its fixed-order
//                 weighted sum (an atomic chunk counter hands them out; each
//                 token's sum is computed by one thread in j order, so the
//                 result does not depend on who computes it).
// The launch is cooperative (all CTAs co-resident, one per SM), every wait
// depends only on work earlier in a fixed order, so the kernel always makes
// progress; every wait is still bounded and gives up cleanly, and every
// decision that precedes a barrier is made once and shared, so no barrier
// can wait for a thread that left.
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemm.cuh"
#include "moves.cuh"
#include "plan.cuh"

namespace mok {

// ---------------------------------------------------------------------------
// Plan kernels
// ---------------------------------------------------------------------------
struct PlanBatch {
    const int32_t* offsets;  // [E+1]
    const int32_t* row_src;  // [T*k]
};
struct PlanBatches {
    PlanBatch b[kMaxBatches];
};

constexpr int kPlanTB = 16;          // tokens per plan block
constexpr int kMaxMbPerBatch = 512;

__host__ __device__ inline int64_t plan_stage_ints(int E) { return 2 + (int64_t)kMaxMbPerBatch * (2 + 2 * E); }

// Per-batch plan: one CTA per macro-batch. Output in a per-batch staging
// area: [0] minibatches, [1] error, then per minibatch: t0, t1 (the tokens
// whose weighted sums it releases), E segment starts, E segment ends
// (indices into the batch's row_src).
//
// Tile cuts (default): the batch's expert-contiguous layout, padded per
// expert to 128-row tiles as for the staged GEMMs, is cut into runs of
// consecutive tiles, each run at most a ring region (and at most
// max_tokens * k rows when max_tokens < T). Only each expert's last tile
// over the whole batch is partial; every token's rows are final once the
// batch's last minibatch is, so that minibatch releases all T tokens.
//
// Token cuts (MOK_FLAG_MB_TOKEN_RANGES): rows of expert e before token t are
// the lower bound of t in the expert's row_src segment (sorted by token);
// one warp cuts minibatches greedily, block (16 tokens) by block, while the
// block range's per-expert padded rows fit a region. Each minibatch releases
// its own tokens, but pads every expert's rows separately.
__global__ void __launch_bounds__(256)
plan_batch_kernel(const PlanBatches batches, int T, int E, int k, int region_rows, int max_tokens,
                  int tile_cuts, int* __restrict__ stage) {
    extern __shared__ int ps[];
    const int b = blockIdx.x;
    const int nblk = ceil_div(T, kPlanTB);
    int* P = ps;  // [(nblk + 1) * E]
    const PlanBatch pb = batches.b[b];
    if (tile_cuts) {
        if (threadIdx.x >= 32) return;
        int* out = stage + (int64_t)b * plan_stage_ints(E);
        const int lane = threadIdx.x;
        int run = 0;   // P[e] = tiles of the experts before e
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int mt = e < E ? ceil_div(pb.offsets[e + 1] - pb.offsets[e], kTileM) : 0;
            int incl = mt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            if (e < E) P[e] = run + incl - mt;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        const int total = run;
        int R = region_rows / kTileM;
        if (max_tokens < T) R = min(R, max(1, ceil_div(max_tokens * k, kTileM)));
        const int nmb = (total == 0 || R < 1) ? 0 : ceil_div(total, R);
        if (R < 1 || nmb > kMaxMbPerBatch) {
            if (lane == 0) { out[0] = 0; out[1] = 1; }
            return;
        }
        for (int j = 0; j < nmb; ++j) {
            int* m = out + 2 + j * (2 + 2 * E);
            const int g0 = j * R, g1 = min(total, g0 + R);
            if (lane == 0) { m[0] = j == nmb - 1 ? 0 : T; m[1] = T; }
            for (int e = lane; e < E; e += 32) {
                const int o0 = pb.offsets[e], c = pb.offsets[e + 1] - o0;
                const int te = P[e], mt = ceil_div(c, kTileM);
                const int lo = max(g0, te), hi = min(g1, te + mt);
                int s0 = o0, s1 = o0;
                if (lo < hi) {
                    s0 = o0 + (lo - te) * kTileM;
                    s1 = o0 + min((hi - te) * kTileM, c);
                }
                m[2 + e] = s0;
                m[2 + E + e] = s1;
            }
        }
        if (lane == 0) { out[0] = nmb; out[1] = 0; }
        return;
    }
    for (int i = threadIdx.x; i < (nblk + 1) * E; i += blockDim.x) {
        const int blk = i / E, e = i % E;
        const int tb = min(blk * kPlanTB, T);
        int lo = pb.offsets[e], hi = pb.offsets[e + 1];
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (pb.row_src[mid] / k < tb) lo = mid + 1; else hi = mid;
        }
        P[i] = lo;
    }
    __syncthreads();
    int* out = stage + (int64_t)b * plan_stage_ints(E);
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    int b0 = 0, nmb = 0, err = 0;
    while (b0 < nblk && !err) {
        // extend the minibatch block by block while its padded rows fit
        int best = b0;
        for (int b1 = b0 + 1; b1 <= nblk; ++b1) {
            if ((b1 - b0) * kPlanTB > max_tokens && b1 > b0 + 1) break;
            int padded = 0;
            for (int e = lane; e < E; e += 32) {
                const int c = P[b1 * E + e] - P[b0 * E + e];
                padded += ceil_div(c, kTileM) * kTileM;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) padded += __shfl_xor_sync(0xffffffffu, padded, off);
            if (padded > region_rows) break;
            best = b1;
        }
        if (best == b0 || nmb >= kMaxMbPerBatch) { err = 1; break; }
        int* m = out + 2 + nmb * (2 + 2 * E);
        if (lane == 0) { m[0] = b0 * kPlanTB; m[1] = min(best * kPlanTB, T); }
        for (int e = lane; e < E; e += 32) {
            m[2 + e] = P[b0 * E + e];
            m[2 + E + e] = P[best * E + e];
        }
        ++nmb;
        b0 = best;
    }
    if (lane == 0) { out[0] = nmb; out[1] = err; }
}

// Flatten the per-batch plans into the global minibatch list and phases.
__global__ void __launch_bounds__(256)
plan_finalize_kernel(int nbatch, int E, int NT1, int NT2, const int* __restrict__ stage, PlanView v) {
    __shared__ int s_base[kMaxBatches + 1];
    __shared__ int s_err;
    if (threadIdx.x == 0) {
        int s = 0, err = 0;
        for (int b = 0; b < nbatch; ++b) {
            const int* o = stage + (int64_t)b * plan_stage_ints(E);
            s_base[b] = s;
            s += o[0];
            err |= o[1];
        }
        s_base[nbatch] = s;
        if (s > kMaxMinibatches) err = 1;
        s_err = err;
    }
    __syncthreads();
    const int n_mb = s_base[nbatch];
    if (s_err) {
        if (threadIdx.x == 0) {
            v.hdr->error = 1;
            v.hdr->n_mb = 0;
            v.hdr->n_phase = 0;
            v.hdr->total_tiles = 0;
        }
        return;
    }
    // per-(mb, e) arrays, one warp per minibatch
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int g = warp; g < n_mb; g += blockDim.x / 32) {
        int b = 0;
        while (s_base[b + 1] <= g) ++b;
        const int lmb = g - s_base[b];
        const int* m = stage + (int64_t)b * plan_stage_ints(E) + 2 + lmb * (2 + 2 * E);
        int run_mt = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            int c = 0, s0 = 0;
            if (e < E) { s0 = m[2 + e]; c = m[2 + E + e] - s0; }
            const int mt = ceil_div(c, kTileM);
            int incl = mt;  // inclusive scan over the lanes
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const int excl = incl - mt;
            if (e < E) {
                v.cnt[g * E + e] = c;
                v.src0[g * E + e] = s0;
                v.roff[g * E + e] = (run_mt + excl) * kTileM;
                v.mtoff[g * (E + 1) + e] = run_mt + excl;
            }
            run_mt += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            v.mtoff[g * (E + 1) + E] = run_mt;
            MbInfo mi;
            mi.batch = b;
            mi.t0 = m[0];
            mi.t1 = m[1];
            mi.rows = run_mt * kTileM;
            mi.mtiles = run_mt;
            mi.region = g & 1;
            mi.pad[0] = mi.pad[1] = 0;
            v.mb[g] = mi;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phases: G1(0), then G1(i+1), G2(i) for each i, the last G2 alone
        int np = 0, tiles = 0;
        auto add = [&](int kind, int mb) {
            v.phase_kind[np] = kind;
            v.phase_mb[np] = mb;
            v.phase_toff[np] = tiles;
            tiles += v.mb[mb].mtiles * (kind == 0 ? NT1 : NT2);
            ++np;
        };
        if (n_mb > 0) add(0, 0);
        for (int i = 0; i < n_mb; ++i) {
            if (i + 1 < n_mb) add(0, i + 1);
            add(1, i);
        }
        v.phase_toff[np] = tiles;
        v.hdr->n_mb = n_mb;
        v.hdr->n_phase = np;
        v.hdr->total_tiles = tiles;
        v.hdr->error = 0;
    }
}

// ---------------------------------------------------------------------------
// The megakernel
// ---------------------------------------------------------------------------
struct MegaBatch {
    const __nv_bfloat16* x;   // [T, H]
    const uint8_t* xq;        // MXFP8: x quantised per token row [T, H] E4M3 (the movers copy these)
    const uint32_t* xsf;      // MXFP8: its scale words [T, H/128]
    const int32_t* row_src;   // [T*k]
    const float* topk_w;      // [T, k]
    __nv_bfloat16* partials;  // [T*k, H]
    const float* shared;      // [T, H] f32 or null
    __nv_bfloat16* out;       // [T, H]
};

struct MegaParams {
    int E, H, I, k, T, nbatch;
    MegaBatch batches[kMaxBatches];
    PlanView plan;
    void* ring;
    uint8_t* ring_sf;
    int region_rows;
    void* hbuf;
    uint8_t* h_sf;
    const uint8_t* gu_sf;
    const uint8_t* dn_sf;
    int* ready;      // [kMaxMinibatches * E] padded rows published per (mb, e)
    int* g1_e;       // [kMaxMinibatches * E] finished gate/up tiles per (mb, e)
    int* g1_mb;      // [kMaxMinibatches]
    int* g2_mb;      // [kMaxMinibatches]
    int* comb_next;  // [kMaxMinibatches]
    int bn2;         // N-tile of the down GEMM (224, 256 or 128)
    int n_movers;
    int test_flags;
    unsigned long long* trace;   // per-CTA records, or NULL
    StatusBlock* status;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// AND of `pred` over the `nthreads` threads arriving at named barrier `id`
// (every participant gets the same answer, so loops break in lockstep).
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Bounded wait until *p >= target (acquire). False: gave up (recorded).
__device__ bool wait_counter(const int* p, int target, StatusBlock* st, uint64_t tmo, int32_t site) {
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire(p) >= target) return true;
        __nanosleep(64);
        if ((it & 31) == 0) {
            if (abort_requested(st)) return false;
            if (globaltimer_ns() - t0 > tmo) {
                record_failure(st, MOK_ERR_TIMEOUT, site);
                return false;
            }
        }
    }
}

struct MegaTile {
    int kind, mb, e, m, n;
    int a_row0;      // first row in the ring (gate/up) or h buffer (down)
    int mt;          // 128-row tiles of (mb, e)
    int local_row0;  // first expert-local row of the tile
};

__device__ __forceinline__ MegaTile mega_decode(const MegaParams& p, int g, int NT1, int NT2) {
    const PlanView& v = p.plan;
    int lo = 0, hi = v.hdr->n_phase - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (v.phase_toff[mid] <= g) lo = mid; else hi = mid - 1;
    }
    MegaTile t;
    t.kind = v.phase_kind[lo];
    t.mb = v.phase_mb[lo];
    const int NT = t.kind == 0 ? NT1 : NT2;
    const int local = g - v.phase_toff[lo];
    const int* mto = v.mtoff + t.mb * (p.E + 1);
    int a = 0, b = p.E - 1;  // last e with mto[e] * NT <= local (skips empty experts)
    while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (mto[mid] * NT <= local) a = mid; else b = mid - 1;
    }
    t.e = a;
    t.mt = mto[a + 1] - mto[a];
    const int l2 = local - mto[a] * NT;
    t.n = l2 / t.mt;
    t.m = l2 % t.mt;
    const int region = v.mb[t.mb].region;
    t.a_row0 = region * p.region_rows + v.roff[t.mb * p.E + t.e] + t.m * kTileM;
    t.local_row0 = t.m * kTileM;
    return t;
}

constexpr int kMoverLoads = 28;    // BF16 mover: 16-byte loads in flight per lane per pass
constexpr int kMoverBlocks = 7;    // MXFP8 mover: 32-element blocks per lane per pass

// One minibatch's pull-gather by the mover CTAs: warps take 8-row chunks of
// the padded minibatch rows; inside a warp, lanes 4r..4r+3 copy row r of the
// chunk (lane part q of a row takes its 16-byte words, or 32-element blocks,
// q, q+4, q+8, ...), so the 8 rows' source lookups and loads are all in
// flight together. A chunk is published (release) once all its rows landed.
template <bool MX>
__device__ void mover_dispatch_mb(const MegaParams& p, int mb, int gwarp, int nwarps, int lane) {
    const PlanView& v = p.plan;
    const MbInfo mi = v.mb[mb];
    const MegaBatch bt = p.batches[mi.batch];
    const int* roff = v.roff + mb * p.E;
    const int* cnt = v.cnt + mb * p.E;
    const int* src0 = v.src0 + mb * p.E;
    const int H = p.H;
    const int nchunks = mi.rows / 8;
    const int rr = lane >> 2, part = lane & 3;
    for (int c = gwarp; c < nchunks; c += nwarps) {
        const int r0 = c * 8;
        int lo = 0, hi = p.E - 1;  // expert owning padded row r0 (skips empty experts)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (roff[mid] <= r0) lo = mid; else hi = mid - 1;
        }
        const int e = lo;   // a chunk never straddles experts: segments are 128-row multiples
        const int row = r0 + rr;
        const int local = row - roff[e];
        const __nv_bfloat16* src = nullptr;
        if (local < cnt[e]) src = bt.x + (int64_t)(bt.row_src[src0[e] + local] / p.k) * H;
        const int64_t grow = (int64_t)mi.region * p.region_rows + row;
        if constexpr (!MX) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.ring) + grow * H);
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            const int n16 = H / 8;
            for (int q0 = part; q0 < n16; q0 += 4 * kMoverLoads) {
                uint4 vv[kMoverLoads];
#pragma unroll
                for (int u = 0; u < kMoverLoads; ++u) {
                    const int q = q0 + 4 * u;
                    vv[u] = (src && q < n16) ? __ldg(s4 + q) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kMoverLoads; ++u) {
                    const int q = q0 + 4 * u;
                    if (q < n16) __stcg(dst + q, vv[u]);
                }
            }
        } else {
            uint8_t* dst = static_cast<uint8_t*>(p.ring) + grow * H;
            const int rt = (int)(grow / kTileM), r = (int)(grow % kTileM);
            const int nb = H / 32;   // a multiple of 4: the 4 lanes of a row share each 128-wide chunk
            for (int b0 = 0; b0 < nb; b0 += 4 * kMoverBlocks) {
                uint4 vv[kMoverBlocks][4];
#pragma unroll
                for (int u = 0; u < kMoverBlocks; ++u) {
                    const int bb = b0 + 4 * u + part;
                    const uint4* s4 = reinterpret_cast<const uint4*>(src + bb * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        vv[u][i] = (src && bb < nb) ? __ldg(s4 + i) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kMoverBlocks; ++u) {
                    const int bb = b0 + 4 * u + part;
                    float f[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        f[8 * i + 0] = bf16_lo(vv[u][i].x); f[8 * i + 1] = bf16_hi(vv[u][i].x);
                        f[8 * i + 2] = bf16_lo(vv[u][i].y); f[8 * i + 3] = bf16_hi(vv[u][i].y);
                        f[8 * i + 4] = bf16_lo(vv[u][i].z); f[8 * i + 5] = bf16_hi(vv[u][i].z);
                        f[8 * i + 6] = bf16_lo(vv[u][i].w); f[8 * i + 7] = bf16_hi(vv[u][i].w);
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
                    const uint32_t code = src ? e8m0_code(amax) : 0u;
                    const float inv = e8m0_inv_scale(code);
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = f32x2_to_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv) |
                               (f32x2_to_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
                    // the row's 4 lanes hold blocks 4c..4c+3 of chunk c: one word of codes
                    uint32_t word = code;
                    word |= __shfl_down_sync(0xffffffffu, code, 1) << 8;
                    word |= __shfl_down_sync(0xffffffffu, code, 2) << 16;
                    word |= __shfl_down_sync(0xffffffffu, code, 3) << 24;
                    if (bb < nb) {
                        __stcg(reinterpret_cast<uint4*>(dst + bb * 32), make_uint4(w[0], w[1], w[2], w[3]));
                        __stcg(reinterpret_cast<uint4*>(dst + bb * 32) + 1, make_uint4(w[4], w[5], w[6], w[7]));
                        if (part == 0)
                            *reinterpret_cast<uint32_t*>(p.ring_sf + ((int64_t)rt * (H / 128) + bb / 4) * 512 +
                                                         sf_chunk_offset(r, 0)) = word;
                    }
                }
            }
        }
        // publish the 8 rows: visible at gpu scope and to the readers' TMA
        __threadfence();
        tc::fence_proxy_async_global();
        __syncwarp();
        const bool withhold = (p.test_flags & MOK_FLAG_TEST_WITHHOLD_PUBLISH) && mb == 0 && c == nchunks - 1;
        if (lane == 0 && !withhold) red_release_add(&p.ready[mb * p.E + e], 8);
    }
}

// Pull-gather through the copy engines: lane 0 of each mover warp pumps the
// rows of its 8-row chunks global -> shared -> ring with bulk copies, two row
// buffers per warp (the load of row r+1 overlaps the store of row r); pad
// rows are not written (the GEMM rows they feed are never stored, and a
// region's old rows are finite or never read back); MXFP8 copies the E4M3
// rows of x quantised once
// per token (quantize_rows, before the launch) and the warp's lanes place
// their scale words in the ring's tile-ordered scale chunks. The chunk is
// published once its stores have completed. A warp keeps two rows in flight
// with one issuing thread, where register copies need every lane for a
// fraction of that. Returns false if a bounded wait gave up.
struct MoverSmem {
    uint32_t bufs;    // [warps][2] row buffers
    uint32_t bars;    // [warps][2] mbarriers (8 bytes each)
};

template <bool MX>
__device__ bool mover_pump_mb(const MegaParams& p, int mb, int gwarp, int nwarps, int lane, int warp,
                              const MoverSmem& ms, uint32_t& phases) {
    const PlanView& v = p.plan;
    const MbInfo mi = v.mb[mb];
    const MegaBatch bt = p.batches[mi.batch];
    const int* roff = v.roff + mb * p.E;
    const int* cnt = v.cnt + mb * p.E;
    const int* src0 = v.src0 + mb * p.E;
    const uint32_t rowb = (uint32_t)p.H * (MX ? 1 : 2);
    const int nchunks = mi.rows / 8;
    const int kc_row = p.H / 128;   // MXFP8 scale words per row
    bool ok = true;
    for (int c = gwarp; c < nchunks; c += nwarps) {
        const int r0 = c * 8;
        int lo = 0, hi = p.E - 1;  // expert owning padded row r0 (skips empty experts)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (roff[mid] <= r0) lo = mid; else hi = mid - 1;
        }
        const int e = lo;
        int my_tok = -1;   // lane r < 8: source token of row r (-1: pad row)
        if (lane < 8) {
            const int local = r0 + lane - roff[e];
            if (local < cnt[e]) my_tok = bt.row_src[src0[e] + local] / p.k;
        }
        const int64_t grow0 = (int64_t)mi.region * p.region_rows + r0;
        if constexpr (MX) {
            // scale words: row r's word kc goes to byte (r%32)*16 + (r/32)*4 of chunk (tile, kc)
            for (int r = 0; r < 8; ++r) {
                const int tok = __shfl_sync(0xffffffffu, my_tok, r);
                const int64_t grow = grow0 + r;
                if (tok < 0) continue;   // pad rows feed only GEMM rows that are never stored
                for (int kc = lane; kc < kc_row; kc += 32) {
                    const uint32_t wd = __ldg(bt.xsf + (int64_t)tok * kc_row + kc);
                    *reinterpret_cast<uint32_t*>(p.ring_sf + ((grow / kTileM) * kc_row + kc) * 512 +
                                                 sf_chunk_offset((int)(grow % kTileM), 0)) = wd;
                }
            }
        }
        int toks[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) toks[r] = __shfl_sync(0xffffffffu, my_tok, r);
        if (lane == 0 && ok) {
            const char* src[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                src[r] = toks[r] < 0 ? nullptr
                         : MX ? reinterpret_cast<const char*>(bt.xq + (int64_t)toks[r] * p.H)
                              : reinterpret_cast<const char*>(bt.x + (int64_t)toks[r] * p.H);
            const uint32_t buf[2] = {ms.bufs + (uint32_t)(2 * warp) * rowb, ms.bufs + (uint32_t)(2 * warp + 1) * rowb};
            const uint32_t bar[2] = {ms.bars + 16u * warp, ms.bars + 16u * warp + 8u};
            char* ring = static_cast<char*>(p.ring) + grow0 * rowb;
            tc::bulk_wait_read<0>();   // the previous chunk's stores no longer read the buffers
            if (src[0]) {
                tc::mbar_expect_tx(bar[0], rowb);
                tc::bulk_load(buf[0], src[0], rowb, bar[0]);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int sl = r & 1;
                if (r + 1 < 8 && src[r + 1]) {
                    tc::bulk_wait_read<0>();   // the store of row r - 1 is done with buffer (r + 1) & 1
                    tc::mbar_expect_tx(bar[sl ^ 1], rowb);
                    tc::bulk_load(buf[sl ^ 1], src[r + 1], rowb, bar[sl ^ 1]);
                }
                if (src[r]) {
                    if (!tc::mbar_wait(bar[sl], (phases >> sl) & 1u, p.status, p.timeout_ns, kSiteCounter)) {
                        ok = false;
                        break;
                    }
                    phases ^= 1u << sl;
                    tc::bulk_store(ring + (int64_t)r * rowb, buf[sl], rowb);
                    tc::bulk_commit();
                }   // pad rows stay unwritten: their GEMM rows are never stored
            }
            tc::bulk_wait<0>();   // the chunk's rows are written
        }
        // every lane's writes (MXFP8 scale words; lane 0's bulk copies) are
        // ordered before lane 0's release, for the readers' TMA as well
        tc::fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) return false;
        const bool withhold = (p.test_flags & MOK_FLAG_TEST_WITHHOLD_PUBLISH) && mb == 0 && c == nchunks - 1;
        if (lane == 0 && !withhold) red_release_add(&p.ready[mb * p.E + e], 8);
    }
    return true;
}

// Fixed-order weighted sum of tokens [t0, t1) of one batch (j ascending).
__device__ void combine_tokens(const MegaParams& p, const MegaBatch& bt, int t0, int t1) {
    const int H = p.H, k = p.k;
    const int n = H / 8;
    for (int t = t0; t < t1; ++t) {
        for (int c = threadIdx.x; c < n; c += blockDim.x) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            // up to 8 slots' loads in flight, then their products in j order
            for (int j0 = 0; j0 < k; j0 += 8) {
                uint4 u[8];
                float wj[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (j0 + q < k) {
                        wj[q] = bt.topk_w[(int64_t)t * k + j0 + q];
                        u[q] = __ldcs(reinterpret_cast<const uint4*>(bt.partials + ((int64_t)t * k + j0 + q) * H) + c);
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (j0 + q < k) {
                        acc[0] = fmaf(wj[q], bf16_lo(u[q].x), acc[0]); acc[1] = fmaf(wj[q], bf16_hi(u[q].x), acc[1]);
                        acc[2] = fmaf(wj[q], bf16_lo(u[q].y), acc[2]); acc[3] = fmaf(wj[q], bf16_hi(u[q].y), acc[3]);
                        acc[4] = fmaf(wj[q], bf16_lo(u[q].z), acc[4]); acc[5] = fmaf(wj[q], bf16_hi(u[q].z), acc[5]);
                        acc[6] = fmaf(wj[q], bf16_lo(u[q].w), acc[6]); acc[7] = fmaf(wj[q], bf16_hi(u[q].w), acc[7]);
                    }
                }
            }
            if (bt.shared) {
                const float4* s = reinterpret_cast<const float4*>(bt.shared + (int64_t)t * H) + 2 * c;
                const float4 a = s[0], b = s[1];
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
                acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            reinterpret_cast<uint4*>(bt.out + (int64_t)t * H)[c] = o;
        }
    }
}

constexpr int kCombineChunk = 4;

// Take combine chunks of every minibatch whose down tiles are all finished,
// in minibatch order. blocking: wait for each minibatch in turn (a CTA with
// no other work); otherwise stop at the first unfinished minibatch. Called
// by every thread of the CTA; all decisions are broadcast through s_word.
__device__ bool combine_loop(const MegaParams& p, int NT2, int* s_word, int& next_mb, bool blocking,
                             int budget = 1 << 30, int* done = nullptr) {
    const PlanView& v = p.plan;
    const int n_mb = v.hdr->n_mb;
    StatusBlock* st = p.status;
    int taken = 0;
    while (next_mb < n_mb && taken < budget) {
        const MbInfo mi = v.mb[next_mb];
        const int tiles2 = mi.mtiles * NT2;
        if (threadIdx.x == 0) {
            int ok;
            if (blocking) ok = wait_counter(&p.g2_mb[next_mb], tiles2, st, p.timeout_ns, kSiteCounter) ? 1 : -1;
            else ok = ld_acquire(&p.g2_mb[next_mb]) >= tiles2 ? 1 : 0;
            s_word[0] = ok;
        }
        __syncthreads();
        const int ok = s_word[0];
        __syncthreads();
        if (ok < 0) return false;
        if (ok == 0) return true;
        const MegaBatch bt = p.batches[mi.batch];
        const int nch = ceil_div(mi.t1 - mi.t0, kCombineChunk);
        bool drained = false;
        while (taken < budget) {
            if (threadIdx.x == 0) s_word[1] = atomicAdd(&p.comb_next[next_mb], 1);
            __syncthreads();
            const int ch = s_word[1];
            __syncthreads();
            if (ch >= nch) { drained = true; break; }
            const int t0 = mi.t0 + ch * kCombineChunk;
            combine_tokens(p, bt, t0, min(mi.t1, t0 + kCombineChunk));
            ++taken;
        }
        if (drained) ++next_mb;
    }
    if (done) *done = taken;
    return true;
}

// Trace record of this CTA (thread 0 keeps the values; MOK_FLAG_TRACE).
struct MegaTrace {
    unsigned long long t_begin = 0, t_first = 0, t_work_end = 0, wait_ns = 0, units = 0, comb_ns = 0;
    __device__ void write(unsigned long long* rec, int role) const {
        rec[0] = (unsigned long long)role;
        rec[1] = t_begin;
        rec[2] = t_first;
        rec[3] = t_work_end;
        rec[4] = globaltimer_ns();
        rec[5] = wait_ns;
        rec[6] = units;
        rec[7] = comb_ns;
    }
};

template <bool MX>
__global__ void __launch_bounds__(GemmCfg<256, MX, false, kEpiSwiGLU, 4, MX ? 1 : 2>::kThreads, 1)
mega_kernel(const __grid_constant__ CUtensorMap tmRing, const __grid_constant__ CUtensorMap tmGU,
            const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmDN, const MegaParams p) {
    // gate/up tiles are 256 wide (gate 128 | up 128); MXFP8 keeps one
    // accumulator because its block scales take the rest of tensor memory,
    // and runs 8 epilogue warps (two per TMEM lane quadrant) that copy a
    // tile to registers and release the accumulator before any arithmetic.
    // Down tiles are bn2 wide and use the first bn2 accumulator columns.
    constexpr int BN = 256;
    constexpr int STAGES = 4;
    constexpr int ACC = MX ? 1 : 2;
    using C = GemmCfg<BN, MX, false, kEpiSwiGLU, STAGES, ACC>;
    constexpr int ET = 32 * C::kEpiWarps;   // epilogue threads
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_word[4];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    StatusBlock* st = p.status;
    const uint64_t tmo = p.timeout_ns;
    const int BN2 = p.bn2;
    const int NT1 = 2 * p.I / BN, NT2 = p.H / BN2;
    const int kb1 = p.H / C::kBK, kb2 = p.I / C::kBK;
    const PlanView& v = p.plan;
    int next_comb = 0;
    const bool tracing = p.trace != nullptr;
    MegaTrace tr;
    if (tracing && threadIdx.x == 0) tr.t_begin = globaltimer_ns();

    if (v.hdr->error) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_failure(st, MOK_ERR_CAPACITY, 0);
        return;
    }

    if ((int)blockIdx.x < p.n_movers) {
        // ------------------------------------------------------------ mover CTA
        const int nwarps = p.n_movers * (blockDim.x / 32);
        const int gwarp = blockIdx.x * (blockDim.x / 32) + warp;
        const int n_mb = v.hdr->n_mb;
        // BF16: rows go through the copy engines when the row buffers fit
        const int nw = blockDim.x / 32;
        const size_t rowb = (size_t)p.H * (MX ? 1 : 2);
        const bool pump = (size_t)(2 * nw) * rowb + 16 * nw <= (size_t)C::kBarOffset &&
                          (!MX || p.batches[0].xq != nullptr);
        MoverSmem ms{};
        uint32_t phases = 0;
        unsigned char* sm =
            reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
        if (pump) {
            const uint32_t base = tc::smem_u32(sm);
            ms.bufs = base;
            ms.bars = base + (uint32_t)(2 * nw * rowb);
            if (lane == 0) {
                tc::mbar_init(ms.bars + 16u * warp, 1);
                tc::mbar_init(ms.bars + 16u * warp + 8u, 1);
            }
            tc::fence_mbar_init();
            __syncthreads();
        }
        for (int mb = 0; mb < n_mb; ++mb) {
            if (mb >= 2) {
                // the region is reused once every gate/up tile of mb-2 is done;
                // until then the movers take weighted-sum chunks of finished
                // minibatches, one at a time, so a free region is never kept
                // waiting (bounded by the same time limit as every wait)
                const int target = v.mb[mb - 2].mtiles * NT1;
                const unsigned long long w0 = globaltimer_ns();
                const unsigned long long comb0 = tr.comb_ns;
                for (;;) {
                    if (threadIdx.x == 0) {
                        int ok = ld_acquire(&p.g1_mb[mb - 2]) >= target ? 1 : 0;
                        if (!ok && abort_requested(st)) ok = -1;
                        if (!ok && globaltimer_ns() - w0 > tmo) {
                            record_failure(st, MOK_ERR_TIMEOUT, kSiteCounter);
                            ok = -1;
                        }
                        s_word[0] = ok;
                    }
                    __syncthreads();
                    const int ok = s_word[0];
                    __syncthreads();
                    if (ok < 0) return;
                    if (ok > 0) break;
                    int did = 0;
                    const unsigned long long c0 = (tracing && threadIdx.x == 0) ? globaltimer_ns() : 0ull;
                    if (!combine_loop(p, NT2, s_word, next_comb, false, 1, &did)) return;
                    if (tracing && threadIdx.x == 0) tr.comb_ns += globaltimer_ns() - c0;
                    if (!did && threadIdx.x == 0) __nanosleep(200);
                }
                if (tracing && threadIdx.x == 0) tr.wait_ns += (globaltimer_ns() - w0) - (tr.comb_ns - comb0);
            }
            if (tracing && threadIdx.x == 0 && mb == 0) tr.t_first = globaltimer_ns();
            if (pump) {
                if (!mover_pump_mb<MX>(p, mb, gwarp, nwarps, lane, warp, ms, phases)) return;
            } else {
                mover_dispatch_mb<MX>(p, mb, gwarp, nwarps, lane);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                s_word[3] = abort_requested(st) ? 1 : 0;
                tr.units++;
            }
            __syncthreads();
            if (s_word[3]) return;   // the same decision in every thread
        }
        if (tracing && threadIdx.x == 0) tr.t_work_end = globaltimer_ns();
        const unsigned long long c1 = (tracing && threadIdx.x == 0) ? globaltimer_ns() : 0ull;
        combine_loop(p, NT2, s_word, next_comb, true);
        if (tracing && threadIdx.x == 0) {
            tr.comb_ns += globaltimer_ns() - c1;
            tr.write(p.trace + 8 * blockIdx.x, 0);
        }
        return;
    }

    // ---------------------------------------------------------------- compute CTA
    const int cidx = blockIdx.x - p.n_movers;
    const int ncomp = gridDim.x - p.n_movers;
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = tc::smem_u32(smem);
    const uint32_t bar_base = smem_base + C::kBarOffset;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto accf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto acce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + ACC + a); };
    const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * ACC);
    auto a_tile = [&](int s) { return smem_base + s * C::kStageBytes; };
    auto b_tile = [&](int s) { return smem_base + s * C::kStageBytes + C::kBytesA; };
    auto sf_tile = [&](int s) { return smem_base + STAGES * C::kStageBytes + s * C::kSfStage; };

    if (threadIdx.x == 32) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full_bar(s), 1);
            tc::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < ACC; ++a) {
            tc::mbar_init(accf_bar(a), 1);
            tc::mbar_init(acce_bar(a), ET);
        }
        tc::mbar_init(drain_bar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmRing);
        tc::prefetch_tmap(&tmGU);
        tc::prefetch_tmap(&tmH);
        tc::prefetch_tmap(&tmDN);
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(&s_tmem_base), C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem_base;
    const int total = v.hdr->total_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int last_par[STAGES];
            for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
            bool ok = true;
            for (int g = cidx; g < total && ok; g += ncomp) {
                const MegaTile t = mega_decode(p, g, NT1, NT2);
                // the tile's inputs must be published before its first load
                const unsigned long long w0 = tracing ? globaltimer_ns() : 0ull;
                if (t.kind == 0)
                    ok = wait_counter(&p.ready[t.mb * p.E + t.e], t.mt * kTileM, st, tmo, kSiteCounter);
                else
                    ok = wait_counter(&p.g1_e[t.mb * p.E + t.e], t.mt * NT1, st, tmo, kSiteCounter);
                if (!ok) break;
                if (tracing) {
                    const unsigned long long w1 = globaltimer_ns();
                    tr.wait_ns += w1 - w0;
                    if (tr.units == 0) tr.t_first = w1;
                    tr.units++;
                }
                tc::fence_proxy_async_global();
                const int nkb = t.kind == 0 ? kb1 : kb2;
                const void* tmA = t.kind == 0 ? (const void*)&tmRing : (const void*)&tmH;
                const void* tmB = t.kind == 0 ? (const void*)&tmGU : (const void*)&tmDN;
                const int bnt = t.kind == 0 ? BN : BN2;
                const int nch = (bnt + 127) / 128;
                const int brow = t.e * (t.kind == 0 ? 2 * p.I : p.H) + t.n * bnt;
                const uint8_t* asf = t.kind == 0 ? p.ring_sf : p.h_sf;
                const uint8_t* bsf = t.kind == 0 ? p.gu_sf : p.dn_sf;
                const int kch = t.kind == 0 ? p.H / 128 : p.I / 128;
                const uint32_t tx = C::kBytesA + bnt * 128 + (MX ? 512 * (1 + nch) : 0);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!tc::mbar_wait(empty_bar(stage), ph ^ 1u, st, tmo, kSiteProducerEmpty)) { ok = false; break; }
                    tc::mbar_expect_tx(full_bar(stage), tx);
                    tc::tma_load_2d(a_tile(stage), tmA, full_bar(stage), kb * C::kBK, t.a_row0);
                    tc::tma_load_2d(b_tile(stage), tmB, full_bar(stage), kb * C::kBK, brow);
                    if constexpr (MX) {
                        tc::bulk_load(sf_tile(stage), asf + ((int64_t)(t.a_row0 / kTileM) * kch + kb) * 512, 512,
                                      full_bar(stage));
                        if (bnt == 224)   // down scales kept per 224-row tile: two chunks in one copy
                            tc::bulk_load(sf_tile(stage) + 512, bsf + ((int64_t)(brow / 224) * kch + kb) * 1024, 1024,
                                          full_bar(stage));
                        else
                            for (int j = 0; j < nch; ++j)
                                tc::bulk_load(sf_tile(stage) + 512 * (1 + j),
                                              bsf + ((int64_t)(brow / kTileM + j) * kch + kb) * 512, 512,
                                              full_bar(stage));
                    }
                    last_par[stage] = (int)ph;
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok)  // let every copy already issued land before the CTA moves on
                for (int s = 0; s < STAGES; ++s)
                    if (last_par[s] >= 0) tc::mbar_wait(full_bar(s), (uint32_t)last_par[s], st, tmo, kSiteDrain);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            bool ok = true, issued = false;
            for (int g = cidx; g < total && ok; g += ncomp) {
                const MegaTile t = mega_decode(p, g, NT1, NT2);
                const int nkb = t.kind == 0 ? kb1 : kb2;
                const int bnt = t.kind == 0 ? BN : BN2;
                const int nch = (bnt + 127) / 128;
                if (!tc::mbar_wait(acce_bar(acc), acc_ph ^ 1u, st, tmo, kSiteMmaAccEmpty)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(acc * C::kAccStride);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!tc::mbar_wait(full_bar(stage), ph, st, tmo, kSiteMmaFull)) { ok = false; break; }
                    tc::fence_after_sync();
                    uint32_t sfa_t = 0, sfb_t = 0;
                    if constexpr (MX) {
                        sfa_t = tmem + (uint32_t)C::sf_col(stage);
                        sfb_t = sfa_t + 4;
                        tc::tmem_cp_32x128b_warpx4(sfa_t, tc::make_sdesc(sf_tile(stage), 0, 128, tc::kLayoutNone));
                        for (int j = 0; j < nch; ++j)
                            tc::tmem_cp_32x128b_warpx4(
                                sfb_t + 4 * j, tc::make_sdesc(sf_tile(stage) + 512 * (1 + j), 0, 128, tc::kLayoutNone));
                    }
#pragma unroll
                    for (int kk = 0; kk < C::kMmasPerStage; ++kk) {
                        const uint64_t ad = tc::make_sdesc(a_tile(stage) + kk * 32, 16, 1024, tc::kLayoutSW128);
                        const uint64_t bd = tc::make_sdesc(b_tile(stage) + kk * 32, 16, 1024, tc::kLayoutSW128);
                        const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (MX) tc::mma_mxf8(d, ad, bd, tc::idesc_mxf8(128, bnt, kk, kk), sfa_t, sfb_t, accum);
                        else tc::mma_bf16(d, ad, bd, tc::idesc_bf16(128, bnt, false, false), accum);
                    }
                    issued = true;
                    tc::mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc::mma_commit(accf_bar(acc));
                if (++acc == ACC) { acc = 0; acc_ph ^= 1u; }
            }
            if (!ok && issued) {  // every MMA issued must finish before TMEM is freed
                tc::mma_commit(drain_bar);
                tc::mbar_wait(drain_bar, 0, st, tmo, kSiteDrain);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int etid = threadIdx.x - 64;  // 0..ET-1
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int g = cidx; g < total; g += ncomp) {
            const MegaTile t = mega_decode(p, g, NT1, NT2);
            const MbInfo mi = v.mb[t.mb];
            if (t.kind == 0 && t.mb >= 2) {
                // h region reuse: the down tiles of mb-2 must have read it
                if (etid == 0)
                    s_word[2] = wait_counter(&p.g2_mb[t.mb - 2], v.mb[t.mb - 2].mtiles * NT2, st, tmo, kSiteCounter);
                asm volatile("bar.sync 1, %0;" ::"r"(ET) : "memory");
                if (!s_word[2]) break;
            }
            const bool okw = tc::mbar_wait(accf_bar(acc), acc_ph, st, tmo, kSiteEpiAccFull);
            if (!bar_and(1, ET, okw)) break;  // all epilogue threads agree
            tc::fence_after_sync();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccStride);
            if constexpr (C::kWideEpi) {
                // MXFP8: this warp's columns to registers, accumulator released
                const int eg = (warp - 2) >> 2;
                if (t.kind == 0) {
                    // 64 h columns: two 32-element blocks, scale codes 2*eg, 2*eg+1
                    uint32_t gr0[32], gr1[32], ur0[32], ur1[32];
                    tc::tmem_ld_32x32b_x32(tbase + 64 * eg, gr0);
                    tc::tmem_ld_32x32b_x32(tbase + 64 * eg + 32, gr1);
                    tc::tmem_ld_32x32b_x32(tbase + BN / 2 + 64 * eg, ur0);
                    tc::tmem_ld_32x32b_x32(tbase + BN / 2 + 64 * eg + 32, ur1);
                    tc::tmem_ld_wait();
                    tc::fence_before_sync();
                    tc::mbar_arrive(acce_bar(acc));
                    const int I = p.I;
                    const int64_t prow = t.a_row0 + row;
                    const int hc0 = t.n * (BN / 2) + 64 * eg;
                    uint32_t codes = 0;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        float hv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            hv[i] = silu_f(__uint_as_float(b ? gr1[i] : gr0[i])) * __uint_as_float(b ? ur1[i] : ur0[i]);
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
                        const uint32_t code = e8m0_code(amax);
                        const float inv = e8m0_inv_scale(code);
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = f32x2_to_e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv) |
                                   (f32x2_to_e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv) << 16);
                        tc::stg_v8(static_cast<uint8_t*>(p.hbuf) + prow * (int64_t)I + hc0 + 32 * b, w);
                        codes |= code << (8 * b);
                    }
                    const int64_t chunk = (prow / kTileM) * (int64_t)(I / 128) + hc0 / 128;
                    *reinterpret_cast<uint16_t*>(p.h_sf + chunk * 512 +
                                                 sf_chunk_offset((int)(prow % kTileM), 2 * eg)) = (uint16_t)codes;
                } else {
                    // 32-column chunks eg, eg+2, eg+4, eg+6 of the bn2-wide tile
                    const MegaBatch bt = p.batches[mi.batch];
                    const int lrow = t.local_row0 + row;
                    int64_t dest = -1;
                    if (lrow < v.cnt[t.mb * p.E + t.e]) dest = bt.row_src[v.src0[t.mb * p.E + t.e] + lrow];
                    const int nch = BN2 / 32;
                    // packed to BF16 two chunks at a time (fewer live registers);
                    // chunks past the tile read its last chunk again, unused
                    uint32_t w0[16], w1[16], w2[16], w3[16];
                    auto load_pair = [&](int c, uint32_t(&wa)[16], uint32_t(&wb)[16]) {
                        uint32_t ra[32], rb[32];
                        tc::tmem_ld_32x32b_x32(tbase + 32 * min(c, nch - 1), ra);
                        tc::tmem_ld_32x32b_x32(tbase + 32 * min(c + 2, nch - 1), rb);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            wa[i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
                            wb[i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
                        }
                    };
                    load_pair(eg, w0, w1);
                    load_pair(eg + 4, w2, w3);
                    tc::fence_before_sync();
                    tc::mbar_arrive(acce_bar(acc));
                    if (dest >= 0) {
                        __nv_bfloat16* orow = bt.partials + dest * p.H + t.n * BN2;
                        auto store_chunk = [&](int c, const uint32_t(&w)[16]) {
                            tc::stg_v8(orow + 32 * c, w);
                            tc::stg_v8(orow + 32 * c + 16, w + 8);
                        };
                        if (eg < nch) store_chunk(eg, w0);
                        if (eg + 2 < nch) store_chunk(eg + 2, w1);
                        if (eg + 4 < nch) store_chunk(eg + 4, w2);
                        if (eg + 6 < nch) store_chunk(eg + 6, w3);
                    }
                }
            } else if (t.kind == 0) {
                const int I = p.I;
                const int64_t prow = t.a_row0 + row;
                uint32_t sfw = 0;   // MXFP8: scale codes of the current 128-wide chunk of h
#pragma unroll 1
                for (int c0 = 0; c0 < BN / 2; c0 += 32) {
                    uint32_t gr[32], ur[32];
                    load_gate_up<BN, !MX>(tbase, c0, gr, ur);
                    const int hc = t.n * (BN / 2) + c0;
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) hv[i] = silu_f(__uint_as_float(gr[i])) * __uint_as_float(ur[i]);
                    if constexpr (MX) {
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
                        const uint32_t code = e8m0_code(amax);
                        const float inv = e8m0_inv_scale(code);
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = f32x2_to_e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv) |
                                   (f32x2_to_e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv) << 16);
                        tc::stg_v8(static_cast<uint8_t*>(p.hbuf) + prow * (int64_t)I + hc, w);
                        // the four codes of a 128-wide chunk leave as one word
                        sfw |= code << (8 * ((hc / 32) & 3));
                        if (((hc / 32) & 3) == 3) {
                            const int64_t chunk = (prow / kTileM) * (int64_t)(I / 128) + hc / 128;
                            *reinterpret_cast<uint32_t*>(p.h_sf + chunk * 512 +
                                                         sf_chunk_offset((int)(prow % kTileM), 0)) = sfw;
                            sfw = 0;
                        }
                    } else {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.hbuf) + prow * (int64_t)I + hc;
                        tc::stg_v8(dst, w);
                        tc::stg_v8(dst + 16, w + 8);
                    }
                }
            } else {
                const MegaBatch bt = p.batches[mi.batch];
                const int lrow = t.local_row0 + row;
                int64_t dest = -1;
                if (lrow < v.cnt[t.mb * p.E + t.e]) dest = bt.row_src[v.src0[t.mb * p.E + t.e] + lrow];
#pragma unroll 1
                for (int c0 = 0; c0 < BN2; c0 += 32) {
                    uint32_t r[32];
                    tc::tmem_ld_32x32b_x32(tbase + c0, r);
                    tc::tmem_ld_wait();
                    if (dest < 0) continue;
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    __nv_bfloat16* dst = bt.partials + dest * p.H + t.n * BN2 + c0;
                    tc::stg_v8(dst, w);
                    tc::stg_v8(dst + 16, w + 8);
                }
            }
            if constexpr (!C::kWideEpi) {
                tc::fence_before_sync();
                tc::mbar_arrive(acce_bar(acc));
            }
            if (++acc == ACC) { acc = 0; acc_ph ^= 1u; }
            // publish the tile: all epilogue threads' stores, then one release
            __threadfence();
            tc::fence_proxy_async_global();
            asm volatile("bar.sync 1, %0;" ::"r"(ET) : "memory");
            if (etid == 0) {
                if (t.kind == 0) {
                    red_release_add(&p.g1_e[t.mb * p.E + t.e], 1);
                    red_release_add(&p.g1_mb[t.mb], 1);
                } else {
                    red_release_add(&p.g2_mb[t.mb], 1);
                }
            }
        }
    }
    // every role of this CTA is done with tiles: join the weighted sums
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (threadIdx.x == 0) {
        s_word[3] = abort_requested(st) ? 1 : 0;
        if (tracing) tr.t_work_end = globaltimer_ns();
    }
    __syncthreads();
    if (!s_word[3]) combine_loop(p, NT2, s_word, next_comb, true);
    __syncthreads();
    if (tracing && threadIdx.x == 0) {
        tr.comb_ns = globaltimer_ns() - tr.t_work_end;
        tr.write(p.trace + 8 * blockIdx.x, 1);
    }
    if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 mega_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Row-major [rows, cols] tensor, box of 128 bytes x box_rows, 128-byte swizzle.
bool tmap2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int eb, int box_rows) {
    auto fn = mega_encode();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * eb)};
    cuuint32_t box[2] = {(cuuint32_t)(128 / eb), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapDataType dt = eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

size_t mega_scratch_bytes(int nbatch, int T, int H, int I, int E, int k, int region_rows, bool mx) {
    (void)T;
    (void)k;
    const int64_t eb = mx ? 1 : 2;
    size_t o = kMegaTraceBytes;
    o += plan_bytes(E);
    o += align_up((int64_t)nbatch * plan_stage_ints(E) * 4, 1024);        // plan staging
    o += align_up((int64_t)kMaxMinibatches * (2 * E + 3) * 4, 1024);      // counters
    o += align_up(2 * (int64_t)region_rows * H * eb, 1024);               // ring
    if (mx) o += align_up(2 * (int64_t)region_rows * H / 32, 1024);
    o += align_up(2 * (int64_t)region_rows * I * eb, 1024);               // h
    if (mx) o += align_up(2 * (int64_t)region_rows * I / 32, 1024);
    if (mx) o += (size_t)nbatch * (align_up((int64_t)T * H, 1024) + align_up((int64_t)T * H / 32, 1024));  // x quantised
    return o;
}

cudaError_t launch_mega(const MegaLaunch& L, cudaStream_t s) {
    const bool mx = L.mx;
    const int E = L.E, H = L.H, I = L.I, k = L.k, T = L.T, nb = L.nbatch;
    const int64_t eb = mx ? 1 : 2;
    char* w = static_cast<char*>(L.scratch) + kMegaTraceBytes;
    if (L.grid > kMegaTraceCtas) return cudaErrorInvalidValue;
    PlanView v = plan_view(w, E);
    w += plan_bytes(E);
    int* stage = reinterpret_cast<int*>(w);
    w += align_up((int64_t)nb * plan_stage_ints(E) * 4, 1024);
    int* counters = reinterpret_cast<int*>(w);
    const size_t counter_bytes = (size_t)kMaxMinibatches * (2 * E + 3) * 4;
    w += align_up(counter_bytes, 1024);
    void* ring = w;
    w += align_up(2 * (int64_t)L.region_rows * H * eb, 1024);
    uint8_t* ring_sf = nullptr;
    if (mx) { ring_sf = reinterpret_cast<uint8_t*>(w); w += align_up(2 * (int64_t)L.region_rows * H / 32, 1024); }
    void* hbuf = w;
    w += align_up(2 * (int64_t)L.region_rows * I * eb, 1024);
    uint8_t* h_sf = nullptr;
    if (mx) { h_sf = reinterpret_cast<uint8_t*>(w); w += align_up(2 * (int64_t)L.region_rows * I / 32, 1024); }
    // MXFP8: every batch's rows quantised once per token; the movers copy them
    uint8_t* xq[kMaxBatches] = {};
    uint8_t* xsf[kMaxBatches] = {};
    if (mx) {
        for (int b = 0; b < nb; ++b) {
            xq[b] = reinterpret_cast<uint8_t*>(w);
            w += align_up((int64_t)T * H, 1024);
            xsf[b] = reinterpret_cast<uint8_t*>(w);
            w += align_up((int64_t)T * H / 32, 1024);
            cudaError_t eq = launch_quantize_rows(L.x[b], T, H, xq[b], xsf[b], s);
            if (eq != cudaSuccess) return eq;
        }
    }

    PlanBatches pbs;
    for (int b = 0; b < nb; ++b) {
        pbs.b[b].offsets = L.offsets[b];
        pbs.b[b].row_src = L.row_src[b];
    }
    cudaError_t e = cudaMemsetAsync(counters, 0, counter_bytes, s);
    if (e != cudaSuccess) return e;

    const int BN = 256, BN2 = down_tile_n(H, mx);
    const int NT1 = 2 * I / BN, NT2 = H / BN2;
    const int nblk = ceil_div(T, kPlanTB);
    const size_t psm = (size_t)(nblk + 1) * E * 4;
    if (psm > 48 * 1024) ensure_smem_attr(reinterpret_cast<const void*>(plan_batch_kernel), (int)psm);
    plan_batch_kernel<<<nb, 256, psm, s>>>(pbs, T, E, k, L.region_rows, L.max_tokens, L.tile_cuts ? 1 : 0, stage);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    plan_finalize_kernel<<<1, 256, 0, s>>>(nb, E, NT1, NT2, stage, v);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    MegaParams p{};
    p.E = E; p.H = H; p.I = I; p.k = k; p.T = T; p.nbatch = nb;
    for (int b = 0; b < nb; ++b) {
        p.batches[b].x = static_cast<const __nv_bfloat16*>(L.x[b]);
        p.batches[b].xq = xq[b];
        p.batches[b].xsf = reinterpret_cast<const uint32_t*>(xsf[b]);
        p.batches[b].row_src = L.row_src[b];
        p.batches[b].topk_w = L.topk_w[b];
        p.batches[b].partials = static_cast<__nv_bfloat16*>(L.partials[b]);
        p.batches[b].shared = L.shared[b];
        p.batches[b].out = static_cast<__nv_bfloat16*>(L.out[b]);
    }
    p.plan = v;
    p.ring = ring; p.ring_sf = ring_sf; p.region_rows = L.region_rows;
    p.hbuf = hbuf; p.h_sf = h_sf;
    p.gu_sf = L.gu_sf; p.dn_sf = L.dn_sf;
    p.ready = counters;
    p.g1_e = counters + kMaxMinibatches * E;
    p.g1_mb = counters + 2 * kMaxMinibatches * E;
    p.g2_mb = p.g1_mb + kMaxMinibatches;
    p.comb_next = p.g2_mb + kMaxMinibatches;
    p.bn2 = BN2;
    p.n_movers = L.n_movers;
    p.test_flags = L.test_flags;
    p.trace = L.trace;
    p.status = L.status;
    p.timeout_ns = L.timeout_ns;

    CUtensorMap tR, tGU, tH, tDN;
    const int64_t rrows = 2 * (int64_t)L.region_rows;
    if (!tmap2d(&tR, ring, rrows, H, (int)eb, 128)) return cudaErrorInvalidValue;
    if (!tmap2d(&tGU, L.gu, (int64_t)E * 2 * I, H, (int)eb, BN)) return cudaErrorInvalidValue;
    if (!tmap2d(&tH, hbuf, rrows, I, (int)eb, 128)) return cudaErrorInvalidValue;
    if (!tmap2d(&tDN, L.dn, (int64_t)E * H, I, (int)eb, BN2)) return cudaErrorInvalidValue;

    // Cooperative launch: refused unless every CTA can be resident at once,
    // which the counter waits between CTAs rely on.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(L.grid);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (mx) {
        using C = GemmCfg<256, true, false, kEpiSwiGLU, 4, 1>;
        ensure_smem_attr(reinterpret_cast<const void*>(mega_kernel<true>), C::kSmemBytes);
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        e = cudaLaunchKernelEx(&cfg, mega_kernel<true>, tR, tGU, tH, tDN, p);
    } else {
        using C = GemmCfg<256, false, false, kEpiSwiGLU, 4, 2>;
        ensure_smem_attr(reinterpret_cast<const void*>(mega_kernel<false>), C::kSmemBytes);
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        e = cudaLaunchKernelEx(&cfg, mega_kernel<false>, tR, tGU, tH, tDN, p);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mok
