// gemm.cuh - persistent grouped GEMM on tcgen05 tensor cores (sm_103a).
//
// One kernel template serves every expert GEMM of the layer ("grouped GEMM"
// over each expert's contiguous token segment, as the KuCoin article on MoK
// describes in section 01): the forward gate/up GEMM with the SwiGLU epilogue,
// the forward down GEMM whose epilogue pushes each row to its (token, slot)
// partial, the backward dgrad GEMMs, and the backward wgrad GEMMs that reduce
// over each expert's rows.
//
// CTA layout (one CTA per SM, persistent over tiles):
//   warp 0     TMA producer: streams A and B K-blocks into a ring of smem
//              stages (and, for MXFP8, the 512-byte scale chunks)
//   warp 1     allocates tensor memory; one lane issues tcgen05.mma into a
//              double-buffered fp32 accumulator in TMEM
//   warps 2-5  epilogue: tcgen05.ld the accumulator (one row per thread) and
//              apply the fused epilogue, then release the accumulator
//   (MXFP8 gate/up: warps 2-9, two per TMEM lane quadrant; its block scales
//   leave room for one accumulator only, so these warps copy the tile to
//   registers and release the accumulator before the SwiGLU arithmetic)
// Every wait is bounded (StatusBlock); nothing traps.
#pragma once

#include "tc.cuh"

namespace mok {

enum EpiKind : int {
    kEpiSwiGLU = 0,   // h = silu(G) * U (bf16 or MXFP8), optional fp32 G/U save
    kEpiScatter = 1,  // row -> slot (or identity) store, bf16 or f32
    kEpiDSwiGLU = 2,  // dh -> dG, dU using saved G, U
    kEpiDense = 3,    // dense tile store (wgrad), column split into two outputs
};

struct GemmParams {
    int E;
    int n_tiles;            // output tiles along N per expert
    int num_kb;             // K-blocks for grouped-M kinds
    int b_rows_per_expert;  // B row stride between experts (K-major B)
    int b_split_kb;         // K-blocks >= this read from tmB2 (dgrad2); large = never
    // row groups
    const int32_t* counts;  // [E] routed rows per expert (grouped kinds)
    int identity_rows;      // > 0: a single group of this many rows, no padding
    int m_fixed;            // wgrad: output rows per expert; 0 otherwise
    // epilogue
    void* out0;
    void* out1;
    int ldo;                // leading dimension (elements) of out0/out1
    int split_col;          // dense: columns >= split go to out1; SwiGLU/DSwiGLU: I
    uint8_t* out_sf;        // MXFP8 h scales (SwiGLU)
    void* gu;               // SwiGLU: G/U save target; DSwiGLU: G/U source ([rows, 2I] fp32)
    const int32_t* offsets; // scatter: unpadded offsets [E+1]
    const int32_t* row_src; // scatter: row -> slot
    int out_f32;            // scatter: store fp32 instead of bf16
    // MXFP8 scales of A and B (tile-ordered chunks)
    const uint8_t* a_sf;
    const uint8_t* b_sf;
    const uint8_t* b_sf2;   // scales of the second B operand (K blocks >= b_split_kb)
    int sf_kchunks;         // 128-wide K chunks per row tile of A (= K / 128)
    int sf_kchunks_b;       // the same for B when it differs (0: as A)
    // weight gradients on K-major MXFP8 operands: A is [m_fixed, K] and B is
    // [N, K] with the tokens as K, each expert reducing over its own token
    // range (the segment of its rows in the padded layout)
    int kmajor_wgrad;
    void* out1_bf16;        // MXFP8 SwiGLU: h also in BF16 [rows, I] (training forward), or NULL
    StatusBlock* status;
    unsigned long long timeout_ns;
};

// CLN = 2: one CTA of a 2-SM pair, which holds its 128 A rows and half of
// the BN B rows of the pair's 256 x BN tile.
template <int BN, bool MX, bool MN_MAJOR, int EPI, int STAGES, int ACC_STAGES, int CLN = 1>
struct GemmCfg {
    static_assert(CLN == 1 || (CLN == 2 && BN % 32 == 0 && (!MX || BN == 256) &&
                               (!MN_MAJOR || (!MX && EPI == kEpiDense && BN == 256))),
                  "2-SM pairs: K-major, or the BF16 MN-major weight gradients");
    // MXFP8 tiles 256 wide keep one accumulator (their scales take the rest
    // of TMEM) and hide the epilogue behind the next tile with 8 epilogue
    // warps.
    static constexpr bool kWideEpi = MX && ACC_STAGES == 1;
    static constexpr int kEpiWarps = kWideEpi ? 8 : 4;
    // BF16 2-SM pairs run an expert's odd last 128-row tile as an M=128 pair
    // (64 rows per CTA; tmX0 then maps A in boxes of 64 rows)
    static constexpr bool kPairTails = CLN == 2 && !MX && !MN_MAJOR && EPI != kEpiDense;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    // BF16 grouped-row forward tiles: an expert's last tile with at most 64
    // rows runs M=64 MMAs (rows 16q..16q+15 land in TMEM lanes 32q..32q+15)
    static constexpr bool kHalfTiles = !MX && !MN_MAJOR && CLN == 1 && (EPI == kEpiSwiGLU || EPI == kEpiScatter);
    static constexpr int kBytesA = 128 * 128;          // 128 rows (or K rows) x 128 bytes
    static constexpr int kBytesB = BN / CLN * 128;
    static constexpr int kStageBytes = kBytesA + kBytesB;
    static constexpr int kNChunks = (BN + 127) / 128;   // 128-row scale chunks of a B tile
    static constexpr int kSfaBytes = MX ? 512 : 0;
    static constexpr int kSfbBytes = MX ? kNChunks * 512 : 0;
    static constexpr int kSfStage = kSfaBytes + kSfbBytes;
    static constexpr int kBK = MX ? 128 : 64;           // K elements per stage (128 bytes)
    static constexpr int kUmmaK = MX ? 32 : 16;
    static constexpr int kMmasPerStage = kBK / kUmmaK;  // 4
    // Accumulator buffers start on 256-column boundaries when BN = 224, so the
    // block scales (MXFP8) fit in the two 32-column gaps behind them.
    static constexpr int kAccStride = BN == 224 ? 256 : BN;
    static constexpr int kAccCols = kAccStride * ACC_STAGES;
    static constexpr int kSfCols = MX ? 4 + 4 * kNChunks : 0;
    static constexpr bool kSfInGaps = MX && BN == 224 && ACC_STAGES == 2;
    static constexpr int kTmemNeed = kSfInGaps ? 512 : kAccCols + STAGES * kSfCols;
    // first tensor-memory column of stage s's scales (A: 4 columns, then B)
    __host__ __device__ static constexpr int sf_col(int s) {
        return kSfInGaps ? BN + (s / 2) * 256 + (s % 2) * kSfCols : kAccCols + s * kSfCols;
    }
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
    static constexpr int kBarOffset = STAGES * (kStageBytes + kSfStage);
    // dense epilogue: per epilogue warp two 32 x 32 BF16 staging blocks for
    // its TMA stores, 1 KB past the barriers
    static constexpr int kEpiStageOffset = kBarOffset + 1024;
    // (the wide MXFP8 dense epilogue stores from registers and stages nothing)
    static constexpr int kEpiStageBytes = (EPI == kEpiDense && !kWideEpi) ? 4 * 2 * 2048 : 0;
    static constexpr int kSmemBytes = 1024 /*align slack*/ + kBarOffset + (EPI == kEpiDense ? 1024 : 256) + kEpiStageBytes;
    static_assert(kTmemNeed <= 512, "tensor memory budget");
    static_assert(BN % 32 == 0 && BN <= 256, "BN");
    static_assert(EPI != kEpiSwiGLU || (BN / 2) % 32 == 0, "SwiGLU tiles hold whole 32-column gate/up chunks");
    static_assert(!(MX && EPI == kEpiSwiGLU) || (BN / 2) % 128 == 0, "MXFP8 h tiles hold whole 128-wide scale chunks");
    static_assert(!kSfInGaps || (STAGES <= 4 && 2 * kSfCols <= 256 - BN), "scale columns must fit the gaps");
    static_assert(!(MX && MN_MAJOR), "MXFP8 operands are K-major");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct TileInfo {
    int e, m, n;
    int a_row0;      // K-major: first A row; MN-major: first K row of the expert segment
    int num_kb;
    int row_base;    // first padded row of the tile (output row space of A rows)
    int local_row0;  // first expert-local row of the tile
    int valid;       // 0: skip
    int half;        // 1: the expert's last tile holds at most 64 rows; one M=64 MMA per K step
    int m128;        // 2-SM pairs: the pair shares one 128-row tile, 64 rows per CTA, M=128 MMAs
};

// Per-CTA copy of the group schedule.
struct Sched {
    int poff[kMaxE + 1];   // padded row offset of each expert segment
    int toff[kMaxE + 1];   // first tile of each expert
};

// Tiles per expert: (m-tiles, or m-tile pairs for 2-SM pairs) x n_tiles.
template <int BN, bool MN_MAJOR, int CLN = 1>
__device__ __forceinline__ void build_sched(const GemmParams& p, Sched& s) {
    if (threadIdx.x == 0) {
        int rows = 0, tiles = 0;
        for (int e = 0; e < p.E; ++e) {
            int cnt = p.identity_rows > 0 ? p.identity_rows : p.counts[e];
            int mt = ceil_div(cnt, kTileM);
            s.poff[e] = rows;
            s.toff[e] = tiles;
            rows += p.identity_rows > 0 ? cnt : mt * kTileM;
            tiles += p.m_fixed > 0 ? ceil_div(p.m_fixed, kTileM * CLN) * p.n_tiles : ceil_div(mt, CLN) * p.n_tiles;
        }
        s.poff[p.E] = rows;
        s.toff[p.E] = tiles;
    }
}

template <int BN, bool MN_MAJOR, int BK>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, const Sched& s, int g) {
    TileInfo ti;
    int lo = 0, hi = p.E - 1;  // last e with toff[e] <= g
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s.toff[mid] <= g) lo = mid; else hi = mid - 1;
    }
    int e = lo;
    int local = g - s.toff[e];
    ti.e = e;
    if (p.m_fixed > 0) {
        int mt = ceil_div(p.m_fixed, kTileM);
        ti.n = local / mt;
        ti.m = local % mt;
        int cnt = p.counts[e];
        ti.a_row0 = s.poff[e];
        ti.num_kb = (ceil_div(cnt, kTileM) * kTileM) / BK;
        ti.row_base = ti.m * kTileM;
        ti.local_row0 = ti.m * kTileM;
    } else {
        int cnt = p.identity_rows > 0 ? p.identity_rows : p.counts[e];
        int mt = ceil_div(cnt, kTileM);
        ti.n = local / mt;
        ti.m = local % mt;
        ti.a_row0 = s.poff[e] + ti.m * kTileM;
        ti.num_kb = p.num_kb;
        ti.row_base = ti.a_row0;
        ti.local_row0 = ti.m * kTileM;
    }
    ti.valid = 1;
    ti.half = 0;
    ti.m128 = 0;
    return ti;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Gate and up pre-activations of 32 consecutive h columns of a gate/up tile
// (tile-local h columns c0 .. c0+31) from the accumulator at tbase. The
// packed weights interleave gate and up rows per `il` rows: BF16 packs 16
// (tile columns 32g .. 32g+15 are gate, 32g+16 .. 32g+31 up, of the same
// 16 features), MXFP8 packs half the 256-wide tile (gate columns 0..127,
// up 128..255).
template <int BN, bool IL16>
__device__ __forceinline__ void load_gate_up(uint32_t tbase, int c0, uint32_t (&gr)[32], uint32_t (&ur)[32]) {
    if constexpr (IL16) {
        uint32_t a[32], b[32];
        tc::tmem_ld_32x32b_x32(tbase + 2 * c0, a);
        tc::tmem_ld_32x32b_x32(tbase + 2 * c0 + 32, b);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            gr[i] = a[i];
            ur[i] = a[16 + i];
            gr[16 + i] = b[i];
            ur[16 + i] = b[16 + i];
        }
    } else {
        tc::tmem_ld_32x32b_x32(tbase + c0, gr);
        tc::tmem_ld_32x32b_x32(tbase + BN / 2 + c0, ur);
        tc::tmem_ld_wait();
    }
}

// 2-SM pairs: pair tile g covers m-tiles 2mp and 2mp+1 of one expert (n
// fastest-varying after mp, as for single tiles); CTA `rank` takes m-tile
// 2mp + rank. An expert with an odd number of m-tiles: with TAILS its last
// pair shares the single last m-tile, CTA `rank` taking its rows 64*rank ..
// 64*rank+63, and runs M=128 MMAs (m128); without, the second CTA's rows lie
// outside the segment (valid = 0) and its epilogue stores nothing.
template <int BK, bool TAILS = false>
__device__ __forceinline__ TileInfo decode_pair_tile(const GemmParams& p, const Sched& s, int g, int rank) {
    TileInfo ti;
    int lo = 0, hi = p.E - 1;  // last e with toff[e] <= g
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s.toff[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int cnt = p.identity_rows > 0 ? p.identity_rows : p.counts[e];
    if (p.m_fixed > 0) {
        // weight gradients: M = the fixed weight rows (a multiple of 256), in
        // pairs of 128-row tiles; K = the expert's padded token segment
        const int mp = p.m_fixed / (2 * kTileM);
        const int local = g - s.toff[e];
        ti.e = e;
        ti.n = local / mp;
        ti.m = 2 * (local % mp) + rank;
        ti.a_row0 = s.poff[e];
        ti.num_kb = (ceil_div(cnt, kTileM) * kTileM) / BK;
        ti.row_base = ti.m * kTileM;
        ti.local_row0 = ti.m * kTileM;
        ti.valid = 1;
        ti.half = 0;
        ti.m128 = 0;
        return ti;
    }
    const int mt = ceil_div(cnt, kTileM);
    const int mp = ceil_div(mt, 2);
    const int local = g - s.toff[e];
    ti.e = e;
    ti.n = local / mp;
    const int pp = local % mp;
    ti.m128 = (TAILS && (mt & 1) && pp == mp - 1) ? 1 : 0;
    ti.m = ti.m128 ? mt - 1 : 2 * pp + rank;
    const int r0 = ti.m * kTileM + (ti.m128 ? 64 * rank : 0);   // first expert-local row of this CTA
    ti.a_row0 = s.poff[e] + r0;
    ti.num_kb = p.num_kb;
    ti.row_base = ti.a_row0;
    ti.local_row0 = r0;
    ti.valid = ti.m < mt ? 1 : 0;
    ti.half = 0;
    return ti;
}

// CLN = 2: launched as clusters of two CTAs forming a 2-SM pair
// (tcgen05 cta_group::2). Both CTAs load their own 128 A rows and half of
// the B rows into their own shared memory, signalling the leader's (rank 0)
// full barrier; the leader's MMA thread issues M=256 MMAs over both CTAs'
// operands, each CTA's tensor memory receiving its own 128 accumulator rows,
// and its commits release the stage and publish the accumulator in both
// CTAs; both CTAs' epilogues drain their own rows and release the
// accumulator on the leader's barrier. Per K-block each CTA stages 32 KB
// instead of 48 KB (BN = 256), so 6 stages fit.
template <int BN, bool MX, bool MN_MAJOR, int EPI, int STAGES, int ACC_STAGES, int CLN>
__global__ void __launch_bounds__(GemmCfg<BN, MX, MN_MAJOR, EPI, STAGES, ACC_STAGES, CLN>::kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmX0,
                    const __grid_constant__ CUtensorMap tmX1, const GemmParams p) {
    // tmX0 / tmX1: MXFP8 2-SM pairs - the A and B scale chunks as 256-byte
    // rows; dense epilogue - the outputs out0 / out1 as [E, m_fixed, width]
    // BF16 (boxes of 32 x 32 x 1); unused otherwise
    using C = GemmCfg<BN, MX, MN_MAJOR, EPI, STAGES, ACC_STAGES, CLN>;
    static_assert(CLN == 1 || (CLN == 2 && (EPI != kEpiDense || MX || MN_MAJOR)),
                  "2-SM pairs: grouped-row GEMMs and the weight gradients");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ Sched sched;
    __shared__ uint32_t s_tmem_base;

    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = tc::smem_u32(smem);
    const uint32_t bar_base = smem_base + C::kBarOffset;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto accf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto acce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + ACC_STAGES + a); };
    const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * ACC_STAGES);
    auto a_tile = [&](int s) { return smem_base + s * C::kStageBytes; };
    auto b_tile = [&](int s) { return smem_base + s * C::kStageBytes + C::kBytesA; };
    auto sf_tile = [&](int s) { return smem_base + STAGES * C::kStageBytes + s * C::kSfStage; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    StatusBlock* st = p.status;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 32) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full_bar(s), 1);
            tc::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < ACC_STAGES; ++a) {
            tc::mbar_init(accf_bar(a), 1);
            // pairs: both CTAs' epilogue threads arrive on the leader's barrier
            tc::mbar_init(acce_bar(a), 32 * C::kEpiWarps * CLN);
        }
        tc::mbar_init(drain_bar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmA);
        tc::prefetch_tmap(&tmB);
        tc::prefetch_tmap(&tmB2);
        if constexpr ((MX && CLN == 2) || EPI == kEpiDense) {
            tc::prefetch_tmap(&tmX0);
            tc::prefetch_tmap(&tmX1);
        }
    }
    if (warp == 1) {
        if constexpr (CLN == 2) {
            tc::tmem_alloc_2sm(tc::smem_u32(&s_tmem_base), C::kTmemCols);
            tc::tmem_relinquish_2sm();
        } else {
            tc::tmem_alloc(tc::smem_u32(&s_tmem_base), C::kTmemCols);
            tc::tmem_relinquish();
        }
    }
    // everything above touches only shared and tensor memory: with a
    // programmatic launch it overlaps the end of the kernel before
    pdl_wait();
    pdl_allow_next();
    build_sched<BN, MN_MAJOR, CLN>(p, sched);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if constexpr (CLN == 2) tc::cluster_sync();   // the peer's barriers and tensor memory exist
    const uint32_t tmem = s_tmem_base;
    const int rank = CLN == 2 ? (int)tc::cluster_ctarank() : 0;
    const int gstart = (int)blockIdx.x / CLN;
    const int gstep = (int)gridDim.x / CLN;
    const int gtotal = sched.toff[p.E];
    // M=64 last tiles: grouped rows only, and not when the forward keeps
    // G|U for the backward (the weight gradients read every padded row)
    const bool half_ok = C::kHalfTiles && p.identity_rows == 0 && p.m_fixed == 0 &&
                         (EPI != kEpiSwiGLU || p.gu == nullptr);
    auto decode = [&](int gi) {
        if constexpr (CLN == 2) {
            return decode_pair_tile<C::kBK, C::kPairTails>(p, sched, gi, rank);
        } else {
            TileInfo ti = decode_tile<BN, MN_MAJOR, C::kBK>(p, sched, gi);
            ti.half = half_ok && p.counts[ti.e] - ti.local_row0 <= 64 ? 1 : 0;
            return ti;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int last_par[STAGES];
            for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
            bool ok = true;
            for (int gi = gstart; gi < gtotal && ok; gi += gstep) {
                TileInfo ti = decode(gi);
                for (int kb = 0; kb < ti.num_kb; ++kb) {
                    if (!tc::mbar_wait(empty_bar(stage), ph ^ 1u, st, tmo, kSiteProducerEmpty)) { ok = false; break; }
                    if constexpr (CLN == 2) {
                        // both halves signal the leader's full barrier, which expects both
                        const uint32_t lead_full = tc::mapa_shared(full_bar(stage), 0);
                        // an M=128 pair tile stages 64 A rows per CTA
                        const uint32_t abytes = (C::kPairTails && ti.m128) ? C::kBytesA / 2 : C::kBytesA;
                        if (rank == 0)
                            tc::mbar_expect_tx(full_bar(stage), 2 * (abytes + C::kBytesB + C::kSfStage));
                        if constexpr (MN_MAJOR) {
                            // BF16 weight gradients: K rows of the expert's token range; A
                            // this CTA's 128 weight columns, B its half of the tile's columns
                            const int krow = ti.a_row0 + kb * 64;
                            const int m0 = ti.m * kTileM;
                            tc::tma_load_2d_2sm(a_tile(stage), &tmA, lead_full, m0, krow);
                            tc::tma_load_2d_2sm(a_tile(stage) + 8192, &tmA, lead_full, m0 + 64, krow);
#pragma unroll
                            for (int j = 0; j < BN / 128; ++j)
                                tc::tma_load_2d_2sm(b_tile(stage) + 8192 * j, &tmB, lead_full,
                                                    ti.n * BN + rank * (BN / 2) + 64 * j, krow);
                            last_par[stage] = (int)ph;
                            if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                            continue;
                        }
                        // K-major weight gradients: K is the expert's token range, A rows
                        // this CTA's 128 weight rows, B rows the tile's N columns
                        const bool kw = p.kmajor_wgrad != 0;
                        const int ax = kw ? ti.a_row0 + kb * C::kBK : kb * C::kBK;
                        const int ay = kw ? ti.m * kTileM : ti.a_row0;
                        if (C::kPairTails && ti.m128) tc::tma_load_2d_2sm(a_tile(stage), &tmX0, lead_full, ax, ay);
                        else tc::tma_load_2d_2sm(a_tile(stage), &tmA, lead_full, ax, ay);
                        const bool b1 = kw || kb < p.b_split_kb;
                        const int brow = kw ? ti.n * BN : ti.e * p.b_rows_per_expert + ti.n * BN;
                        tc::tma_load_2d_2sm(b_tile(stage), b1 ? (const void*)&tmB : (const void*)&tmB2, lead_full,
                                            kw ? ax : (b1 ? kb : kb - p.b_split_kb) * C::kBK, brow + rank * (BN / 2));
                        if constexpr (MX) {
                            // scale chunks (512 B = two 256-byte rows of tmX0 / tmX1): this CTA's A
                            // rows, and all BN rows of B (the pair MMA reads B's scales in each CTA)
                            const int akc = kw ? ax / 128 : kb;
                            const int art = kw ? ti.m : ti.a_row0 / kTileM;
                            const int bkn = kw ? p.sf_kchunks_b : p.sf_kchunks;
                            tc::tma_load_2d_2sm(sf_tile(stage), &tmX0, lead_full, 0, 2 * (art * p.sf_kchunks + akc));
#pragma unroll
                            for (int j = 0; j < C::kNChunks; ++j)
                                tc::tma_load_2d_2sm(sf_tile(stage) + 512 * (1 + j), &tmX1, lead_full, 0,
                                                    2 * ((brow / kTileM + j) * bkn + akc));
                        }
                        last_par[stage] = (int)ph;
                        if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                        continue;
                    }
                    tc::mbar_expect_tx(full_bar(stage), C::kStageBytes + C::kSfStage);
                    if constexpr (MN_MAJOR) {
                        const int krow = ti.a_row0 + kb * 64;
                        const int m0 = ti.m * kTileM;
                        tc::tma_load_2d(a_tile(stage), &tmA, full_bar(stage), m0, krow);
                        tc::tma_load_2d(a_tile(stage) + 8192, &tmA, full_bar(stage), m0 + 64, krow);
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tc::tma_load_2d(b_tile(stage) + 8192 * j, &tmB, full_bar(stage), ti.n * BN + 64 * j, krow);
                    } else {
                        // K-major: A box at (K offset, row), B box at (K offset, row); the
                        // K-major weight gradients take the expert's token range as K
                        const bool kw = p.kmajor_wgrad != 0;
                        const int ax = kw ? ti.a_row0 + kb * C::kBK : kb * C::kBK;
                        const int ay = kw ? ti.m * kTileM : ti.a_row0;
                        tc::tma_load_2d(a_tile(stage), &tmA, full_bar(stage), ax, ay);
                        const int brow = kw ? ti.n * BN : ti.e * p.b_rows_per_expert + ti.n * BN;
                        const bool b1 = kb < p.b_split_kb;
                        if (b1)
                            tc::tma_load_2d(b_tile(stage), &tmB, full_bar(stage), kw ? ax : kb * C::kBK, brow);
                        else
                            tc::tma_load_2d(b_tile(stage), &tmB2, full_bar(stage), (kb - p.b_split_kb) * C::kBK, brow);
                        if constexpr (MX) {
                            const int art = kw ? ti.m : ti.a_row0 / kTileM;
                            const int akc = kw ? ax / 128 : kb;
                            tc::bulk_load(sf_tile(stage), p.a_sf + ((int64_t)art * p.sf_kchunks + akc) * 512, 512,
                                          full_bar(stage));
                            const uint8_t* bsf = b1 ? p.b_sf : p.b_sf2;
                            const int bkc = kw ? ax / 128 : (b1 ? kb : kb - p.b_split_kb);
                            const int bkn = p.sf_kchunks_b > 0 ? p.sf_kchunks_b : p.sf_kchunks;
                            if constexpr (BN == 224) {
                                // B scales packed per 224-row tile: two chunks side by side
                                tc::bulk_load(sf_tile(stage) + 512, bsf + ((int64_t)(brow / 224) * bkn + bkc) * 1024,
                                              1024, full_bar(stage));
                            } else {
#pragma unroll
                                for (int j = 0; j < C::kNChunks; ++j) {
                                    const int brt = brow / kTileM + j;
                                    tc::bulk_load(sf_tile(stage) + 512 * (1 + j), bsf + ((int64_t)brt * bkn + bkc) * 512,
                                                  512, full_bar(stage));
                                }
                            }
                        }
                    }
                    last_par[stage] = (int)ph;
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (last_par[s] >= 0) tc::mbar_wait(full_bar(s), (uint32_t)last_par[s], st, tmo, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (pairs: the leader issues for both CTAs; the peer's warp 1 only
        // allocated the tensor memory)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_ph = 0;
            bool ok = true, issued = false;
            for (int gi = gstart; gi < gtotal && ok; gi += gstep) {
                TileInfo ti = decode(gi);
                if (ti.num_kb == 0) continue;
                if (!tc::mbar_wait(acce_bar(acc), acc_ph ^ 1u, st, tmo, kSiteMmaAccEmpty)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(acc * C::kAccStride);
                for (int kb = 0; kb < ti.num_kb; ++kb) {
                    if (!tc::mbar_wait(full_bar(stage), ph, st, tmo, kSiteMmaFull)) { ok = false; break; }
                    tc::fence_after_sync();
                    uint32_t sfa_t = 0, sfb_t = 0;
                    if constexpr (MX) {
                        sfa_t = tmem + (uint32_t)C::sf_col(stage);
                        sfb_t = sfa_t + 4;
                        if constexpr (CLN == 2) {
                            tc::tmem_cp_2sm_32x128b_warpx4(sfa_t, tc::make_sdesc(sf_tile(stage), 0, 128, tc::kLayoutNone));
#pragma unroll
                            for (int j = 0; j < C::kNChunks; ++j)
                                tc::tmem_cp_2sm_32x128b_warpx4(
                                    sfb_t + 4 * j, tc::make_sdesc(sf_tile(stage) + 512 * (1 + j), 0, 128, tc::kLayoutNone));
                        } else {
                            tc::tmem_cp_32x128b_warpx4(sfa_t, tc::make_sdesc(sf_tile(stage), 0, 128, tc::kLayoutNone));
#pragma unroll
                            for (int j = 0; j < C::kNChunks; ++j)
                                tc::tmem_cp_32x128b_warpx4(
                                    sfb_t + 4 * j, tc::make_sdesc(sf_tile(stage) + 512 * (1 + j), 0, 128, tc::kLayoutNone));
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < C::kMmasPerStage; ++kk) {
                        uint64_t ad, bd;
                        if constexpr (MN_MAJOR) {
                            ad = tc::make_sdesc(a_tile(stage) + kk * 2048, 8192, 1024, tc::kLayoutSW128);
                            bd = tc::make_sdesc(b_tile(stage) + kk * 2048, 8192, 1024, tc::kLayoutSW128);
                        } else {
                            ad = tc::make_sdesc(a_tile(stage) + kk * 32, 16, 1024, tc::kLayoutSW128);
                            bd = tc::make_sdesc(b_tile(stage) + kk * 32, 16, 1024, tc::kLayoutSW128);
                        }
                        const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (MX && CLN == 2) {
                            tc::mma_mxf8_2sm(d, ad, bd, tc::idesc_mxf8(256, BN, kk, kk), sfa_t, sfb_t, accum);
                        } else if constexpr (MX) {
                            tc::mma_mxf8(d, ad, bd, tc::idesc_mxf8(128, BN, kk, kk), sfa_t, sfb_t, accum);
                        } else if constexpr (CLN == 2) {
                            tc::mma_bf16_2sm(d, ad, bd, tc::idesc_bf16(ti.m128 ? 128 : 256, BN, MN_MAJOR, MN_MAJOR),
                                             accum);
                        } else {
                            tc::mma_bf16(d, ad, bd, tc::idesc_bf16(ti.half ? 64 : 128, BN, MN_MAJOR, MN_MAJOR), accum);
                        }
                    }
                    issued = true;
                    if constexpr (CLN == 2) tc::mma_commit_2sm_multicast(empty_bar(stage), (uint16_t)0x3);
                    else tc::mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if constexpr (CLN == 2) tc::mma_commit_2sm_multicast(accf_bar(acc), (uint16_t)0x3);
                else tc::mma_commit(accf_bar(acc));
                if (++acc == ACC_STAGES) { acc = 0; acc_ph ^= 1u; }
            }
            if (!ok && issued) {
                // every MMA issued so far must finish before tensor memory is freed
                if constexpr (CLN == 2) tc::mma_commit_2sm(drain_bar);
                else tc::mma_commit(drain_bar);
                tc::mbar_wait(drain_bar, 0, st, tmo, kSiteDrain);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;          // TMEM lane quadrant of this warp
        int acc = 0;
        uint32_t acc_ph = 0;
        for (int gi = gstart; gi < gtotal; gi += gstep) {
            TileInfo ti = decode(gi);
            // tile row owned by this thread (-1: none, in the empty lanes of an M=64 tile)
            // (an M=128 pair tile: lanes 32q.. hold rows 32(q%2).. of this CTA's 64 for the
            // tile columns (q/2)*BN/2 .. +BN/2, in tensor-memory columns 0 .. BN/2)
            const int row = ti.m128 ? 32 * (q & 1) + lane : ti.half ? (lane < 16 ? q * 16 + lane : -1) : q * 32 + lane;
            const int cbeg = ti.m128 ? (q >> 1) * (BN / 2) : 0;   // first tile column of this warp
            const int cspan = ti.m128 ? BN / 2 : BN;              // its tile columns
            const bool has_acc = ti.num_kb > 0;
            if (has_acc) {
                if (!tc::mbar_wait(accf_bar(acc), acc_ph, st, tmo, kSiteEpiAccFull)) break;
                tc::fence_after_sync();
            }
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccStride);

            if constexpr (C::kWideEpi && EPI == kEpiDense) {
                // weight gradients, 256 columns: this warp's 32-column chunks
                // eg, eg+2, eg+4, eg+6 to registers (packed to BF16), the
                // accumulator released, then each row segment written with
                // 32-byte stores (whole sectors); an expert without tokens
                // writes zeros
                const int eg = (warp - 2) >> 2;
                uint32_t w0[16], w1[16], w2[16], w3[16];
                if (has_acc) {
                    auto load_pair = [&](int c, uint32_t(&wa)[16], uint32_t(&wb)[16]) {
                        uint32_t ra[32], rb[32];
                        tc::tmem_ld_32x32b_x32(tbase + 32 * c, ra);
                        tc::tmem_ld_32x32b_x32(tbase + 32 * (c + 2), rb);
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
                    if constexpr (CLN == 2) tc::mbar_arrive_cluster(tc::mapa_shared(acce_bar(acc), 0));
                    else tc::mbar_arrive(acce_bar(acc));
                    if (++acc == ACC_STAGES) { acc = 0; acc_ph ^= 1u; }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) w0[i] = w1[i] = w2[i] = w3[i] = 0u;
                }
                const int mrow = ti.row_base + row;
                if (mrow < p.m_fixed) {
                    auto store_chunk = [&](int c, const uint32_t(&w)[16]) {
                        const int col = ti.n * BN + 32 * c;
                        __nv_bfloat16* o = col < p.split_col
                            ? static_cast<__nv_bfloat16*>(p.out0) + ((int64_t)ti.e * p.m_fixed + mrow) * p.ldo + col
                            : static_cast<__nv_bfloat16*>(p.out1) + ((int64_t)ti.e * p.m_fixed + mrow) * p.ldo +
                                  (col - p.split_col);
                        tc::stg_v8(o, w);
                        tc::stg_v8(o + 16, w + 8);
                    };
                    store_chunk(eg, w0);
                    store_chunk(eg + 2, w1);
                    store_chunk(eg + 4, w2);
                    store_chunk(eg + 6, w3);
                }
            } else if constexpr (C::kWideEpi && EPI == kEpiDSwiGLU) {
                // dgrad of h, 256 columns: this warp's 32-column chunks eg,
                // eg+2, eg+4, eg+6 of dh (fp32) to registers, the accumulator
                // released, then dG = dh U silu'(G) and dU = dh silu(G) from
                // the saved fp32 pre-activations, 8 columns at a time
                static_assert(CLN == 1, "dSwiGLU wide epilogue: single CTAs");
                const int eg = (warp - 2) >> 2;
                const int I = p.split_col;
                const int64_t prow = ti.row_base + row;
                uint32_t r[4][32];
#pragma unroll
                for (int j = 0; j < 4; ++j) tc::tmem_ld_32x32b_x32(tbase + 32 * (eg + 2 * j), r[j]);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                tc::mbar_arrive(acce_bar(acc));
                if (++acc == ACC_STAGES) { acc = 0; acc_ph ^= 1u; }
                if (ti.valid) {
                    const float* gb = static_cast<const float*>(p.gu) + prow * (int64_t)(2 * I);
                    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out0) + prow * (int64_t)(2 * I);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = ti.n * BN + 32 * (eg + 2 * j);
#pragma unroll
                        for (int h16 = 0; h16 < 2; ++h16) {
                            uint32_t dgw[8], duw[8];
#pragma unroll
                            for (int g8 = 0; g8 < 2; ++g8) {
                                const int c8 = 16 * h16 + 8 * g8;
                                uint32_t gw[8], uw[8];
                                tc::ldg_v8(gb + col + c8, gw);
                                tc::ldg_v8(gb + I + col + c8, uw);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    float dg2[2], du2[2];
#pragma unroll
                                    for (int q2 = 0; q2 < 2; ++q2) {
                                        const float G = __uint_as_float(gw[2 * i + q2]);
                                        const float U = __uint_as_float(uw[2 * i + q2]);
                                        const float dh = __uint_as_float(r[j][c8 + 2 * i + q2]);
                                        const float sg = 1.0f / (1.0f + expf(-G));
                                        dg2[q2] = dh * U * (sg * (1.0f + G * (1.0f - sg)));
                                        du2[q2] = dh * (G * sg);
                                    }
                                    dgw[4 * g8 + i] = pack_bf16x2(dg2[0], dg2[1]);
                                    duw[4 * g8 + i] = pack_bf16x2(du2[0], du2[1]);
                                }
                            }
                            tc::stg_v8(ob + col + 16 * h16, dgw);
                            tc::stg_v8(ob + I + col + 16 * h16, duw);
                        }
                    }
                }
            } else if constexpr (C::kWideEpi && EPI == kEpiScatter) {
                // this warp's 32-column chunks eg, eg+2, eg+4, eg+6 to
                // registers (packed to BF16 two at a time), accumulator
                // released, then pushed to the row's slot
                const int eg = (warp - 2) >> 2;
                int64_t dest = -1;
                const int lrow = ti.local_row0 + row;
                if (p.identity_rows > 0) {
                    if (lrow < p.identity_rows) dest = lrow;
                } else if (ti.valid && lrow < p.counts[ti.e]) {
                    dest = p.row_src[p.offsets[ti.e] + lrow];
                }
                constexpr int nch = BN / 32;
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
                if constexpr (CLN == 2) tc::mbar_arrive_cluster(tc::mapa_shared(acce_bar(acc), 0));
                else tc::mbar_arrive(acce_bar(acc));
                if (++acc == ACC_STAGES) { acc = 0; acc_ph ^= 1u; }
                if (dest >= 0) {
                    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out0) + dest * p.ldo + ti.n * BN;
                    auto store_chunk = [&](int c, const uint32_t(&w)[16]) {
                        tc::stg_v8(orow + 32 * c, w);
                        tc::stg_v8(orow + 32 * c + 16, w + 8);
                    };
                    if (eg < nch) store_chunk(eg, w0);
                    if (eg + 2 < nch) store_chunk(eg + 2, w1);
                    if (eg + 4 < nch) store_chunk(eg + 4, w2);
                    if (eg + 6 < nch) store_chunk(eg + 6, w3);
                }
            } else if constexpr (C::kWideEpi && EPI == kEpiSwiGLU) {
                // this warp's 64 h columns: gate and up pre-activations to
                // registers, accumulator released, then SwiGLU and two
                // 32-element MXFP8 blocks (scale codes 2*eg and 2*eg+1 of the
                // tile's 128-wide scale chunk)
                const int eg = (warp - 2) >> 2;
                const int I = p.split_col;
                const int64_t prow = ti.row_base + row;
                const bool live = (p.identity_rows > 0 ? (prow < p.identity_rows) : true) && ti.valid;
                uint32_t gr0[32], gr1[32], ur0[32], ur1[32];
                tc::tmem_ld_32x32b_x32(tbase + 64 * eg, gr0);
                tc::tmem_ld_32x32b_x32(tbase + 64 * eg + 32, gr1);
                tc::tmem_ld_32x32b_x32(tbase + BN / 2 + 64 * eg, ur0);
                tc::tmem_ld_32x32b_x32(tbase + BN / 2 + 64 * eg + 32, ur1);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                if constexpr (CLN == 2) tc::mbar_arrive_cluster(tc::mapa_shared(acce_bar(acc), 0));
                else tc::mbar_arrive(acce_bar(acc));
                if (++acc == ACC_STAGES) { acc = 0; acc_ph ^= 1u; }
                if (live) {
                    const int hc0 = ti.n * (BN / 2) + 64 * eg;
                    if (p.gu != nullptr) {
                        // training forward: the fp32 pre-activations for the backward's dSwiGLU
                        float* gb = static_cast<float*>(p.gu) + prow * (int64_t)(2 * I);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            tc::stg_v8(gb + hc0 + 8 * i, gr0 + 8 * i);
                            tc::stg_v8(gb + hc0 + 32 + 8 * i, gr1 + 8 * i);
                            tc::stg_v8(gb + I + hc0 + 8 * i, ur0 + 8 * i);
                            tc::stg_v8(gb + I + hc0 + 32 + 8 * i, ur1 + 8 * i);
                        }
                    }
                    uint32_t codes = 0;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        float hv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float gv = __uint_as_float(b ? gr1[i] : gr0[i]);
                            const float uv = __uint_as_float(b ? ur1[i] : ur0[i]);
                            hv[i] = silu_f(gv) * uv;
                        }
                        if (p.out1_bf16 != nullptr) {
                            // training forward: h in BF16 for the weight gradient of W_down
                            uint32_t hw[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) hw[i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
                            __nv_bfloat16* hd = static_cast<__nv_bfloat16*>(p.out1_bf16) + prow * (int64_t)I + hc0 + 32 * b;
                            tc::stg_v8(hd, hw);
                            tc::stg_v8(hd + 16, hw + 8);
                        }
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
                        const uint32_t code = e8m0_code(amax);
                        const float inv = e8m0_inv_scale(code);
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            uint32_t lo = f32x2_to_e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv);
                            uint32_t hi = f32x2_to_e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv);
                            w[i] = lo | (hi << 16);
                        }
                        tc::stg_v8(static_cast<uint8_t*>(p.out0) + prow * (int64_t)I + hc0 + 32 * b, w);
                        codes |= code << (8 * b);
                    }
                    const int64_t chunk = (prow / kTileM) * (int64_t)(I / 128) + hc0 / 128;
                    *reinterpret_cast<uint16_t*>(p.out_sf + chunk * 512 +
                                                 sf_chunk_offset((int)(prow % kTileM), 2 * eg)) = (uint16_t)codes;
                }
            } else if constexpr (EPI == kEpiSwiGLU) {
                const int I = p.split_col;
                const int64_t prow = ti.row_base + row;
                const bool live = (p.identity_rows > 0 ? (prow < p.identity_rows) : true) && ti.valid && row >= 0;
                uint32_t sfw = 0;   // MXFP8: scale codes of the current 128-wide chunk of h
#pragma unroll 1
                for (int c0 = 0; c0 < cspan / 2; c0 += 32) {
                    uint32_t gr[32], ur[32];
                    load_gate_up<BN, !MX>(tbase, c0, gr, ur);
                    const int hc = ti.n * (BN / 2) + cbeg / 2 + c0;
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float gv = __uint_as_float(gr[i]), uv = __uint_as_float(ur[i]);
                        hv[i] = silu_f(gv) * uv;
                    }
                    if (!live) continue;
                    if constexpr (MX) {
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
                        const uint32_t code = e8m0_code(amax);
                        const float inv = e8m0_inv_scale(code);
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            uint32_t lo = f32x2_to_e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv);
                            uint32_t hi = f32x2_to_e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv);
                            w[i] = lo | (hi << 16);
                        }
                        tc::stg_v8(static_cast<uint8_t*>(p.out0) + prow * (int64_t)I + hc, w);
                        // the four codes of a 128-wide chunk leave as one word
                        sfw |= code << (8 * ((hc / 32) & 3));
                        if (((hc / 32) & 3) == 3) {
                            const int64_t chunk = (prow / kTileM) * (int64_t)(I / 128) + hc / 128;
                            *reinterpret_cast<uint32_t*>(p.out_sf + chunk * 512 +
                                                         sf_chunk_offset((int)(prow % kTileM), 0)) = sfw;
                            sfw = 0;
                        }
                    } else {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out0) + prow * (int64_t)I + hc;
                        tc::stg_v8(dst, w);
                        tc::stg_v8(dst + 16, w + 8);
                    }
                    if (p.gu != nullptr) {
                        // pre-activations kept in fp32 for the backward's dSwiGLU
                        float* gb = static_cast<float*>(p.gu) + prow * (int64_t)(2 * I);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            tc::stg_v8(gb + hc + 8 * i, gr + 8 * i);
                            tc::stg_v8(gb + I + hc + 8 * i, ur + 8 * i);
                        }
                    }
                }
            } else if constexpr (EPI == kEpiScatter) {
                int64_t dest = -1;
                const int lrow = ti.local_row0 + row;
                if (row < 0) {
                    // an empty lane of an M=64 tile
                } else if (p.identity_rows > 0) {
                    if (lrow < p.identity_rows) dest = lrow;
                } else if (lrow < p.counts[ti.e]) {
                    dest = p.row_src[p.offsets[ti.e] + lrow];
                }
#pragma unroll 1
                for (int c0 = 0; c0 < cspan; c0 += 32) {
                    uint32_t r[32];
                    tc::tmem_ld_32x32b_x32(tbase + c0, r);
                    tc::tmem_ld_wait();
                    if (dest < 0) continue;
                    const int col = ti.n * BN + cbeg + c0;
                    if (p.out_f32) {
                        float* dst = static_cast<float*>(p.out0) + dest * p.ldo + col;
#pragma unroll
                        for (int i = 0; i < 4; ++i) tc::stg_v8(dst + 8 * i, r + 8 * i);
                    } else {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out0) + dest * p.ldo + col;
                        tc::stg_v8(dst, w);
                        tc::stg_v8(dst + 16, w + 8);
                    }
                }
            } else if constexpr (EPI == kEpiDSwiGLU) {
                const int I = p.split_col;
                const int64_t prow = ti.row_base + row;
                const float* gb = static_cast<const float*>(p.gu) + prow * (int64_t)(2 * I);
                __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out0) + prow * (int64_t)(2 * I);
#pragma unroll 1
                for (int c0 = 0; c0 < cspan && ti.valid; c0 += 32) {   // pairs: no rows outside the expert
                    uint32_t r[32];
                    tc::tmem_ld_32x32b_x32(tbase + c0, r);
                    tc::tmem_ld_wait();
                    const int col = ti.n * BN + cbeg + c0;
                    uint32_t dgw[16], duw[16];
                    uint32_t gw32[32], uw32[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        tc::ldg_v8(gb + col + 8 * i, gw32 + 8 * i);
                        tc::ldg_v8(gb + I + col + 8 * i, uw32 + 8 * i);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float Gv[4] = {__uint_as_float(gw32[4 * i]), __uint_as_float(gw32[4 * i + 1]),
                                             __uint_as_float(gw32[4 * i + 2]), __uint_as_float(gw32[4 * i + 3])};
                        const float Uv[4] = {__uint_as_float(uw32[4 * i]), __uint_as_float(uw32[4 * i + 1]),
                                             __uint_as_float(uw32[4 * i + 2]), __uint_as_float(uw32[4 * i + 3])};
                        float dg4[4], du4[4];
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            const float G = Gv[q2], U = Uv[q2];
                            const float dh = __uint_as_float(r[4 * i + q2]);
                            const float sg = 1.0f / (1.0f + expf(-G));
                            dg4[q2] = dh * U * (sg * (1.0f + G * (1.0f - sg)));
                            du4[q2] = dh * (G * sg);
                        }
                        dgw[2 * i] = pack_bf16x2(dg4[0], dg4[1]);
                        dgw[2 * i + 1] = pack_bf16x2(dg4[2], dg4[3]);
                        duw[2 * i] = pack_bf16x2(du4[0], du4[1]);
                        duw[2 * i + 1] = pack_bf16x2(du4[2], du4[3]);
                    }
                    tc::stg_v8(ob + col, dgw);
                    tc::stg_v8(ob + col + 16, dgw + 8);
                    tc::stg_v8(ob + I + col, duw);
                    tc::stg_v8(ob + I + col + 16, duw + 8);
                }
            } else {  // kEpiDense
                // 32 x 32 BF16 blocks through shared memory, written by TMA
                // stores (rows past m_fixed are clipped by the map's extent);
                // a warp's two staging blocks alternate, and a block is
                // rewritten only once the store issued from it two chunks
                // earlier has read it
                const int ew = warp - 2;
                const int mrow0 = ti.row_base + q * 32;   // first row of this warp's 32, within the expert
                const int rot = (lane >> 1) & 3;           // store order: 4-way bank conflicts at most
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t r[32];
                    if (has_acc) {
                        tc::tmem_ld_32x32b_x32(tbase + c0, r);
                        tc::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0u;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    const uint32_t buf = smem_base + C::kEpiStageOffset + (uint32_t)(ew * 2 + ((c0 >> 5) & 1)) * 2048u;
                    if (lane == 0) tc::bulk_wait_read<1>();
                    __syncwarp();
                    const uint32_t rowp = buf + (uint32_t)lane * 64u;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int j = (t + rot) & 3;
                        const uint32_t a0 = j == 0 ? w[0] : j == 1 ? w[4] : j == 2 ? w[8] : w[12];
                        const uint32_t a1 = j == 0 ? w[1] : j == 1 ? w[5] : j == 2 ? w[9] : w[13];
                        const uint32_t a2 = j == 0 ? w[2] : j == 1 ? w[6] : j == 2 ? w[10] : w[14];
                        const uint32_t a3 = j == 0 ? w[3] : j == 1 ? w[7] : j == 2 ? w[11] : w[15];
                        tc::st_shared_v4(rowp + (uint32_t)j * 16u, a0, a1, a2, a3);
                    }
                    tc::fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0 && mrow0 < p.m_fixed) {
                        const int col = ti.n * BN + c0;
                        if (col < p.split_col) tc::tma_store_3d(&tmX0, buf, col, mrow0, ti.e);
                        else tc::tma_store_3d(&tmX1, buf, col - p.split_col, mrow0, ti.e);
                        tc::bulk_commit();
                    }
                }
            }
            if (has_acc && !C::kWideEpi) {
                tc::fence_before_sync();
                if constexpr (CLN == 2) tc::mbar_arrive_cluster(tc::mapa_shared(acce_bar(acc), 0));
                else tc::mbar_arrive(acce_bar(acc));
                if (++acc == ACC_STAGES) { acc = 0; acc_ph ^= 1u; }
            }
        }
        if constexpr (EPI == kEpiDense) {
            if (lane == 0) tc::bulk_wait<0>();   // stores done with shared memory (and written) before exit
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if constexpr (CLN == 2) {
        tc::cluster_sync();   // no CTA frees or leaves while its peer may still use the pair's resources
        if (warp == 1) tc::tmem_dealloc_2sm(tmem, C::kTmemCols);
    } else {
        if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace mok
