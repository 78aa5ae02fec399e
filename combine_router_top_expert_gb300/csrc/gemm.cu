// gemm.cu - host launchers of the grouped tcgen05 GEMM: tensor maps, tile
// shapes per call site, persistent grid sizing.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <map>
#include <set>
#include <utility>

#include "gemm.cuh"
#include "gemm_swap.cuh"
#include "moves.cuh"

namespace mok {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D row-major [rows, cols] tensor; box = box_cols x box_rows with a
// 128-byte swizzle (box_cols * elem_bytes == 128). Out-of-range rows read 0.
bool make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int elem_bytes, int box_cols,
               int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * elem_bytes)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Scale chunks as a 2-D byte tensor: a 512-byte chunk is two 256-byte rows
// (no swizzle); the pair kernels load one chunk per TMA box of 256 x 2.
bool make_tmap_chunks(CUtensorMap* m, const void* base, int64_t chunks) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {256, (cuuint64_t)(2 * chunks)};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, 2};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Dense-epilogue output [E, rows, width] BF16 with row pitch ld elements,
// stored in 32 x 32 x 1 boxes from unswizzled shared memory.
bool make_tmap_out3d(CUtensorMap* m, void* base, int E, int64_t rows, int64_t width, int64_t ld) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(rows * ld * 2)};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

// 2-D row-major [rows, cols] tensor read in unswizzled boxes of box_cols x
// box_rows (box_cols * elem_bytes a multiple of 16); rows and columns out of
// range read 0.
bool make_tmap_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int elem_bytes, int box_cols,
                    int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * elem_bytes)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// Clusters of two CTAs that can be resident at once for kernel `kern` with
// launch configuration `cfg` (dynamic shared memory and block size fixed per
// kernel), queried once per device and kernel: the occupancy query is a
// driver call that measured slow when another process polled the GPU.
int max_pair_clusters(const void* kern, cudaLaunchConfig_t cfg, int num_sms) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(dev, kern);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return std::min(it->second, num_sms / 2);
    }
    int dev_sms = 0;
    cudaDeviceGetAttribute(&dev_sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(2 * (dev_sms / 2));
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        clusters = dev_sms / 2;
    }
    {
        std::lock_guard<std::mutex> g(mu);
        cache[key] = clusters;
    }
    return std::min(clusters, num_sms / 2);
}

template <int BN, bool MX, bool MN, int EPI, int S, int ACC, int CLN = 1>
cudaError_t run(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const CUtensorMap& sa,
                const CUtensorMap& sb, const GemmParams& p, int64_t tiles_ub, int num_sms, cudaStream_t s) {
    using C = GemmCfg<BN, MX, MN, EPI, S, ACC, CLN>;
    auto kern = grouped_gemm_kernel<BN, MX, MN, EPI, S, ACC, CLN>;
    ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = s;
    int grid;
    if constexpr (CLN == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // persistent: as many CTA pairs as can be resident at once
        const int clusters = max_pair_clusters(reinterpret_cast<const void*>(kern), cfg, num_sms);
        grid = 2 * (int)std::min<int64_t>((tiles_ub + 1) / 2, clusters);
    } else {
        grid = (int)std::min<int64_t>(tiles_ub, num_sms);
    }
    if (grid < 1) return cudaSuccess;
    cfg.gridDim = dim3(grid);
    // the prologue (barriers, tensor memory, tensor-map prefetch) may overlap
    // the end of the kernel before on the stream (the kernel waits before it
    // reads anything that kernel writes)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs += 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, b, b2, sa, sb, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int BN, bool MX, bool MN, int EPI, int S, int ACC, int CLN = 1>
cudaError_t run(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const GemmParams& p,
                int64_t tiles_ub, int num_sms, cudaStream_t s) {
    return run<BN, MX, MN, EPI, S, ACC, CLN>(a, b, b2, b, b, p, tiles_ub, num_sms, s);
}

// Swapped-operand pair kernel: persistent clusters of two CTAs.
template <int EPI, int S>
cudaError_t run_swap(const CUtensorMap& w, const CUtensorMap& x64, const CUtensorMap& x32, const CUtensorMap& x16,
                     const SwapParams& p, int num_sms, cudaStream_t s) {
    using C = SwapCfg<S>;
    auto kern = grouped_gemm_swap_kernel<EPI, S>;
    ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = s;
    const int clusters = max_pair_clusters(reinterpret_cast<const void*>(kern), cfg, num_sms);
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(2 * clusters);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, w, x64, x32, x16, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

SwapParams swap_params(const GemmCommon& c, int policy) {
    SwapParams p{};
    p.status = c.status;
    p.timeout_ns = c.timeout_ns;
    p.tile_policy = policy;
    p.l2_prefetch = c.l2_prefetch;
    return p;
}

GemmParams base_params(const GemmCommon& c) {
    GemmParams p{};
    p.b_split_kb = 1 << 30;
    p.status = c.status;
    p.timeout_ns = c.timeout_ns;
    return p;
}

// Upper bound on 128-row tiles of a grouped layout with `rows` routed rows.
int64_t mtiles_ub(int64_t rows, int E) { return (rows + kTileM - 1) / kTileM + E; }

}  // namespace

void ensure_smem_attr(const void* func, int bytes) {
    // The limit is raised whenever a launch needs more than any earlier one
    // (kernels whose shared memory depends on the problem, e.g. the router).
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> limit;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> g(mu);
    auto key = std::make_pair(dev, func);
    auto it = limit.find(key);
    if (it != limit.end() && it->second >= bytes) return;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess)
        limit[key] = bytes;
}

cudaError_t gemm_gateup(bool mx, const void* A, const uint8_t* A_sf, const void* Bgu, const uint8_t* Bgu_sf,
                        int E, int H, int I, const int32_t* counts, int identity_rows, int64_t a_rows, void* h,
                        uint8_t* h_sf, void* gu_save, const GemmCommon& c, cudaStream_t s, void* h_bf16) {
    const int BN = (2 * I) >= 256 ? 256 : 128;
    const int eb = mx ? 1 : 2;
    const int bk = 128 / eb;
    GemmParams p = base_params(c);
    p.E = identity_rows > 0 ? 1 : E;
    p.counts = counts;
    p.identity_rows = identity_rows;
    p.num_kb = H / bk;
    p.b_rows_per_expert = 2 * I;
    p.out0 = h;
    p.out_sf = h_sf;
    p.gu = gu_save;
    p.out1_bf16 = h_bf16;
    p.split_col = I;
    p.a_sf = A_sf;
    p.b_sf = Bgu_sf;
    p.sf_kchunks = H / 128;
    p.n_tiles = 2 * I / BN;
    // 2-SM pairs (256-wide, grouped rows): each CTA loads half of B
    const bool cl = c.cluster == 2 && BN == 256 && (identity_rows == 0 || !mx);
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A, a_rows, H, eb, bk, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, Bgu, (int64_t)p.E * 2 * I, H, eb, bk, cl ? BN / 2 : BN)) return cudaErrorInvalidValue;
    const int64_t mt = identity_rows > 0 ? (identity_rows + kTileM - 1) / kTileM : mtiles_ub(a_rows, E);
    const int64_t tub = mt * p.n_tiles;
    if (mx) {
        // MXFP8: 256-wide tiles (gate 128 | up 128) with one accumulator (the
        // block scales need the rest of tensor memory); I is a multiple of 128
        if (BN != 256) return cudaErrorInvalidValue;
        if (cl) {
            CUtensorMap tsa, tsb;
            if (!make_tmap_chunks(&tsa, A_sf, (a_rows / kTileM) * (H / 128)) ||
                !make_tmap_chunks(&tsb, Bgu_sf, (int64_t)p.E * 2 * I / kTileM * (H / 128)))
                return cudaErrorInvalidValue;
            return run<256, true, false, kEpiSwiGLU, 6, 1, 2>(ta, tb, tb, tsa, tsb, p, tub, c.num_sms, s);
        }
        return run<256, true, false, kEpiSwiGLU, 4, 1>(ta, tb, tb, p, tub, c.num_sms, s);
    }
    if (BN == 256) {
        if (cl) {
            // the odd last 128-row tile of an expert runs as an M=128 pair: 64-row A boxes
            CUtensorMap ta64;
            if (!make_tmap(&ta64, A, a_rows, H, 2, 64, 64)) return cudaErrorInvalidValue;
            return run<256, false, false, kEpiSwiGLU, 6, 2, 2>(ta, tb, tb, ta64, ta64, p, tub, c.num_sms, s);
        }
        return run<256, false, false, kEpiSwiGLU, 4, 2>(ta, tb, tb, p, tub, c.num_sms, s);
    }
    return run<128, false, false, kEpiSwiGLU, 6, 2>(ta, tb, tb, p, tub, c.num_sms, s);
}

cudaError_t gemm_down(bool mx, const void* h, const uint8_t* h_sf, const void* Bdn, const uint8_t* Bdn_sf, int E,
                      int H, int I, const int32_t* counts, const int32_t* offsets, const int32_t* row_src,
                      int identity_rows, int64_t a_rows, void* out, const GemmCommon& c, cudaStream_t s) {
    const int eb = mx ? 1 : 2;
    const int bk = 128 / eb;
    GemmParams p = base_params(c);
    p.E = identity_rows > 0 ? 1 : E;
    p.counts = counts;
    p.offsets = offsets;
    p.row_src = row_src;
    p.identity_rows = identity_rows;
    p.num_kb = I / bk;
    p.b_rows_per_expert = H;
    p.out0 = out;
    p.ldo = H;
    p.out_f32 = identity_rows > 0 ? 1 : 0;
    p.a_sf = h_sf;
    p.b_sf = Bdn_sf;
    p.sf_kchunks = I / 128;
    // MXFP8: 256-wide tiles when H allows (one accumulator, 8 epilogue warps
    // that release it before their stores), else 224 (double-buffered
    // accumulator with the scales in the tensor-memory gaps), else 128;
    // BF16: 256 or 128
    const int BN = down_tile_n(H, mx);
    p.n_tiles = H / BN;
    const bool cl = c.cluster == 2 && !mx && BN == 256;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, h, a_rows, I, eb, bk, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, Bdn, (int64_t)p.E * H, I, eb, bk, cl ? BN / 2 : BN)) return cudaErrorInvalidValue;
    const int64_t mt = identity_rows > 0 ? (identity_rows + kTileM - 1) / kTileM : mtiles_ub(a_rows, E);
    const int64_t tub = mt * p.n_tiles;
    if (mx) {
        if (BN == 256) return run<256, true, false, kEpiScatter, 4, 1>(ta, tb, tb, p, tub, c.num_sms, s);
        if (BN == 224) return run<224, true, false, kEpiScatter, 4, 2>(ta, tb, tb, p, tub, c.num_sms, s);
        return run<128, true, false, kEpiScatter, 6, 2>(ta, tb, tb, p, tub, c.num_sms, s);
    }
    if (BN == 256) {
        if (cl) {
            CUtensorMap ta64;
            if (!make_tmap(&ta64, h, a_rows, I, 2, 64, 64)) return cudaErrorInvalidValue;
            return run<256, false, false, kEpiScatter, 6, 2, 2>(ta, tb, tb, ta64, ta64, p, tub, c.num_sms, s);
        }
        return run<256, false, false, kEpiScatter, 4, 2>(ta, tb, tb, p, tub, c.num_sms, s);
    }
    return run<128, false, false, kEpiScatter, 6, 2>(ta, tb, tb, p, tub, c.num_sms, s);
}

bool swap_supported(int H, int I) { return I % 128 == 0 && H % 256 == 0 && H % 64 == 0; }

cudaError_t gemm_gateup_swap(const void* A, const void* Bgu, int E, int H, int I, const int32_t* counts,
                             int64_t a_rows, void* h, int policy, const GemmCommon& c, cudaStream_t s) {
    if (!swap_supported(H, I)) return cudaErrorInvalidValue;
    SwapParams p = swap_params(c, policy);
    p.E = E;
    p.num_kb = H / 64;
    p.m_tiles = 2 * I / 256;
    p.w_rows_per_expert = 2 * I;
    p.counts = counts;
    p.out = h;
    p.ldo = I;
    CUtensorMap tw, tx64, tx32, tx16;
    if (!make_tmap(&tw, Bgu, (int64_t)E * 2 * I, H, 2, 64, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tx64, A, a_rows, H, 2, 64, 64) || !make_tmap(&tx32, A, a_rows, H, 2, 64, 32) ||
        !make_tmap(&tx16, A, a_rows, H, 2, 64, 16))
        return cudaErrorInvalidValue;
    return run_swap<kSwapSwiGLU, 6>(tw, tx64, tx32, tx16, p, c.num_sms, s);
}

cudaError_t gemm_down_swap(const void* h, const void* Bdn, int E, int H, int I, const int32_t* counts,
                           const int32_t* offsets, const int32_t* row_src, int64_t a_rows, void* out, int policy,
                           const GemmCommon& c, cudaStream_t s) {
    if (!swap_supported(H, I)) return cudaErrorInvalidValue;
    SwapParams p = swap_params(c, policy);
    p.E = E;
    p.num_kb = I / 64;
    p.m_tiles = H / 256;
    p.w_rows_per_expert = H;
    p.counts = counts;
    p.offsets = offsets;
    p.row_src = row_src;
    p.out = out;
    p.ldo = H;
    CUtensorMap tw, tx64, tx32, tx16;
    if (!make_tmap(&tw, Bdn, (int64_t)E * H, I, 2, 64, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tx64, h, a_rows, I, 2, 64, 64) || !make_tmap(&tx32, h, a_rows, I, 2, 64, 32) ||
        !make_tmap(&tx16, h, a_rows, I, 2, 64, 16))
        return cudaErrorInvalidValue;
    return run_swap<kSwapScatter, 6>(tw, tx64, tx32, tx16, p, c.num_sms, s);
}

cudaError_t gemm_dgrad_h(const void* dy, const void* W_down, int E, int H, int I, const int32_t* counts,
                         int64_t a_rows, const void* gu, void* dgu, const GemmCommon& c, cudaStream_t s) {
    GemmParams p = base_params(c);
    p.E = E;
    p.counts = counts;
    p.num_kb = H / 64;
    p.b_rows_per_expert = I;
    p.out0 = dgu;
    p.gu = const_cast<void*>(gu);
    p.split_col = I;
    const int BN = I % 256 == 0 ? 256 : (I % 128 == 0 ? 128 : 64);
    p.n_tiles = I / BN;
    const bool cl = c.cluster == 2 && BN == 256;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, dy, a_rows, H, 2, 64, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, W_down, (int64_t)E * I, H, 2, 64, cl ? BN / 2 : BN)) return cudaErrorInvalidValue;
    const int64_t tub = mtiles_ub(a_rows, E) * p.n_tiles;
    if (cl) {
        CUtensorMap ta64;
        if (!make_tmap(&ta64, dy, a_rows, H, 2, 64, 64)) return cudaErrorInvalidValue;
        return run<256, false, false, kEpiDSwiGLU, 6, 2, 2>(ta, tb, tb, ta64, ta64, p, tub, c.num_sms, s);
    }
    if (BN == 256) return run<256, false, false, kEpiDSwiGLU, 4, 2>(ta, tb, tb, p, tub, c.num_sms, s);
    if (BN == 128) return run<128, false, false, kEpiDSwiGLU, 6, 2>(ta, tb, tb, p, tub, c.num_sms, s);
    return run<64, false, false, kEpiDSwiGLU, 8, 2>(ta, tb, tb, p, tub, c.num_sms, s);
}

cudaError_t gemm_dgrad_a(const void* dgu, const void* W_gate, const void* W_up, int E, int H, int I,
                         const int32_t* counts, const int32_t* offsets, const int32_t* row_src, int64_t a_rows,
                         void* da, const GemmCommon& c, cudaStream_t s) {
    GemmParams p = base_params(c);
    p.E = E;
    p.counts = counts;
    p.offsets = offsets;
    p.row_src = row_src;
    p.num_kb = 2 * I / 64;
    p.b_split_kb = I / 64;
    p.b_rows_per_expert = H;
    p.out0 = da;
    p.ldo = H;
    const int BN = H % 256 == 0 ? 256 : 128;
    p.n_tiles = H / BN;
    const bool cl = c.cluster == 2 && BN == 256;
    CUtensorMap ta, tb, tb2;
    if (!make_tmap(&ta, dgu, a_rows, 2 * I, 2, 64, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, W_gate, (int64_t)E * H, I, 2, 64, cl ? BN / 2 : BN)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb2, W_up, (int64_t)E * H, I, 2, 64, cl ? BN / 2 : BN)) return cudaErrorInvalidValue;
    const int64_t tub = mtiles_ub(a_rows, E) * p.n_tiles;
    if (cl) {
        CUtensorMap ta64;
        if (!make_tmap(&ta64, dgu, a_rows, 2 * I, 2, 64, 64)) return cudaErrorInvalidValue;
        return run<256, false, false, kEpiScatter, 6, 2, 2>(ta, tb, tb2, ta64, ta64, p, tub, c.num_sms, s);
    }
    if (BN == 256) return run<256, false, false, kEpiScatter, 4, 2>(ta, tb, tb2, p, tub, c.num_sms, s);
    return run<128, false, false, kEpiScatter, 6, 2>(ta, tb, tb2, p, tub, c.num_sms, s);
}

cudaError_t gemm_dgrad_h_mx(const void* dy_q, const uint8_t* dy_sf, const void* Wd_q, const uint8_t* Wd_sf, int E,
                            int H, int I, const int32_t* counts, int64_t a_rows, const void* gu, void* dgu,
                            const GemmCommon& c, cudaStream_t s) {
    if (H % 128 || I % 128) return cudaErrorInvalidValue;
    GemmParams p = base_params(c);
    p.E = E;
    p.counts = counts;
    p.num_kb = H / 128;
    p.b_rows_per_expert = I;
    p.out0 = dgu;
    p.gu = const_cast<void*>(gu);
    p.split_col = I;
    p.a_sf = dy_sf;
    p.b_sf = Wd_sf;
    p.sf_kchunks = H / 128;
    // 256-wide tiles (one accumulator, 8 epilogue warps holding dh in
    // registers) load a third less per FLOP than 128-wide ones
    const int BN = I % 256 == 0 ? 256 : 128;
    p.n_tiles = I / BN;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, dy_q, a_rows, H, 1, 128, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, Wd_q, (int64_t)E * I, H, 1, 128, BN)) return cudaErrorInvalidValue;
    const int64_t tub = mtiles_ub(a_rows, E) * p.n_tiles;
    if (BN == 256) return run<256, true, false, kEpiDSwiGLU, 4, 1>(ta, tb, tb, p, tub, c.num_sms, s);
    return run<128, true, false, kEpiDSwiGLU, 6, 2>(ta, tb, tb, p, tub, c.num_sms, s);
}

cudaError_t gemm_dgrad_a_mx(const void* dgu_q, const uint8_t* dgu_sf, const void* Wg_q, const uint8_t* Wg_sf,
                            const void* Wu_q, const uint8_t* Wu_sf, int E, int H, int I, const int32_t* counts,
                            const int32_t* offsets, const int32_t* row_src, int64_t a_rows, void* da,
                            const GemmCommon& c, cudaStream_t s) {
    if (H % 128 || I % 128) return cudaErrorInvalidValue;
    GemmParams p = base_params(c);
    p.E = E;
    p.counts = counts;
    p.offsets = offsets;
    p.row_src = row_src;
    p.num_kb = 2 * I / 128;
    p.b_split_kb = I / 128;
    p.b_rows_per_expert = H;
    p.out0 = da;
    p.ldo = H;
    p.a_sf = dgu_sf;
    p.b_sf = Wg_sf;
    p.b_sf2 = Wu_sf;
    p.sf_kchunks = 2 * I / 128;
    p.sf_kchunks_b = I / 128;
    const int BN = H % 256 == 0 ? 256 : 128;
    p.n_tiles = H / BN;
    CUtensorMap ta, tb, tb2;
    if (!make_tmap(&ta, dgu_q, a_rows, 2 * I, 1, 128, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, Wg_q, (int64_t)E * H, I, 1, 128, BN)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb2, Wu_q, (int64_t)E * H, I, 1, 128, BN)) return cudaErrorInvalidValue;
    const int64_t tub = mtiles_ub(a_rows, E) * p.n_tiles;
    if (BN == 256) return run<256, true, false, kEpiScatter, 4, 1>(ta, tb, tb2, p, tub, c.num_sms, s);
    return run<128, true, false, kEpiScatter, 6, 2>(ta, tb, tb2, p, tub, c.num_sms, s);
}

cudaError_t gemm_wgrad_mx(const void* AT_q, const uint8_t* AT_sf, int M, const void* BT_q, const uint8_t* BT_sf,
                          int N, int E, const int32_t* counts, int64_t rows_pad, void* out0, void* out1,
                          int split_col, const GemmCommon& c, cudaStream_t s) {
    if (M % 128 || N % 128 || rows_pad % 128) return cudaErrorInvalidValue;
    GemmParams p = base_params(c);
    p.E = E;
    p.counts = counts;
    p.m_fixed = M;
    p.kmajor_wgrad = 1;
    p.out0 = out0;
    p.out1 = out1;
    p.split_col = split_col;
    p.ldo = split_col < N ? split_col : N;
    p.a_sf = AT_sf;
    p.b_sf = BT_sf;
    p.sf_kchunks = (int)(rows_pad / 128);
    p.sf_kchunks_b = (int)(rows_pad / 128);
    // 256-wide tiles (one accumulator, 8 epilogue warps storing 32-byte row
    // segments) halve the A bytes loaded per FLOP against 128-wide ones; they
    // need 32-byte aligned outputs
    const bool wide = N % 256 == 0 && (reinterpret_cast<uintptr_t>(out0) & 31) == 0 &&
                      (split_col >= N || (reinterpret_cast<uintptr_t>(out1) & 31) == 0);
    const int BN = wide ? 256 : 128;
    // 2-SM pairs over two 128-row M tiles: each CTA loads its 128 weight rows
    // and half of the 256 B rows per K block (a third less per FLOP)
    const bool pair = wide && M % 256 == 0;
    p.n_tiles = N / BN;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, AT_q, M, rows_pad, 1, 128, 128)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, BT_q, N, rows_pad, 1, 128, pair ? BN / 2 : BN)) return cudaErrorInvalidValue;
    if (pair) {
        CUtensorMap tsa, tsb;
        if (!make_tmap_chunks(&tsa, AT_sf, (int64_t)(M / kTileM) * p.sf_kchunks) ||
            !make_tmap_chunks(&tsb, BT_sf, (int64_t)(N / kTileM) * p.sf_kchunks_b))
            return cudaErrorInvalidValue;
        const int64_t tub = (int64_t)E * (M / kTileM) * p.n_tiles;   // in 128-row tiles, two per pair
        return run<256, true, false, kEpiDense, 6, 1, 2>(ta, tb, tb, tsa, tsb, p, tub, c.num_sms, s);
    }
    CUtensorMap to0, to1;
    if (!make_tmap_out3d(&to0, out0, E, M, p.ldo, p.ldo)) return cudaErrorInvalidValue;
    if (split_col < N) {
        if (!out1 || !make_tmap_out3d(&to1, out1, E, M, N - split_col, p.ldo)) return cudaErrorInvalidValue;
    } else {
        to1 = to0;
    }
    const int64_t tub = (int64_t)E * (M / kTileM) * p.n_tiles;
    if (wide) return run<256, true, false, kEpiDense, 4, 1>(ta, tb, tb, to0, to1, p, tub, c.num_sms, s);
    return run<128, true, false, kEpiDense, 6, 2>(ta, tb, tb, to0, to1, p, tub, c.num_sms, s);
}

cudaError_t gemm_wgrad(const void* Aact, int M, const void* B, int N, int E, const int32_t* counts, int64_t a_rows,
                       void* out0, void* out1, int split_col, const GemmCommon& c, cudaStream_t s) {
    GemmParams p = base_params(c);
    p.E = E;
    p.counts = counts;
    p.m_fixed = M;
    p.out0 = out0;
    p.out1 = out1;
    p.split_col = split_col;
    p.ldo = split_col < N ? split_col : N;
    const int BN = N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64);
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, Aact, a_rows, M, 2, 64, 64)) return cudaErrorInvalidValue;
    if (!make_tmap(&tb, B, a_rows, N, 2, 64, 64)) return cudaErrorInvalidValue;
    p.n_tiles = N / BN;
    // outputs: out0 holds columns [0, min(split, N)), out1 (if any) [split, N)
    CUtensorMap to0, to1;
    if (!make_tmap_out3d(&to0, out0, E, M, p.ldo, p.ldo)) return cudaErrorInvalidValue;
    if (split_col < N) {
        if (!out1 || !make_tmap_out3d(&to1, out1, E, M, N - split_col, p.ldo)) return cudaErrorInvalidValue;
    } else {
        to1 = to0;
    }
    const int64_t tub = (int64_t)E * ((M + kTileM - 1) / kTileM) * p.n_tiles;
    // 2-SM pairs over two 128-row weight tiles (each CTA: its 128 weight rows,
    // half of the 256 columns; 32 KB per K block, 6 stages)
    if (BN == 256 && c.cluster == 2 && M % 256 == 0)
        return run<256, false, true, kEpiDense, 6, 2, 2>(ta, tb, tb, to0, to1, p, tub, c.num_sms, s);
    if (BN == 256) return run<256, false, true, kEpiDense, 4, 2>(ta, tb, tb, to0, to1, p, tub, c.num_sms, s);
    if (BN == 128) return run<128, false, true, kEpiDense, 6, 2>(ta, tb, tb, to0, to1, p, tub, c.num_sms, s);
    return run<64, false, true, kEpiDense, 8, 2>(ta, tb, tb, to0, to1, p, tub, c.num_sms, s);
}

}  // namespace mok
