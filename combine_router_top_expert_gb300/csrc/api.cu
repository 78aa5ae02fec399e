// api.cu - the C ABI declared in include/mok.h.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "moves.cuh"
#include "plan.cuh"

using namespace mok;

namespace {

constexpr int kDefaultTimeoutMs = 4000;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Gate/up rows interleaved per this many rows in the packed weights. BF16:
// 16, so any 32 consecutive packed rows hold the gate and up rows of the same
// 16 features (one TMEM lane quadrant of a tile whose rows are weight rows
// sees both). MXFP8: half the 256-wide N-tile of the gate/up GEMM.
int gu_interleave(int I, int dtype) {
    if (dtype == MOK_BF16) return 16;
    return 2 * I >= 256 ? 128 : 64;
}

bool dims_ok(int E, int H, int I, int dtype) {
    if (E < 1 || E > kMaxE || H <= 0 || I <= 0) return false;
    if (H % 128 || H > 65536) return false;
    if (dtype == MOK_BF16) return I == 64 || I % 128 == 0;
    if (dtype == MOK_MXFP8) return I % 128 == 0;
    return false;
}

bool problem_ok(const mok_problem* p) {
    if (!p) return false;
    if (p->T < 0 || p->k < 1 || p->k > p->E) return false;
    if (!dims_ok(p->E, p->H, p->I, p->dtype)) return false;
    if (p->I_shared < 0 || (p->I_shared > 0 && !(p->I_shared == 64 || p->I_shared % 128 == 0))) return false;
    if ((int64_t)p->T * p->k >= (int64_t)1 << 30) return false;
    return true;
}

struct PackedLayout {
    size_t gu, gu_sf, dn, dn_sf, total;
};

PackedLayout packed_layout(int E, int H, int I, int dtype) {
    PackedLayout L{};
    const int64_t eb = dtype == MOK_MXFP8 ? 1 : 2;
    size_t o = 0;
    L.gu = o; o += align_up((int64_t)E * 2 * I * H * eb, 1024);
    L.gu_sf = o; if (dtype == MOK_MXFP8) o += align_up((int64_t)E * 2 * I * H / 32, 1024);
    L.dn = o; o += align_up((int64_t)E * H * I * eb, 1024);
    L.dn_sf = o;
    if (dtype == MOK_MXFP8) {
        const int tn = down_tile_n(H, true);   // scales per tile of tn rows, whole 512-byte chunks
        o += align_up((int64_t)E * (H / tn) * ((tn + 127) / 128) * (I / 128) * 512, 1024);
    }
    L.total = o;
    return L;
}

// The MXFP8 backward's weight copies: W_down as [E*I, H] blocked along H,
// W_gate and W_up as [E*H, I] blocked along I (codes, then chunk-ordered
// scales).
struct PackedBwdLayout {
    size_t wd, wdsf, wg, wgsf, wu, wusf, total;
};

PackedBwdLayout packed_bwd_layout(int E, int H, int I) {
    PackedBwdLayout L{};
    const int64_t n = (int64_t)E * H * I;
    size_t o = 0;
    L.wd = o; o += align_up(n, 1024);
    L.wdsf = o; o += align_up(n / 32, 1024);
    L.wg = o; o += align_up(n, 1024);
    L.wgsf = o; o += align_up(n / 32, 1024);
    L.wu = o; o += align_up(n, 1024);
    L.wusf = o; o += align_up(n / 32, 1024);
    L.total = o;
    return L;
}

cudaError_t pack_bwd(const void* Wg, const void* Wu, const void* Wd, int E, int H, int I, char* b, cudaStream_t s) {
    PackedBwdLayout L = packed_bwd_layout(E, H, I);
    cudaError_t e = launch_quantize_rows_tiled(Wd, (int64_t)E * I, H, b + L.wd, b + L.wdsf, s);
    if (e == cudaSuccess) e = launch_quantize_rows_tiled(Wg, (int64_t)E * H, I, b + L.wg, b + L.wgsf, s);
    if (e == cudaSuccess) e = launch_quantize_rows_tiled(Wu, (int64_t)E * H, I, b + L.wu, b + L.wusf, s);
    return e;
}

// Forward buffers. When `saved` is given (BF16 training), A, GU, h and the
// partials live there so the backward can read them.
struct FwdLayout {
    size_t A, A_sf, h, h_sf, partials, xq, xsf, shared, hs, total;   // workspace offsets
    size_t sA, sGU, sh, spart, saved_total;                  // saved offsets
};

// Rows of the padded layout rounded up to whole 128-row tiles: buffers the
// MXFP8 tile-order and column quantisers read or write cover whole tiles.
int64_t rows_tiles(const mok_problem* p) { return align_up(padded_rows_max(p->T, p->E, p->k), kTileM); }

FwdLayout fwd_layout(const mok_problem* p, bool training) {
    FwdLayout L{};
    const int64_t rows = rows_tiles(p);
    const bool mx = p->dtype == MOK_MXFP8;
    const int64_t eb = mx ? 1 : 2;
    size_t o = kStatusBytes;
    // MXFP8 training keeps the BF16 rows and h in `saved` and the GEMMs' MXFP8
    // copies here
    if (!training || mx) { L.A = o; o += align_up(rows * p->H * eb, 1024); }
    L.A_sf = o; if (p->dtype == MOK_MXFP8) o += align_up(rows * p->H / 32, 1024);
    if (!training || mx) { L.h = o; o += align_up(rows * p->I * eb, 1024); }
    L.h_sf = o; if (p->dtype == MOK_MXFP8) o += align_up(rows * p->I / 32, 1024);
    if (!training) { L.partials = o; o += align_up((int64_t)p->T * p->k * p->H * 2, 1024); }
    if (!training && p->dtype == MOK_MXFP8) {   // x quantised once per token before the gather
        L.xq = o; o += align_up((int64_t)p->T * p->H, 1024);
        L.xsf = o; o += align_up((int64_t)p->T * p->H / 32, 1024);
    }
    if (p->I_shared > 0) {
        L.shared = o; o += align_up((int64_t)p->T * p->H * 4, 1024);
        L.hs = o; o += align_up((int64_t)p->T * p->I_shared * 2, 1024);
    }
    L.total = o;
    size_t q = 0;
    L.sA = q; q += align_up(rows * p->H * 2, 1024);
    L.sGU = q; q += align_up(rows * 2 * p->I * 4, 1024);   // fp32 G | U
    L.sh = q; q += align_up(rows * p->I * 2, 1024);
    L.spart = q; q += align_up((int64_t)p->T * p->k * p->H * 2, 1024);
    L.saved_total = q;
    return L;
}

struct BwdLayout {
    size_t dy, dgu, da, gw, dl, dl_full, part, wrt, total;
    // MXFP8: the dgrad operands (rows blocked along their K), the backward's
    // weight copies, and the weight-gradient operands transposed (tokens as K)
    size_t dyq, dysf, dguq, dgusf, wdq, wdsf, wgq, wgsf, wuq, wusf, atq, atsf, gutq, gutsf, htq, htsf, dytq, dytsf;
};

BwdLayout bwd_layout(const mok_problem* p) {
    BwdLayout L{};
    const int64_t rows = rows_tiles(p);
    size_t o = kStatusBytes;
    L.dy = o; o += align_up(rows * p->H * 2, 1024);
    L.dgu = o; o += align_up(rows * 2 * p->I * 2, 1024);
    L.da = o; o += align_up((int64_t)p->T * p->k * p->H * 2, 1024);
    L.gw = o; o += align_up((int64_t)p->T * p->k * 4, 1024);
    L.dl = o; o += align_up((int64_t)p->T * p->k * 4, 1024);
    L.dl_full = o; o += align_up((int64_t)p->T * p->E * 4, 1024);
    L.part = o; o += align_up(dwr_partial_floats(p->H, p->E) * 4, 1024);
    L.wrt = o; o += align_up((int64_t)p->E * p->H * 4, 1024);
    if (p->dtype == MOK_MXFP8) {
        const int64_t H = p->H, I = p->I, E = p->E;
        auto q = [&](size_t& codes, size_t& sf, int64_t R, int64_t K) {
            codes = o; o += align_up(R * K, 1024);
            sf = o; o += align_up(R * K / 32, 1024);
        };
        q(L.dyq, L.dysf, rows, H);
        q(L.dguq, L.dgusf, rows, 2 * I);
        L.wdq = o;   // the weights' backward copies when the caller passes none
        o += packed_bwd_layout((int)E, (int)H, (int)I).total;
        q(L.atq, L.atsf, H, rows);
        q(L.gutq, L.gutsf, 2 * I, rows);
        q(L.htq, L.htsf, I, rows);
        q(L.dytq, L.dytsf, H, rows);
    }
    L.total = o;
    return L;
}

mok_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA; }

constexpr int kDefaultMovers = 8;
// The grouped GEMMs' producers prefetch the weight box this many K blocks
// ahead of its load into L2 (beyond the shared-memory ring).
constexpr int kL2PrefetchBlocks = 8;

// Megakernel tiles: gate/up 256 wide (gate 128 | up 128), down as the staged
// down GEMM (down_tile_n).
bool mega_supported(const mok_problem* p) {
    return (2 * p->I) % 256 == 0 && p->H % down_tile_n(p->H, p->dtype == MOK_MXFP8) == 0;
}

int mega_region_rows(const mok_problem* p, const mok_config* cfg) {
    if (cfg && cfg->ring_rows > 0) return (cfg->ring_rows / 2) / kTileM * kTileM;
    return (int)align_up(padded_rows_max(p->T, p->E, p->k), kTileM);
}

struct MegaLayout {
    size_t scratch, partials, shared, hs, total;
};

MegaLayout mega_layout(const mok_problem* p, int nbatch, const mok_config* cfg) {
    MegaLayout L{};
    size_t o = kStatusBytes;
    L.scratch = o;
    o += align_up(mega_scratch_bytes(nbatch, p->T, p->H, p->I, p->E, p->k, mega_region_rows(p, cfg),
                                     p->dtype == MOK_MXFP8), 1024);
    L.partials = o;
    o += (size_t)nbatch * align_up((int64_t)p->T * p->k * p->H * 2, 1024);
    L.shared = o;
    if (p->I_shared > 0) o += (size_t)nbatch * align_up((int64_t)p->T * p->H * 4, 1024);
    L.hs = o;
    if (p->I_shared > 0) o += align_up((int64_t)p->T * p->I_shared * 2, 1024);
    L.total = o;
    return L;
}

// 2-SM pairs (cta_group::2) run the BF16 grouped GEMMs by default: measured
// on the 32-expert H=7168/I=2048 layer (GEMM pair alone, L2 flushed,
// interleaved repeats), 14-24 % faster than single CTAs when every expert has
// an even number of 128-row tiles and 3-8 % faster with random routing, where
// an odd last tile leaves half a pair idle. MXFP8 stays on single CTAs (its
// pairs measured slower); MOK_FLAG_GEMM_PAIRS forces pairs, MOK_FLAG_ROW_TILES
// single CTAs.
GemmCommon make_common(void* ws, const mok_config* cfg, int dtype = MOK_BF16) {
    GemmCommon c{};
    c.status = static_cast<StatusBlock*>(ws);
    int ms = (cfg && cfg->timeout_ms > 0) ? cfg->timeout_ms : kDefaultTimeoutMs;
    c.timeout_ns = (unsigned long long)ms * 1000000ull;
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (cfg && cfg->num_sms > 0) n = std::min(n, (int)cfg->num_sms);
    c.num_sms = n > 0 ? n : 1;
    const int flags = cfg ? cfg->flags : 0;
    c.cluster = (flags & MOK_FLAG_GEMM_PAIRS) ? 2 : (flags & MOK_FLAG_ROW_TILES) ? 1 : (dtype == MOK_BF16 ? 2 : 1);
    c.l2_prefetch = (cfg && (cfg->flags & MOK_FLAG_NO_L2_PREFETCH)) ? 0 : kL2PrefetchBlocks;
    return c;
}

// BF16 inference GEMMs: swapped-operand pair tiles (weight rows as M, token
// tiles of 256 rows plus a remainder as N) or the 128-row token tiles.
// Measured on the 32-expert H=7168/I=2048 layer (GEMM pair alone, L2
// flushed, three interleaved repeats): the token tiles were as fast or
// faster at 512, 640, 768 and 1024 rows per expert, with exact and with
// random routing (random, 640 rows: 1430 against 1390 TFLOP/s; 1024 rows:
// 1540 against 1397), so they are the default; MOK_FLAG_SWAPPED_TILES selects
// the swapped tiles (the autotuner times both).
bool use_swap(const mok_problem* p, const mok_config* cfg, bool training) {
    if (p->dtype != MOK_BF16 || training) return false;
    if (!swap_supported(p->H, p->I)) return false;
    const int flags = cfg ? cfg->flags : 0;
    if (flags & (MOK_FLAG_ROW_TILES | MOK_FLAG_GEMM_PAIRS)) return false;
    return (flags & MOK_FLAG_SWAPPED_TILES) != 0;
}
int swap_policy(const mok_config* cfg) { return (cfg && (cfg->flags & MOK_FLAG_TOKEN_TILES_BALANCED)) ? 1 : 0; }

// Routing arrays present (the per-token ones may be empty when T == 0).
bool routing_ok(const mok_routing* r, int32_t T = 1) {
    return r && r->counts && r->offsets &&
           (T == 0 || (r->topk_idx && r->topk_w && r->row_src && r->slot_row));
}

// Requires an sm_103-class device for the tensor-core kernels.
bool device_ok() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

}  // namespace

extern "C" {

const char* mok_version(void) { return "mok-gb300 0.1 (sm_103a)"; }

const char* mok_status_string(mok_status s) {
    switch (s) {
        case MOK_OK: return "ok";
        case MOK_ERR_INVALID: return "invalid argument";
        case MOK_ERR_CUDA: return "CUDA error";
        case MOK_ERR_TIMEOUT: return "device wait timed out";
        case MOK_ERR_CAPACITY: return "ring buffer smaller than one minibatch";
        case MOK_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

size_t mok_route_workspace_size(int32_t T, int32_t H, int32_t E, int32_t k) {
    if (T < 0 || H <= 0 || E < 1 || E > kMaxE || k < 1 || k > E) return 0;
    return route_workspace_bytes(T, H, E, k);
}

mok_status mok_route_layout(const void* x, const float* W_r, const float* bias, int32_t T, int32_t H, int32_t E,
                            int32_t k, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                            int32_t* row_src, int32_t* slot_row, void* workspace, size_t ws_bytes,
                            mok_stream_t stream) {
    if (T < 0 || H <= 0 || H % 8 || E < 1 || E > kMaxE || k < 1 || k > E) return MOK_ERR_INVALID;
    if ((int64_t)T * k >= (int64_t)1 << 30) return MOK_ERR_INVALID;
    if (!counts || !offsets || !workspace || !W_r) return MOK_ERR_INVALID;
    if (T > 0 && (!x || !topk_idx || !topk_w || !row_src || !slot_row)) return MOK_ERR_INVALID;
    if (ws_bytes < route_workspace_bytes(T, H, E, k) || !aligned(workspace, 256) || !aligned(x, 16))
        return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return cuda_status(launch_route_layout(x, W_r, bias, T, H, E, k, topk_idx, topk_w, counts, offsets, row_src,
                                           slot_row, workspace, (cudaStream_t)stream));
}

size_t mok_packed_weights_bwd_size(int32_t E, int32_t H, int32_t I, int32_t dtype) {
    if (dtype != MOK_MXFP8 || !dims_ok(E, H, I, dtype)) return 0;
    return packed_bwd_layout(E, H, I).total;
}

mok_status mok_pack_weights_bwd(int32_t E, int32_t H, int32_t I, int32_t dtype, const void* W_gate, const void* W_up,
                                const void* W_down, void* packed_bwd, size_t bytes, mok_stream_t stream) {
    if (dtype != MOK_MXFP8 || !dims_ok(E, H, I, dtype) || !W_gate || !W_up || !W_down || !packed_bwd)
        return MOK_ERR_INVALID;
    if (bytes < packed_bwd_layout(E, H, I).total || !aligned(packed_bwd, 256)) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return cuda_status(pack_bwd(W_gate, W_up, W_down, E, H, I, static_cast<char*>(packed_bwd), (cudaStream_t)stream));
}

size_t mok_packed_weights_size(int32_t E, int32_t H, int32_t I, int32_t dtype) {
    if (!dims_ok(E, H, I, dtype)) return 0;
    return packed_layout(E, H, I, dtype).total;
}

mok_status mok_pack_weights(int32_t E, int32_t H, int32_t I, int32_t dtype, const void* W_gate, const void* W_up,
                            const void* W_down, void* packed, size_t packed_bytes, mok_stream_t stream) {
    if (!dims_ok(E, H, I, dtype) || !W_gate || !W_up || !W_down || !packed) return MOK_ERR_INVALID;
    PackedLayout L = packed_layout(E, H, I, dtype);
    if (packed_bytes < L.total || !aligned(packed, 256)) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    char* b = static_cast<char*>(packed);
    const bool mx = dtype == MOK_MXFP8;
    cudaError_t e = launch_pack(mx, W_gate, W_up, E, H, I, gu_interleave(I, dtype), b + L.gu,
                                mx ? reinterpret_cast<uint8_t*>(b + L.gu_sf) : nullptr, 128, s);
    if (e == cudaSuccess)
        e = launch_pack(mx, W_down, nullptr, E, I, H, 0, b + L.dn, mx ? reinterpret_cast<uint8_t*>(b + L.dn_sf) : nullptr,
                        down_tile_n(H, mx), s);
    return cuda_status(e);
}

int64_t mok_padded_rows_max(int32_t T, int32_t E, int32_t k) { return padded_rows_max(T, E, k); }

size_t mok_saved_size(const mok_problem* p) {
    if (!problem_ok(p)) return 0;
    return fwd_layout(p, true).saved_total;
}

size_t mok_workspace_size(const mok_problem* p, const mok_config* cfg) {
    if (!problem_ok(p)) return 0;
    size_t f = fwd_layout(p, false).total;
    size_t b = bwd_layout(p).total;
    size_t m = mega_supported(p) ? mega_layout(p, 1, cfg).total : 0;
    return std::max(std::max(f, b), m);
}

size_t mok_workspace_size_batches(const mok_problem* p, int32_t nbatch, const mok_config* cfg) {
    if (!problem_ok(p) || nbatch < 1 || nbatch > kMaxBatches || !mega_supported(p)) return 0;
    return mega_layout(p, nbatch, cfg).total;
}

mok_status mok_dispatch(const mok_problem* p, const void* x, const mok_routing* r, void* A, void* A_sf,
                        mok_stream_t stream) {
    if (!problem_ok(p) || !routing_ok(r, p->T) || !A || (p->T > 0 && !x)) return MOK_ERR_INVALID;
    if (p->dtype == MOK_MXFP8 && !A_sf) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return cuda_status(launch_dispatch(p->dtype == MOK_MXFP8, x, p->T, p->H, p->E, p->k, r->counts, r->offsets,
                                       r->row_src, A, static_cast<uint8_t*>(A_sf), nullptr, nullptr,
                                       (cudaStream_t)stream));
}

mok_status mok_quantize_rows(const void* x, int32_t T, int32_t H, void* x_q, void* x_sf, mok_stream_t stream) {
    if (T < 0 || H <= 0 || H % 128 != 0) return MOK_ERR_INVALID;
    if (T > 0 && (!x || !x_q || !x_sf || !aligned(x, 16) || !aligned(x_q, 16) || !aligned(x_sf, 4)))
        return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return cuda_status(launch_quantize_rows(x, T, H, x_q, x_sf, (cudaStream_t)stream));
}

mok_status mok_dispatch_quantized(const mok_problem* p, const void* x_q, const void* x_sf, const mok_routing* r,
                                  void* A, void* A_sf, mok_stream_t stream) {
    if (!problem_ok(p) || p->dtype != MOK_MXFP8 || !routing_ok(r, p->T) || !A || !A_sf || !aligned(A, 16))
        return MOK_ERR_INVALID;
    if (p->T > 0 && (!x_q || !x_sf || !aligned(x_q, 16) || !aligned(x_sf, 4))) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    if (p->T == 0) return MOK_OK;
    return cuda_status(launch_dispatch_q(x_q, x_sf, p->T, p->H, p->E, p->k, r->counts, r->offsets, r->row_src, A,
                                         static_cast<uint8_t*>(A_sf), (cudaStream_t)stream));
}

mok_status mok_dispatch_tokens(const mok_problem* p, const void* x, const mok_routing* r, void* A, void* A_sf,
                               mok_stream_t stream) {
    if (!problem_ok(p) || p->dtype != MOK_MXFP8 || !routing_ok(r, p->T) || !A || !A_sf || !aligned(A, 32))
        return MOK_ERR_INVALID;
    if (p->T > 0 && (!x || !aligned(x, 16))) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return cuda_status(launch_dispatch_tokens(x, p->T, p->H, p->E, p->k, r->topk_idx, r->slot_row, r->counts,
                                              r->offsets, A, static_cast<uint8_t*>(A_sf), (cudaStream_t)stream));
}

mok_status mok_expert_ffn(const mok_problem* p, const void* A, const void* A_sf, const void* packed,
                          const mok_routing* r, void* h, void* h_sf, void* partials, const mok_config* cfg,
                          void* workspace, mok_stream_t stream) {
    if (!problem_ok(p) || !routing_ok(r, p->T) || !A || !packed || !h || !partials || !workspace) return MOK_ERR_INVALID;
    const bool mx = p->dtype == MOK_MXFP8;
    if (mx && (!A_sf || !h_sf)) return MOK_ERR_INVALID;
    if (!aligned(A, 1024) || !aligned(h, 1024) || !aligned(packed, 256) || !aligned(workspace, 256) ||
        !aligned(partials, 32))
        return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    cudaMemsetAsync(workspace, 0, kStatusBytes, s);
    if (p->T == 0) return MOK_OK;
    GemmCommon c = make_common(workspace, cfg, p->dtype);
    PackedLayout L = packed_layout(p->E, p->H, p->I, p->dtype);
    const char* pk = static_cast<const char*>(packed);
    const int64_t rows = padded_rows_max(p->T, p->E, p->k);
    cudaError_t e;
    if (use_swap(p, cfg, false)) {
        e = gemm_gateup_swap(A, pk + L.gu, p->E, p->H, p->I, r->counts, rows, h, swap_policy(cfg), c, s);
        if (e == cudaSuccess)
            e = gemm_down_swap(h, pk + L.dn, p->E, p->H, p->I, r->counts, r->offsets, r->row_src, rows, partials,
                               swap_policy(cfg), c, s);
        return cuda_status(e);
    }
    e = gemm_gateup(mx, A, static_cast<const uint8_t*>(A_sf), pk + L.gu,
                    reinterpret_cast<const uint8_t*>(pk + L.gu_sf), p->E, p->H, p->I, r->counts, 0, rows,
                    h, static_cast<uint8_t*>(h_sf), nullptr, c, s);
    if (e == cudaSuccess)
        e = gemm_down(mx, h, static_cast<const uint8_t*>(h_sf), pk + L.dn, reinterpret_cast<const uint8_t*>(pk + L.dn_sf),
                      p->E, p->H, p->I, r->counts, r->offsets, r->row_src, 0, rows, partials, c, s);
    return cuda_status(e);
}

mok_status mok_combine(const mok_problem* p, const void* partials, const float* topk_w, const float* shared,
                       void* out, mok_stream_t stream) {
    if (!problem_ok(p) || (p->T > 0 && (!partials || !topk_w || !out))) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return cuda_status(launch_combine(partials, topk_w, shared, out, p->T, p->H, p->k, (cudaStream_t)stream));
}

static mok_status forward_mega(const mok_problem* p, int32_t nbatch, const mok_fwd_args* a,
                               const mok_config* cfg, mok_stream_t stream) {
    cudaStream_t s = (cudaStream_t)stream;
    const bool mx = p->dtype == MOK_MXFP8;
    char* ws = static_cast<char*>(a[0].workspace);
    MegaLayout ML = mega_layout(p, nbatch, cfg);
    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (p->T == 0 || e != cudaSuccess) return cuda_status(e);
    GemmCommon c = make_common(ws, cfg, p->dtype);
    const int movers = (cfg && cfg->mover_ctas > 0) ? cfg->mover_ctas : kDefaultMovers;
    if (movers >= c.num_sms) return MOK_ERR_INVALID;
    // shared expert first (BF16 tensor-core GEMMs over every token)
    const float* shared[kMaxBatches] = {};
    if (p->I_shared > 0) {
        PackedLayout SL = packed_layout(1, p->H, p->I_shared, MOK_BF16);
        const char* sp = static_cast<const char*>(a[0].packed_shared);
        void* hs = ws + ML.hs;
        const GemmCommon cs = make_common(ws, cfg, MOK_BF16);   // the shared expert is BF16 in every mode
        for (int b = 0; b < nbatch && e == cudaSuccess; ++b) {
            float* sh = reinterpret_cast<float*>(ws + ML.shared + (size_t)b * align_up((int64_t)p->T * p->H * 4, 1024));
            shared[b] = sh;
            e = gemm_gateup(false, a[b].x, nullptr, sp + SL.gu, nullptr, 1, p->H, p->I_shared, nullptr, p->T, p->T, hs,
                            nullptr, nullptr, cs, s);
            if (e == cudaSuccess)
                e = gemm_down(false, hs, nullptr, sp + SL.dn, nullptr, 1, p->H, p->I_shared, nullptr, nullptr,
                              nullptr, p->T, p->T, sh, cs, s);
        }
        if (e != cudaSuccess) return cuda_status(e);
    }
    PackedLayout PL = packed_layout(p->E, p->H, p->I, p->dtype);
    const char* pk = static_cast<const char*>(a[0].packed);
    MegaLaunch L{};
    L.mx = mx;
    L.E = p->E; L.H = p->H; L.I = p->I; L.k = p->k; L.T = p->T; L.nbatch = nbatch;
    for (int b = 0; b < nbatch; ++b) {
        L.x[b] = a[b].x;
        L.offsets[b] = a[b].routing.offsets;
        L.row_src[b] = a[b].routing.row_src;
        L.topk_w[b] = a[b].routing.topk_w;
        L.partials[b] = ws + ML.partials + (size_t)b * align_up((int64_t)p->T * p->k * p->H * 2, 1024);
        L.shared[b] = shared[b];
        L.out[b] = a[b].out;
    }
    L.gu = pk + PL.gu;
    L.dn = pk + PL.dn;
    L.gu_sf = mx ? reinterpret_cast<const uint8_t*>(pk + PL.gu_sf) : nullptr;
    L.dn_sf = mx ? reinterpret_cast<const uint8_t*>(pk + PL.dn_sf) : nullptr;
    L.scratch = ws + ML.scratch;
    L.region_rows = mega_region_rows(p, cfg);
    L.max_tokens = (cfg && cfg->minibatch_tokens > 0) ? cfg->minibatch_tokens : p->T;
    L.tile_cuts = !(cfg && (cfg->flags & MOK_FLAG_MB_TOKEN_RANGES));
    L.n_movers = movers;
    L.grid = c.num_sms;
    L.test_flags = cfg ? cfg->flags : 0;
    L.trace = (cfg && (cfg->flags & MOK_FLAG_TRACE)) ? reinterpret_cast<unsigned long long*>(ws + ML.scratch)
                                                     : nullptr;
    L.status = c.status;
    L.timeout_ns = c.timeout_ns;
    return cuda_status(launch_mega(L, s));
}

mok_status mok_moe_forward_batches(const mok_problem* p, int32_t nbatch, const mok_fwd_args* a,
                                   const mok_config* cfg, mok_stream_t stream) {
    if (!problem_ok(p) || !a || nbatch < 1 || nbatch > kMaxBatches || !mega_supported(p)) return MOK_ERR_INVALID;
    if (!a[0].packed || !a[0].workspace || (p->I_shared > 0) != (a[0].packed_shared != nullptr))
        return MOK_ERR_INVALID;
    if (a[0].ws_bytes < mok_workspace_size_batches(p, nbatch, cfg) || !aligned(a[0].workspace, 1024) ||
        !aligned(a[0].packed, 256))
        return MOK_ERR_INVALID;
    for (int b = 0; b < nbatch; ++b) {
        if (!routing_ok(&a[b].routing, p->T) || !a[b].out || a[b].saved) return MOK_ERR_INVALID;
        if (p->T > 0 && (!a[b].x || !aligned(a[b].x, 16) || !aligned(a[b].out, 16))) return MOK_ERR_INVALID;
    }
    if (mega_region_rows(p, cfg) < kTileM) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    return forward_mega(p, nbatch, a, cfg, stream);
}

mok_status mok_moe_forward(const mok_problem* p, const mok_fwd_args* a, const mok_config* cfg,
                           mok_stream_t stream) {
    if (!problem_ok(p) || !a || !routing_ok(&a->routing, p->T) || !a->packed || !a->out || !a->workspace)
        return MOK_ERR_INVALID;
    if (p->T > 0 && !a->x) return MOK_ERR_INVALID;
    if ((p->I_shared > 0) != (a->packed_shared != nullptr)) return MOK_ERR_INVALID;
    const bool training = a->saved != nullptr;
    const bool mx = p->dtype == MOK_MXFP8;
    if (a->ws_bytes < mok_workspace_size(p, cfg) || !aligned(a->workspace, 1024) || !aligned(a->packed, 256) ||
        !aligned(a->x, 16) || !aligned(a->out, 16) || (training && !aligned(a->saved, 1024)))
        return MOK_ERR_INVALID;
    if (p->I_shared > 0 && !aligned(a->packed_shared, 256)) return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    if (!training && cfg && (cfg->flags & MOK_FLAG_MEGAKERNEL) && mega_supported(p)) {
        if (mega_region_rows(p, cfg) < kTileM) return MOK_ERR_INVALID;
        return forward_mega(p, 1, a, cfg, stream);
    }
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = static_cast<char*>(a->workspace);
    char* sv = static_cast<char*>(a->saved);
    FwdLayout L = fwd_layout(p, training);
    void* A = (training && !mx) ? sv + L.sA : ws + L.A;
    void* h = (training && !mx) ? sv + L.sh : ws + L.h;
    void* partials = training ? sv + L.spart : ws + L.partials;
    void* gu = training ? sv + L.sGU : nullptr;
    uint8_t* A_sf = mx ? reinterpret_cast<uint8_t*>(ws + L.A_sf) : nullptr;
    uint8_t* h_sf = mx ? reinterpret_cast<uint8_t*>(ws + L.h_sf) : nullptr;
    const mok_routing& r = a->routing;

    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (p->T == 0) return cuda_status(e);
    GemmCommon c = make_common(ws, cfg, p->dtype);
    PackedLayout PL = packed_layout(p->E, p->H, p->I, p->dtype);
    const char* pk = static_cast<const char*>(a->packed);
    const int64_t rows = padded_rows_max(p->T, p->E, p->k);
    if (e == cudaSuccess) {
        // pad rows stay unwritten for inference (their GEMM rows are never
        // stored); training keeps them zero for the weight gradients
        if (mx && !training)
            e = launch_dispatch_tokens(a->x, p->T, p->H, p->E, p->k, r.topk_idx, r.slot_row, r.counts, r.offsets, A,
                                       A_sf, s);
        else if (mx) {
            // MXFP8 training: the BF16 rows saved for the weight gradients (pads
            // zero), and the E4M3 rows for the GEMM quantised once per token from
            // x, their pads zeroed so the saved G|U and h of pad rows stay zero
            e = launch_dispatch(false, a->x, p->T, p->H, p->E, p->k, r.counts, r.offsets, r.row_src, sv + L.sA,
                                nullptr, nullptr, nullptr, s, true);
            if (e == cudaSuccess)
                e = launch_dispatch_tokens(a->x, p->T, p->H, p->E, p->k, r.topk_idx, r.slot_row, r.counts,
                                           r.offsets, A, A_sf, s);
            if (e == cudaSuccess) e = launch_zero_pad_rows_q(r.counts, rows, p->E, p->H, A, A_sf, s);
        } else {
            e = launch_dispatch(mx, a->x, p->T, p->H, p->E, p->k, r.counts, r.offsets, r.row_src, A, A_sf, nullptr,
                                nullptr, s, training);
        }
    }
    if (e == cudaSuccess && use_swap(p, cfg, training)) {
        e = gemm_gateup_swap(A, pk + PL.gu, p->E, p->H, p->I, r.counts, rows, h, swap_policy(cfg), c, s);
        if (e == cudaSuccess)
            e = gemm_down_swap(h, pk + PL.dn, p->E, p->H, p->I, r.counts, r.offsets, r.row_src, rows, partials,
                               swap_policy(cfg), c, s);
    } else {
        if (e == cudaSuccess)
            e = gemm_gateup(mx, A, A_sf, pk + PL.gu, reinterpret_cast<const uint8_t*>(pk + PL.gu_sf), p->E, p->H,
                            p->I, r.counts, 0, rows, h, h_sf, gu, c, s, (training && mx) ? sv + L.sh : nullptr);
        if (e == cudaSuccess)
            e = gemm_down(mx, h, h_sf, pk + PL.dn, reinterpret_cast<const uint8_t*>(pk + PL.dn_sf), p->E, p->H, p->I,
                          r.counts, r.offsets, r.row_src, 0, rows, partials, c, s);
    }
    float* shared = nullptr;
    if (e == cudaSuccess && p->I_shared > 0) {
        PackedLayout SL = packed_layout(1, p->H, p->I_shared, MOK_BF16);
        const char* sp = static_cast<const char*>(a->packed_shared);
        shared = reinterpret_cast<float*>(ws + L.shared);
        void* hs = ws + L.hs;
        const GemmCommon cs = make_common(ws, cfg, MOK_BF16);   // the shared expert is BF16 in every mode
        e = gemm_gateup(false, a->x, nullptr, sp + SL.gu, nullptr, 1, p->H, p->I_shared, nullptr, p->T, p->T, hs,
                        nullptr, nullptr, cs, s);
        if (e == cudaSuccess)
            e = gemm_down(false, hs, nullptr, sp + SL.dn, nullptr, 1, p->H, p->I_shared, nullptr, nullptr, nullptr,
                          p->T, p->T, shared, cs, s);
    }
    if (e == cudaSuccess) e = launch_combine(partials, r.topk_w, shared, a->out, p->T, p->H, p->k, s);
    return cuda_status(e);
}

mok_status mok_moe_backward(const mok_problem* p, const mok_bwd_args* a, const mok_config* cfg,
                            mok_stream_t stream) {
    if (!problem_ok(p) || !a || !routing_ok(&a->routing, p->T)) return MOK_ERR_INVALID;
    if (p->I_shared > 0) return MOK_ERR_UNSUPPORTED;
    const bool mx = p->dtype == MOK_MXFP8;
    if (!a->W_r || !a->W_gate || !a->W_up || !a->W_down || !a->saved || !a->dW_gate || !a->dW_up || !a->dW_down ||
        !a->dW_r || !a->workspace)
        return MOK_ERR_INVALID;
    if (p->T > 0 && (!a->x || !a->dY || !a->dX)) return MOK_ERR_INVALID;   // token arrays may be empty
    if (a->packed_bwd && (p->dtype != MOK_MXFP8 || !aligned(a->packed_bwd, 256))) return MOK_ERR_INVALID;
    if (a->ws_bytes < mok_workspace_size(p, cfg) || !aligned(a->workspace, 1024) || !aligned(a->saved, 1024) ||
        !aligned(a->dW_gate, 16) || !aligned(a->dW_up, 16) || !aligned(a->dW_down, 16))
        return MOK_ERR_INVALID;
    if (!device_ok()) return MOK_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = static_cast<char*>(a->workspace);
    const char* sv = static_cast<const char*>(a->saved);
    FwdLayout FL = fwd_layout(p, true);
    BwdLayout L = bwd_layout(p);
    const mok_routing& r = a->routing;
    const int T = p->T, H = p->H, I = p->I, E = p->E, k = p->k;
    const int64_t rows = padded_rows_max(T, E, k);
    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (T == 0) {
        // no tokens: every gradient is zero
        if (e == cudaSuccess) e = cudaMemsetAsync(a->dW_gate, 0, (size_t)E * H * I * 2, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(a->dW_up, 0, (size_t)E * H * I * 2, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(a->dW_down, 0, (size_t)E * H * I * 2, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(a->dW_r, 0, (size_t)E * H * 4, s);
        return cuda_status(e);
    }
    GemmCommon c = make_common(ws, cfg, p->dtype);
    void* dy = ws + L.dy;
    void* dgu = ws + L.dgu;
    void* da = ws + L.da;
    float* gw = reinterpret_cast<float*>(ws + L.gw);
    float* dl = reinterpret_cast<float*>(ws + L.dl);
    float* dl_full = reinterpret_cast<float*>(ws + L.dl_full);
    float* part = reinterpret_cast<float*>(ws + L.part);
    float* WrT = reinterpret_cast<float*>(ws + L.wrt);
    // reverse-combine (pull): dy rows in expert order, gate gradients
    if (e == cudaSuccess) e = launch_transpose_wr(a->W_r, WrT, H, E, 1, s);
    if (e == cudaSuccess)
        e = launch_dispatch(false, a->dY, T, H, E, k, r.counts, r.offsets, r.row_src, dy, nullptr, a->dY, r.topk_w, s);
    if (e == cudaSuccess)
        e = launch_bwd_small(a->dY, sv + FL.spart, r.topk_w, r.topk_idx, a->x, WrT, da, T, H, E, k, gw, dl, dl_full,
                             part, a->dX, a->dW_r, 0, s);
    if (mx) {
        // MXFP8: every GEMM operand quantised along that GEMM's reduction
        // dimension; the weights' backward copies are made per call (the
        // weights change with every optimizer step)
        auto Q = [&](size_t off) { return ws + off; };
        auto QS = [&](size_t off) { return reinterpret_cast<uint8_t*>(ws + off); };
        const int64_t rp = rows_tiles(p);
        // the weights' backward copies: packed once by the caller
        // (mok_pack_weights_bwd), or made here into the workspace
        const PackedBwdLayout PB = packed_bwd_layout(E, H, I);
        char* pb = a->packed_bwd ? static_cast<char*>(const_cast<void*>(a->packed_bwd)) : nullptr;
        if (!pb && e == cudaSuccess) {
            pb = ws + L.wdq;   // the workspace's weight-copy region has the same layout
            e = pack_bwd(a->W_gate, a->W_up, a->W_down, E, H, I, pb, s);
        }
        auto WQ = [&](size_t off) { return pb + off; };
        auto WS = [&](size_t off) { return reinterpret_cast<uint8_t*>(pb + off); };
        // dh = dy W_down^T (K = H), dSwiGLU -> dG|dU (BF16)
        // dy and dG|dU: quantised along both of their GEMMs' reduction dimensions in one read each
        if (e == cudaSuccess)
            e = launch_quantize_rows_cols_tiled(dy, rp, H, Q(L.dyq), QS(L.dysf), Q(L.dytq), QS(L.dytsf), s);
        if (e == cudaSuccess)
            e = gemm_dgrad_h_mx(Q(L.dyq), QS(L.dysf), WQ(PB.wd), WS(PB.wdsf), E, H, I, r.counts, rows, sv + FL.sGU,
                                dgu, c, s);
        // da = dG W_gate^T + dU W_up^T (K = I), pushed to the slots
        if (e == cudaSuccess)
            e = launch_quantize_rows_cols_tiled(dgu, rp, 2 * I, Q(L.dguq), QS(L.dgusf), Q(L.gutq), QS(L.gutsf), s);
        if (e == cudaSuccess)
            e = gemm_dgrad_a_mx(Q(L.dguq), QS(L.dgusf), WQ(PB.wg), WS(PB.wgsf), WQ(PB.wu), WS(PB.wusf), E, H, I,
                                r.counts, r.offsets, r.row_src, rows, da, c, s);
        // weight gradients over each expert's tokens: operands blocked along the tokens
        if (e == cudaSuccess) e = launch_quantize_cols_tiled(sv + FL.sA, rp, H, Q(L.atq), QS(L.atsf), s);
        if (e == cudaSuccess) e = launch_quantize_cols_tiled(sv + FL.sh, rp, I, Q(L.htq), QS(L.htsf), s);
        if (e == cudaSuccess)
            e = gemm_wgrad_mx(Q(L.atq), QS(L.atsf), H, Q(L.gutq), QS(L.gutsf), 2 * I, E, r.counts, rp, a->dW_gate,
                              a->dW_up, I, c, s);
        if (e == cudaSuccess)
            e = gemm_wgrad_mx(Q(L.htq), QS(L.htsf), I, Q(L.dytq), QS(L.dytsf), H, E, r.counts, rp, a->dW_down,
                              nullptr, H, c, s);
    } else {
        // expert dgrad
        if (e == cudaSuccess) e = gemm_dgrad_h(dy, a->W_down, E, H, I, r.counts, rows, sv + FL.sGU, dgu, c, s);
        if (e == cudaSuccess)
            e = gemm_dgrad_a(dgu, a->W_gate, a->W_up, E, H, I, r.counts, r.offsets, r.row_src, rows, da, c, s);
        // expert wgrad (each expert's rows, in row order)
        if (e == cudaSuccess)
            e = gemm_wgrad(sv + FL.sA, H, dgu, 2 * I, E, r.counts, rows, a->dW_gate, a->dW_up, I, c, s);
        if (e == cudaSuccess) e = gemm_wgrad(sv + FL.sh, I, dy, H, E, r.counts, rows, a->dW_down, nullptr, H, c, s);
    }
    // reverse-dispatch (push) + reduce, router gradient
    if (e == cudaSuccess)
        e = launch_bwd_small(a->dY, sv + FL.spart, r.topk_w, r.topk_idx, a->x, WrT, da, T, H, E, k, gw, dl, dl_full,
                             part, a->dX, a->dW_r, 1, s);
    return cuda_status(e);
}

mok_status mok_route_test_hook(int32_t withhold_copy, int32_t timeout_ms) {
    if (timeout_ms < 0) return MOK_ERR_INVALID;
    set_route_test_hook(withhold_copy != 0, (uint64_t)timeout_ms * 1000000ull);
    return MOK_OK;
}

mok_status mok_device_status(const void* workspace, mok_stream_t stream, int32_t* detail, int32_t reset) {
    if (!workspace) {
        // the status block of mok_route_layout_static's array on this device
        void* p = nullptr;
        if (route_static_scratch(&p) != cudaSuccess || !p) return MOK_ERR_CUDA;
        workspace = p;
    }
    StatusBlock hb{};
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&hb, workspace, sizeof(hb), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOK_ERR_CUDA;
    if (reset) {
        if (cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(hb), s) != cudaSuccess) return MOK_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOK_ERR_CUDA;
    }
    if (detail) *detail = hb.detail;
    return (mok_status)hb.code;
}

}  // extern "C"
