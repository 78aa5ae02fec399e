// moves.cu - the layer's memory-bound kernels: pull-dispatch (gather, with
// MXFP8 quantisation fused in), the fixed-order combine, weight packing, and
// the backward's reverse-combine and reverse-dispatch / router-gradient pass.
//
// Pages (KuCoin article on Cursor's MoK, section 02): the expert side pulls
// the tokens it needs ("pull dispatch") and results are pushed back to the
// tokens they belong to ("push combine"); in the backward the directions are
// pull on reverse-combine and push on reverse-dispatch. MXFP8 quantisation of
// activations is fused into the dispatch path instead of a separate kernel.
// The layer ends with a weighted sum (section 03) in a fixed floating-point
// order (RuntimeWire, "Rebuilding the MoE layer around communication").
#include <algorithm>

#include "common.cuh"
#include "moves.cuh"
#include "tc.cuh"

namespace mok {

// Padded segment offsets (each expert starts on a 128-row boundary).
__device__ __forceinline__ void padded_offsets(const int32_t* counts, int E, int32_t* poff) {
    if (threadIdx.x == 0) {
        int s = 0;
        for (int e = 0; e < E; ++e) {
            poff[e] = s;
            s += ceil_div(counts[e], kTileM) * kTileM;
        }
        poff[E] = s;
    }
    __syncthreads();
}

// expert owning padded row pr: last e with poff[e] <= pr (skips empty experts)
__device__ __forceinline__ int find_expert(const int32_t* poff, int E, int pr) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (poff[mid] <= pr) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// Pull-dispatch: one warp per padded row.
// ---------------------------------------------------------------------------
// One 32-element MXFP8 block: E8M0 code of its amax, E4M3 bytes of x / scale.
// Every quantiser of the library goes through quantize32.
__device__ __forceinline__ uint32_t quantize32(const float (&f)[32], uint4& o0, uint4& o1) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const uint32_t code = e8m0_code(amax);
    const float inv = e8m0_inv_scale(code);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = f32x2_to_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv) |
               (f32x2_to_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
    o0 = make_uint4(w[0], w[1], w[2], w[3]);
    o1 = make_uint4(w[4], w[5], w[6], w[7]);
    return code;
}

// 32 BF16 values (four 16-byte words) to fp32.
__device__ __forceinline__ void unpack32(const uint4 (&v)[4], float (&f)[32]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[8 * i + 0] = bf16_lo(v[i].x); f[8 * i + 1] = bf16_hi(v[i].x);
        f[8 * i + 2] = bf16_lo(v[i].y); f[8 * i + 3] = bf16_hi(v[i].y);
        f[8 * i + 4] = bf16_lo(v[i].z); f[8 * i + 5] = bf16_hi(v[i].z);
        f[8 * i + 6] = bf16_lo(v[i].w); f[8 * i + 7] = bf16_hi(v[i].w);
    }
}

__device__ __forceinline__ uint32_t quantize_block32(const __nv_bfloat16* src, uint4& o0, uint4& o1) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(s4 + i);
    float f[32];
    unpack32(v, f);
    return quantize32(f, o0, o1);
}

// Row-wise MXFP8 quantisation of x (warp per row; the codes the dispatch
// writes): x_q [T, H] E4M3, x_sf bytes [T, H/32] (= words [T, H/128], byte j
// of word c = scale of 32-block 4c + j).
__global__ void __launch_bounds__(256)
quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, uint8_t* __restrict__ xq,
                     uint8_t* __restrict__ xsf) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = H / 32;
    for (int64_t t = (int64_t)blockIdx.x * 8 + warp; t < T; t += (int64_t)gridDim.x * 8) {
        for (int b = lane; b < nb; b += 32) {
            uint4 o0, o1;
            const uint32_t code = quantize_block32(x + t * H + b * 32, o0, o1);
            uint4* dst = reinterpret_cast<uint4*>(xq + t * H + b * 32);
            dst[0] = o0;
            dst[1] = o1;
            xsf[t * nb + b] = (uint8_t)code;
        }
    }
}

// Pull-dispatch of rows already quantised once per token (quantize_rows):
// each routed row copies its token's E4M3 bytes, and the row's scale words
// (four codes per 128-wide chunk) go to the tile-ordered scale chunks. Pad
// rows are not written (inference: their GEMM rows are never stored). The
// bytes equal the fused quantising dispatch's, each token quantised once
// instead of k times.
__global__ void __launch_bounds__(256)
dispatch_q_kernel(const uint8_t* __restrict__ xq, const uint32_t* __restrict__ xsf, int H, int E, int k,
                  const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ row_src, uint8_t* __restrict__ A, uint8_t* __restrict__ A_sf) {
    __shared__ int32_t poff[kMaxE + 1];
    padded_offsets(counts, E, poff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = poff[E];
    const int kc_row = H / 128;
    for (int pr = blockIdx.x * 8 + warp; pr < total; pr += gridDim.x * 8) {
        const int e = find_expert(poff, E, pr);
        const int local = pr - poff[e];
        if (local >= counts[e]) continue;
        const int64_t tok = row_src[offsets[e] + local] / k;
        const uint4* s4 = reinterpret_cast<const uint4*>(xq + tok * H);
        uint4* dst = reinterpret_cast<uint4*>(A + (int64_t)pr * H);
        const int n = H / 16;
        // batches of eight 16-byte loads in flight per lane (the last one masked)
        for (int c = lane; c < n; c += 256) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + 32 * u < n) v[u] = __ldg(s4 + c + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + 32 * u < n) __stcs(dst + c + 32 * u, v[u]);
        }
        const int rt = pr / kTileM, r = pr % kTileM;
        for (int q = lane; q < kc_row; q += 32)
            *reinterpret_cast<uint32_t*>(A_sf + ((int64_t)rt * kc_row + q) * 512 + sf_chunk_offset(r, 0)) =
                __ldg(xsf + tok * kc_row + q);
    }
}

// MXFP8 pull-dispatch in one token-major pass: W warps (1 or 2) take a token
// and lane L of warp w quantises the 32-element blocks 32w + L, 32w + L + 32W,
// ... of its row once (the encoder of quantize_rows), then writes each
// block's 32 codes with one 32-byte store to each of the token's k rows of
// the padded expert-contiguous layout (a warp store covers 1 KB of a row);
// the four scale codes of a 128-wide chunk, held by four neighbouring lanes,
// leave as one word. Every token row is read once and no quantised copy of x
// is written and read back. Pad rows are not written. The bytes equal those
// of quantize_rows + dispatch_q. Two warps per token keep twice the loads in
// flight when there are too few tokens to fill the GPU with one each.
__global__ void __launch_bounds__(256)
dispatch_tokens_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int E, int k, int W,
                       const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_row,
                       const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                       uint8_t* __restrict__ A, uint8_t* __restrict__ A_sf) {
    __shared__ int32_t poff[kMaxE + 1];
    pdl_wait();
    pdl_allow_next();
    padded_offsets(counts, E, poff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = H / 32, kc_row = H / 128;
    const int64_t units = (int64_t)T * W;
    for (int64_t u = (int64_t)blockIdx.x * 8 + warp; u < units; u += (int64_t)gridDim.x * 8) {
        const int64_t t = u / W;
        const int bw = (int)(u % W) * 32;   // this warp's first block
        // padded destination row of slot j (lane j holds it when k <= 32)
        auto dest = [&](int j) {
            const int64_t sl = t * k + j;
            const int e = topk_idx[sl];
            return poff[e] + slot_row[sl] - offsets[e];
        };
        const int my_pr = (k <= 32 && lane < k) ? dest(lane) : 0;
        // lane L quantises blocks bw + L, bw + L + 32W, ...; the next
        // iteration's four 16-byte loads are issued before this one's blocks
        // are quantised and stored
        const uint4* xs = reinterpret_cast<const uint4*>(x + t * H);
        const int step = 32 * W;
        uint4 nv[4];
        if (bw + lane < nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) nv[i] = __ldg(xs + (bw + lane) * 4 + i);
        // every lane runs the same trip counts (the shuffles need the whole
        // warp); nb % 4 == 0, so the four lanes of a chunk are all active or
        // all idle
        for (int b0 = bw; b0 < nb; b0 += step) {
            const int b = b0 + lane;
            const bool act = b < nb;
            const uint4 cv[4] = {nv[0], nv[1], nv[2], nv[3]};
            if (b + step < nb)
#pragma unroll
                for (int i = 0; i < 4; ++i) nv[i] = __ldg(xs + (b + step) * 4 + i);
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
            uint32_t code = 0;
            if (act) {
                float f[32];
                unpack32(cv, f);
                code = quantize32(f, o0, o1);
            }
            // the chunk's four codes, byte j = block 4c + j, in the chunk's first lane
            uint32_t word = code;
            word |= __shfl_down_sync(0xffffffffu, code, 1) << 8;
            word |= __shfl_down_sync(0xffffffffu, code, 2) << 16;
            word |= __shfl_down_sync(0xffffffffu, code, 3) << 24;
            const uint32_t w8[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
            for (int j = 0; j < k; ++j) {
                const int pr = k <= 32 ? __shfl_sync(0xffffffffu, my_pr, j) : dest(j);
                if (!act) continue;
                tc::stg_v8(A + (int64_t)pr * H + b * 32, w8);
                if ((lane & 3) == 0)
                    *reinterpret_cast<uint32_t*>(A_sf + ((int64_t)(pr / kTileM) * kc_row + b / 4) * 512 +
                                                 sf_chunk_offset(pr % kTileM, 0)) = word;
            }
        }
    }
}

// Pad rows of an MXFP8 expert-contiguous buffer (rows past each expert's
// count up to its 128-row boundary): zero E4M3 codes and the scale code of an
// all-zero block (0), the bytes a quantiser writes for zero rows. One warp
// per padded row; routed rows are left alone.
__global__ void __launch_bounds__(256)
zero_pad_rows_q_kernel(const int32_t* __restrict__ counts, int E, int H, uint8_t* __restrict__ A,
                       uint8_t* __restrict__ A_sf) {
    __shared__ int32_t poff[kMaxE + 1];
    padded_offsets(counts, E, poff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = poff[E];
    const int kc_row = H / 128;
    for (int pr = blockIdx.x * 8 + warp; pr < total; pr += gridDim.x * 8) {
        const int e = find_expert(poff, E, pr);
        if (pr - poff[e] < counts[e]) continue;
        uint4* dst = reinterpret_cast<uint4*>(A + (int64_t)pr * H);
        for (int c = lane; c < H / 16; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        for (int q = lane; q < kc_row; q += 32)
            *reinterpret_cast<uint32_t*>(A_sf + ((int64_t)(pr / kTileM) * kc_row + q) * 512 +
                                         sf_chunk_offset(pr % kTileM, 0)) = 0u;
    }
}

template <bool MX>
__global__ void __launch_bounds__(256)
dispatch_kernel(const __nv_bfloat16* __restrict__ x, int H, int E, int k, const int32_t* __restrict__ counts,
                const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_src, void* __restrict__ A,
                uint8_t* __restrict__ A_sf, const __nv_bfloat16* __restrict__ scale_src, const float* __restrict__ wslot,
                int zero_pads) {
    __shared__ int32_t poff[kMaxE + 1];
    pdl_wait();
    pdl_allow_next();
    padded_offsets(counts, E, poff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = poff[E];
    for (int pr = blockIdx.x * 8 + warp; pr < total; pr += gridDim.x * 8) {
        const int e = find_expert(poff, E, pr);
        const int local = pr - poff[e];
        const __nv_bfloat16* src = nullptr;
        float wmul = 1.f;
        if (local < counts[e]) {
            const int slot = row_src[offsets[e] + local];
            src = (scale_src ? scale_src : x) + (int64_t)(slot / k) * H;
            if (wslot) wmul = wslot[slot];
        } else if (!zero_pads) {
            continue;   // inference: pad rows feed only GEMM rows that are never stored
        }
        if constexpr (!MX) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(A) + (int64_t)pr * H);
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            const int n = H / 8;
            if (!src) {
                for (int c = lane; c < n; c += 32) __stcs(dst + c, make_uint4(0, 0, 0, 0));
            } else if (!wslot) {
                // batches of eight 16-byte loads in flight per lane before
                // their stores (the last batch masked); the rows stream out
                // (evict-first: read back only by the GEMM)
                for (int c = lane; c < n; c += 256) {
                    uint4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (c + 32 * u < n) v[u] = __ldg(s4 + c + 32 * u);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (c + 32 * u < n) __stcs(dst + c + 32 * u, v[u]);
                }
            } else {
                // reverse-combine: dy = w[t,j] * dY[t], rounded to bf16
                // (eight 16-byte loads in flight per lane, as above)
                auto scale = [&](const uint4& v) {
                    uint4 o;
                    o.x = pack_bf16x2(wmul * bf16_lo(v.x), wmul * bf16_hi(v.x));
                    o.y = pack_bf16x2(wmul * bf16_lo(v.y), wmul * bf16_hi(v.y));
                    o.z = pack_bf16x2(wmul * bf16_lo(v.z), wmul * bf16_hi(v.z));
                    o.w = pack_bf16x2(wmul * bf16_lo(v.w), wmul * bf16_hi(v.w));
                    return o;
                };
                for (int c = lane; c < n; c += 256) {
                    uint4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (c + 32 * u < n) v[u] = __ldg(s4 + c + 32 * u);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (c + 32 * u < n) dst[c + 32 * u] = scale(v[u]);
                }
            }
        } else {
            uint8_t* dst = static_cast<uint8_t*>(A) + (int64_t)pr * H;
            const int nb = H / 32;
            const int rt = pr / kTileM, r = pr % kTileM;
            // lane b%32 quantises block b; the four blocks of a 128-wide chunk
            // (lanes 4c..4c+3) store their codes as one 32-bit word
            for (int b0 = 0; b0 < nb; b0 += 32) {
                const int b = b0 + lane;
                const bool act = b < nb;   // nb is a multiple of 4: chunks are whole
                uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
                uint32_t code = 0;
                if (src && act) code = quantize_block32(src + b * 32, o0, o1);
                uint32_t word = code;
                word |= __shfl_down_sync(0xffffffffu, code, 1) << 8;
                word |= __shfl_down_sync(0xffffffffu, code, 2) << 16;
                word |= __shfl_down_sync(0xffffffffu, code, 3) << 24;
                if (act) {
                    reinterpret_cast<uint4*>(dst + b * 32)[0] = o0;
                    reinterpret_cast<uint4*>(dst + b * 32)[1] = o1;
                    if ((lane & 3) == 0)
                        *reinterpret_cast<uint32_t*>(A_sf + ((int64_t)rt * (H / 128) + b / 4) * 512 +
                                                     sf_chunk_offset(r, 0)) = word;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Fixed-order combine: out[t] = bf16(sum_j w[t,j] * y[t,j] (+ shared[t])).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
combine_kernel(const __nv_bfloat16* __restrict__ partials, const float* __restrict__ w,
               const float* __restrict__ shared, __nv_bfloat16* __restrict__ out, int H, int k) {
    pdl_wait();
    pdl_allow_next();
    const int t = blockIdx.x;
    const int n = H / 8;
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        // up to 8 slots' loads in flight, then their products in j order
        for (int j0 = 0; j0 < k; j0 += 8) {
            uint4 v[8];
            float wj[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (j0 + q < k) {
                    wj[q] = __ldg(w + (int64_t)t * k + j0 + q);
                    v[q] = __ldcs(reinterpret_cast<const uint4*>(partials + ((int64_t)t * k + j0 + q) * H) + c);
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (j0 + q < k) {
                    acc[0] = fmaf(wj[q], bf16_lo(v[q].x), acc[0]); acc[1] = fmaf(wj[q], bf16_hi(v[q].x), acc[1]);
                    acc[2] = fmaf(wj[q], bf16_lo(v[q].y), acc[2]); acc[3] = fmaf(wj[q], bf16_hi(v[q].y), acc[3]);
                    acc[4] = fmaf(wj[q], bf16_lo(v[q].z), acc[4]); acc[5] = fmaf(wj[q], bf16_hi(v[q].z), acc[5]);
                    acc[6] = fmaf(wj[q], bf16_lo(v[q].w), acc[6]); acc[7] = fmaf(wj[q], bf16_hi(v[q].w), acc[7]);
                }
            }
        }
        if (shared) {
            const float4* s = reinterpret_cast<const float4*>(shared + (int64_t)t * H) + 2 * c;
            float4 a = __ldg(s), b = __ldg(s + 1);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(out + (int64_t)t * H)[c] = o;
    }
}

// ---------------------------------------------------------------------------
// Weight packing: src [E][K][Nsrc] (row-major, K = reduction dim) ->
// dst rows [E][Ndst][K] (K-major). With src1 != NULL the destination
// interleaves the two sources per group of `il` columns:
//   dst row q*2il + r  = src0 column q*il + r       (r <  il)
//                      = src1 column q*il + r - il  (r >= il)
// One thread = one destination row x 32 K values.
// ---------------------------------------------------------------------------
template <bool MX>
__global__ void __launch_bounds__(256)
pack_kernel(const __nv_bfloat16* __restrict__ src0, const __nv_bfloat16* __restrict__ src1, int K, int Nsrc,
            int il, void* __restrict__ dst, uint8_t* __restrict__ dst_sf, int sf_tile) {
    const int Ndst = src1 ? 2 * Nsrc : Nsrc;
    const int e = blockIdx.z;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int kb = blockIdx.y;  // 32-wide K block
    if (n >= Ndst) return;
    const __nv_bfloat16* src;
    int col;
    if (src1) {
        const int q = n / (2 * il), r = n % (2 * il);
        src = r < il ? src0 : src1;
        col = q * il + (r < il ? r : r - il);
    } else {
        src = src0;
        col = n;
    }
    const __nv_bfloat16* s = src + (int64_t)e * K * Nsrc + (int64_t)(kb * 32) * Nsrc + col;
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __bfloat162float(s[(int64_t)i * Nsrc]);
    const int64_t grow = (int64_t)e * Ndst + n;
    if constexpr (!MX) {
        uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst) + grow * K + kb * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d[i] = make_uint4(pack_bf16x2(f[8 * i], f[8 * i + 1]), pack_bf16x2(f[8 * i + 2], f[8 * i + 3]),
                              pack_bf16x2(f[8 * i + 4], f[8 * i + 5]), pack_bf16x2(f[8 * i + 6], f[8 * i + 7]));
    } else {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
        const uint32_t code = e8m0_code(amax);
        const float inv = e8m0_inv_scale(code);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = f32x2_to_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv) |
                   (f32x2_to_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
        uint4* d = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dst) + grow * K + kb * 32);
        d[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d[1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (sf_tile == 224) {
            const int64_t nt = grow / 224;
            const int rr = (int)(grow % 224);
            dst_sf[((nt * (K / 128) + kb / 4) * 2 + rr / 128) * 512 + sf_chunk_offset(rr % 128, kb & 3)] = (uint8_t)code;
        } else {
            const int64_t rt = grow / kTileM;
            dst_sf[(rt * (K / 128) + kb / 4) * 512 + sf_chunk_offset((int)(grow % kTileM), kb & 3)] = (uint8_t)code;
        }
    }
}

// ---------------------------------------------------------------------------
// Backward helpers
// ---------------------------------------------------------------------------
// gw[t*k+j] = <dY[t], y[t,j]> (fp32, fixed order: lane-strided partial sums
// then a butterfly). One warp per slot.
__global__ void __launch_bounds__(256)
gate_grad_kernel(const __nv_bfloat16* __restrict__ dY, const __nv_bfloat16* __restrict__ partials, int T, int H,
                 int k, float* __restrict__ gw) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = blockIdx.x * 8 + warp;
    if (slot >= T * k) return;
    const int t = slot / k;
    const uint4* a = reinterpret_cast<const uint4*>(dY + (int64_t)t * H);
    const uint4* b = reinterpret_cast<const uint4*>(partials + (int64_t)slot * H);
    float s = 0.f;
    for (int c = lane; c < H / 8; c += 32) {
        uint4 u = __ldg(a + c), v = __ldg(b + c);
        s = fmaf(bf16_lo(u.x), bf16_lo(v.x), s); s = fmaf(bf16_hi(u.x), bf16_hi(v.x), s);
        s = fmaf(bf16_lo(u.y), bf16_lo(v.y), s); s = fmaf(bf16_hi(u.y), bf16_hi(v.y), s);
        s = fmaf(bf16_lo(u.z), bf16_lo(v.z), s); s = fmaf(bf16_hi(u.z), bf16_hi(v.z), s);
        s = fmaf(bf16_lo(u.w), bf16_lo(v.w), s); s = fmaf(bf16_hi(u.w), bf16_hi(v.w), s);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s = s + __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) gw[slot] = s;
}

// dl[t,j] = w_j (gw_j - sum_i w_i gw_i), i ascending.
__global__ void router_dlogit_kernel(const float* __restrict__ w, const float* __restrict__ gw, int T, int k,
                                     float* __restrict__ dl) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float m = 0.f;
    for (int j = 0; j < k; ++j) m = fmaf(w[(int64_t)t * k + j], gw[(int64_t)t * k + j], m);
    for (int j = 0; j < k; ++j) dl[(int64_t)t * k + j] = w[(int64_t)t * k + j] * (gw[(int64_t)t * k + j] - m);
}

// Reverse-dispatch push + reduce: dX[t] = bf16( sum_j da[t,j] + sum_j dl[t,j] W_r[:, e_j] ),
// j ascending in both sums, the expert term first.
__global__ void __launch_bounds__(128)
dx_kernel(const __nv_bfloat16* __restrict__ da, const float* __restrict__ dl, const int32_t* __restrict__ idx,
          const float* __restrict__ WrT, int H, int k, __nv_bfloat16* __restrict__ dX) {
    const int t = blockIdx.x;
    for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        // up to 8 slots' loads in flight, then their sums in j order
        for (int j0 = 0; j0 < k; j0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (j0 + q < k) v[q] = __ldcs(reinterpret_cast<const uint4*>(da + ((int64_t)t * k + j0 + q) * H) + c);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (j0 + q < k) {
                    acc[0] += bf16_lo(v[q].x); acc[1] += bf16_hi(v[q].x); acc[2] += bf16_lo(v[q].y);
                    acc[3] += bf16_hi(v[q].y); acc[4] += bf16_lo(v[q].z); acc[5] += bf16_hi(v[q].z);
                    acc[6] += bf16_lo(v[q].w); acc[7] += bf16_hi(v[q].w);
                }
            }
        }
        for (int j = 0; j < k; ++j) {
            const float d = dl[(int64_t)t * k + j];
            const float4* wr = reinterpret_cast<const float4*>(WrT + (int64_t)idx[(int64_t)t * k + j] * H) + 2 * c;
            float4 a = __ldg(wr), b = __ldg(wr + 1);
            acc[0] = fmaf(d, a.x, acc[0]); acc[1] = fmaf(d, a.y, acc[1]);
            acc[2] = fmaf(d, a.z, acc[2]); acc[3] = fmaf(d, a.w, acc[3]);
            acc[4] = fmaf(d, b.x, acc[4]); acc[5] = fmaf(d, b.y, acc[5]);
            acc[6] = fmaf(d, b.z, acc[6]); acc[7] = fmaf(d, b.w, acc[7]);
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(dX + (int64_t)t * H)[c] = o;
    }
}

// dl_full[t, e] = dl[t, j] where idx[t, j] == e, else 0.
__global__ void dl_scatter_kernel(const float* __restrict__ dl, const int32_t* __restrict__ idx, int T, int E,
                                  int k, float* __restrict__ dl_full) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    for (int e = 0; e < E; ++e) dl_full[(int64_t)t * E + e] = 0.f;
    for (int j = 0; j < k; ++j) dl_full[(int64_t)t * E + idx[(int64_t)t * k + j]] = dl[(int64_t)t * k + j];
}

// dW_r partial sums over a token range: part[split][h][e] = sum_{t in split}
// x[t,h] dl_full[t,e], t ascending. One thread per h, 32 experts per pass.
// 32 token ranges keep about six CTAs per SM busy at T = 4096 (the work is
// a few hundred dependent FMAs per loaded x value, so it needs warps).
constexpr int kDwrSplits = 32;
// Thread: two adjacent h (H is even), 32 experts at a time, the split's
// tokens in ascending order (each (h, e) partial is one fp32 chain over its
// token range); four tokens' x pairs are loaded before their products.
__global__ void __launch_bounds__(256)
dwr_partial_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ dl_full, int T, int H, int E,
                   float* __restrict__ part) {
    __shared__ float dls[64][32];
    const int h = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    const int split = blockIdx.y;
    const int per = ceil_div(T, kDwrSplits);
    const int ts = split * per, te = min(T, ts + per);
    const bool live = h < H;
    for (int eg = 0; eg < E; eg += 32) {
        float a0[32], a1[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) a0[e] = a1[e] = 0.f;
        for (int t0 = ts; t0 < te; t0 += 64) {
            const int nt = min(64, te - t0);
            __syncthreads();
            for (int i = threadIdx.x; i < 64 * 32; i += blockDim.x) {
                const int tt = i / 32, e = eg + i % 32;
                dls[tt][i % 32] = (tt < nt && e < E) ? dl_full[(int64_t)(t0 + tt) * E + e] : 0.f;
            }
            __syncthreads();
            if (!live) continue;
            const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(x + (int64_t)t0 * H + h);
            const int hs = H / 2;   // row stride in pairs
            int tt = 0;
            for (; tt + 4 <= nt; tt += 4) {
                __nv_bfloat162 xv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) xv[u] = xp[(int64_t)(tt + u) * hs];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float x0 = __low2float(xv[u]), x1 = __high2float(xv[u]);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float d = dls[tt + u][e];
                        a0[e] = fmaf(x0, d, a0[e]);
                        a1[e] = fmaf(x1, d, a1[e]);
                    }
                }
            }
            for (; tt < nt; ++tt) {
                const __nv_bfloat162 xv = xp[(int64_t)tt * hs];
                const float x0 = __low2float(xv), x1 = __high2float(xv);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float d = dls[tt][e];
                    a0[e] = fmaf(x0, d, a0[e]);
                    a1[e] = fmaf(x1, d, a1[e]);
                }
            }
        }
        // partials [split][e][h]: a warp's stores of one expert cover 256
        // contiguous bytes
        if (live) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (eg + e < E)
                    *reinterpret_cast<float2*>(part + ((int64_t)split * E + eg + e) * H + h) = make_float2(a0[e], a1[e]);
        }
    }
}

// dW_r[h, e] = sum over splits in ascending order (thread i: e = i / H,
// h = i % H, so the partials are read in contiguous runs of h).
__global__ void dwr_reduce_kernel(const float* __restrict__ part, int H, int E, float* __restrict__ dWr) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)H * E) return;
    const int e = (int)(i / H), h = (int)(i % H);
    float s = 0.f;
    for (int sp = 0; sp < kDwrSplits; ++sp) s += part[((int64_t)sp * E + e) * H + h];
    dWr[(int64_t)h * E + e] = s;
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

cudaError_t launch_dispatch(bool mx, const void* x, int T, int H, int E, int k, const int32_t* counts,
                            const int32_t* offsets, const int32_t* row_src, void* A, uint8_t* A_sf,
                            const void* scale_src, const float* wslot, cudaStream_t s, bool zero_pads) {
    int64_t rows = padded_rows_max(T, E, k);
    int blocks = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 8);
    if (blocks < 1) blocks = 1;
    const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* ss = static_cast<const __nv_bfloat16*>(scale_src);
    const float* noslot = nullptr;
    cudaError_t e =
        mx ? launch_after(dispatch_kernel<true>, dim3(blocks), dim3(256), 0, s, xs, H, E, k, counts, offsets, row_src,
                          A, A_sf, static_cast<const __nv_bfloat16*>(nullptr), noslot, zero_pads ? 1 : 0)
           : launch_after(dispatch_kernel<false>, dim3(blocks), dim3(256), 0, s, xs, H, E, k, counts, offsets, row_src,
                          A, static_cast<uint8_t*>(nullptr), ss, wslot, zero_pads ? 1 : 0);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dispatch_tokens(const void* x, int T, int H, int E, int k, const int32_t* topk_idx,
                                   const int32_t* slot_row, const int32_t* counts, const int32_t* offsets, void* A,
                                   uint8_t* A_sf, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    // two warps per token while one each would leave the GPU short of loads in
    // flight (fewer tokens than about 27 per SM: a warp per token then fills
    // at most 27 of the ~32 warp slots an SM holds at this register count)
    const int W = (int64_t)T < (int64_t)sm_count() * 27 ? 2 : 1;
    const int blocks = (int)std::min<int64_t>(ceil_div((int64_t)T * W, 8), (int64_t)sm_count() * 8);
    cudaError_t e = launch_after(dispatch_tokens_kernel, dim3(blocks), dim3(256), 0, s,
                                 static_cast<const __nv_bfloat16*>(x), T, H, E, k, W, topk_idx, slot_row, counts,
                                 offsets, static_cast<uint8_t*>(A), A_sf);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_zero_pad_rows_q(const int32_t* counts, int64_t rows, int E, int H, void* A, uint8_t* A_sf,
                                  cudaStream_t s) {
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 8));
    zero_pad_rows_q_kernel<<<blocks, 256, 0, s>>>(counts, E, H, static_cast<uint8_t*>(A), A_sf);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_q(const void* x_q, const void* x_sf, int T, int H, int E, int k, const int32_t* counts,
                              const int32_t* offsets, const int32_t* row_src, void* A, uint8_t* A_sf,
                              cudaStream_t s) {
    int64_t rows = padded_rows_max(T, E, k);
    int blocks = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 8);
    if (blocks < 1) blocks = 1;
    dispatch_q_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(x_q), static_cast<const uint32_t*>(x_sf), H, E,
                                             k, counts, offsets, row_src, static_cast<uint8_t*>(A), A_sf);
    return cudaGetLastError();
}

// MXFP8 quantisation of a row-major [R, F] BF16 matrix (R % 128 == 0,
// F % 128 == 0) in tiles of 32 rows x 128 columns, in one read of the source:
//  ROWS: along F, codes [R, F] E4M3 and scales in the tensor-core chunk order
//        of that [R, F] operand (chunk (r / 128, c / 128) of 512 bytes at
//        ((r / 128) * (F / 128) + c / 128) * 512, byte
//        sf_chunk_offset(r % 128, (c / 32) % 4));
//  COLS: along R in blocks of 32 rows, written transposed: codes [F, R] (row
//        f holds column f, so a GEMM reducing over R reads it K-major) and
//        scales in the chunk order of that [F, R] operand (chunk
//        (f / 128, r / 128), byte sf_chunk_offset(f % 128, (r / 32) % 4)).
// A CTA of 128 threads takes tile after tile: the tile arrives in 16-byte
// loads into shared memory (raw BF16, rows padded by 16 bytes), the next
// tile's loads are issued before this one is quantised, then thread t
// quantises column t (COLS) and row t / 4's 32-column block t % 4 (ROWS).
// Every block goes through quantize32, so both layouts hold the codes of the
// same rule as the other quantisers.
template <bool ROWS, bool COLS>
__global__ void __launch_bounds__(128)
quantize_tiles_kernel(const __nv_bfloat16* __restrict__ src, int64_t R, int F, uint8_t* __restrict__ q,
                      uint8_t* __restrict__ sf, uint8_t* __restrict__ qT, uint8_t* __restrict__ sfT) {
    constexpr int kPitch = 136;   // bf16 per shared row (128 + 8)
    __shared__ __align__(16) __nv_bfloat16 tile[32 * kPitch];
    const int tid = threadIdx.x;
    const int nfc = F / 128;
    const int64_t ntiles = (R / 32) * nfc;
    const int64_t nkc = R / 128;
    uint4 v[4];
    auto load = [&](int64_t blk) {
        const int64_t r0 = (blk / nfc) * 32;
        const int f0 = (int)(blk % nfc) * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = tid / 16 + 8 * u, c = tid % 16;
            v[u] = __ldg(reinterpret_cast<const uint4*>(src + (r0 + r) * F + f0 + 8 * c));
        }
    };
    int64_t blk = blockIdx.x;
    if (blk < ntiles) load(blk);
    for (; blk < ntiles; blk += gridDim.x) {
        const int64_t r0 = (blk / nfc) * 32;
        const int f0 = (int)(blk % nfc) * 128;
        __syncthreads();   // the previous tile's shared reads are done
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = tid / 16 + 8 * u, c = tid % 16;
            *reinterpret_cast<uint4*>(tile + r * kPitch + 8 * c) = v[u];
        }
        __syncthreads();
        if (blk + gridDim.x < ntiles) load(blk + gridDim.x);
        if constexpr (COLS) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __bfloat162float(tile[i * kPitch + tid]);
            uint4 o0, o1;
            const uint32_t code = quantize32(f, o0, o1);
            const int fc = f0 + tid;
            uint4* dst = reinterpret_cast<uint4*>(qT + (int64_t)fc * R + r0);
            dst[0] = o0;
            dst[1] = o1;
            sfT[((int64_t)(fc / kTileM) * nkc + r0 / 128) * 512 + sf_chunk_offset(fc % kTileM, (int)((r0 / 32) % 4))] =
                (uint8_t)code;
        }
        if constexpr (ROWS) {
            const int r = tid >> 2, b = tid & 3;
            float f[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 w = *reinterpret_cast<const uint4*>(tile + r * kPitch + 32 * b + 8 * i);
                f[8 * i + 0] = bf16_lo(w.x); f[8 * i + 1] = bf16_hi(w.x);
                f[8 * i + 2] = bf16_lo(w.y); f[8 * i + 3] = bf16_hi(w.y);
                f[8 * i + 4] = bf16_lo(w.z); f[8 * i + 5] = bf16_hi(w.z);
                f[8 * i + 6] = bf16_lo(w.w); f[8 * i + 7] = bf16_hi(w.w);
            }
            uint4 o0, o1;
            const uint32_t code = quantize32(f, o0, o1);
            const int64_t rg = r0 + r;
            uint4* dst = reinterpret_cast<uint4*>(q + rg * F + f0 + 32 * b);
            dst[0] = o0;
            dst[1] = o1;
            sf[((rg / kTileM) * nfc + f0 / 128) * 512 + sf_chunk_offset((int)(rg % kTileM), b)] = (uint8_t)code;
        }
    }
}

namespace {
template <bool ROWS, bool COLS>
cudaError_t launch_quantize_tiles(const void* src, int64_t R, int F, void* q, void* sf, void* qT, void* sfT,
                                  cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    // whole 128-row scale chunks on both sides
    if (R % 128 || F % 128) return cudaErrorInvalidValue;
    const int64_t n = (R / 32) * (F / 128);
    const int blocks = (int)std::min<int64_t>(n, (int64_t)sm_count() * 16);
    quantize_tiles_kernel<ROWS, COLS><<<blocks, 128, 0, s>>>(
        static_cast<const __nv_bfloat16*>(src), R, F, static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf),
        static_cast<uint8_t*>(qT), static_cast<uint8_t*>(sfT));
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_quantize_rows_tiled(const void* src, int64_t R, int K, void* q, void* sf, cudaStream_t s) {
    return launch_quantize_tiles<true, false>(src, R, K, q, sf, nullptr, nullptr, s);
}

cudaError_t launch_quantize_cols_tiled(const void* src, int64_t R, int F, void* qT, void* sfT, cudaStream_t s) {
    return launch_quantize_tiles<false, true>(src, R, F, nullptr, nullptr, qT, sfT, s);
}

cudaError_t launch_quantize_rows_cols_tiled(const void* src, int64_t R, int F, void* q, void* sf, void* qT, void* sfT,
                                            cudaStream_t s) {
    return launch_quantize_tiles<true, true>(src, R, F, q, sf, qT, sfT, s);
}

cudaError_t launch_quantize_rows(const void* x, int T, int H, void* x_q, void* x_sf, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>(ceil_div(T, 8), (int64_t)sm_count() * 8);
    quantize_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), T, H,
                                                static_cast<uint8_t*>(x_q), static_cast<uint8_t*>(x_sf));
    return cudaGetLastError();
}

cudaError_t launch_combine(const void* partials, const float* w, const float* shared, void* out, int T, int H,
                           int k, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    cudaError_t e = launch_after(combine_kernel, dim3(T), dim3(128), 0, s,
                                 static_cast<const __nv_bfloat16*>(partials), w, shared,
                                 static_cast<__nv_bfloat16*>(out), H, k);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_pack(bool mx, const void* src0, const void* src1, int E, int K, int Nsrc, int il, void* dst,
                        uint8_t* dst_sf, int sf_tile, cudaStream_t s) {
    const int Ndst = src1 ? 2 * Nsrc : Nsrc;
    dim3 grid(ceil_div(Ndst, 128), K / 32, E);
    if (mx)
        pack_kernel<true><<<grid, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(src0),
                                               static_cast<const __nv_bfloat16*>(src1), K, Nsrc, il, dst, dst_sf,
                                               sf_tile);
    else
        pack_kernel<false><<<grid, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(src0),
                                                static_cast<const __nv_bfloat16*>(src1), K, Nsrc, il, dst, dst_sf,
                                                sf_tile);
    return cudaGetLastError();
}

int64_t dwr_partial_floats(int H, int E) { return (int64_t)kDwrSplits * H * E; }

cudaError_t launch_bwd_small(const void* dY, const void* partials, const float* w, const int32_t* idx,
                             const void* x, const float* WrT, const void* da, int T, int H, int E, int k, float* gw,
                             float* dl, float* dl_full, float* part, void* dX, float* dWr, int stage,
                             cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (stage == 0) {
        gate_grad_kernel<<<ceil_div(T * k, 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(dY),
                                                            static_cast<const __nv_bfloat16*>(partials), T, H, k, gw);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        router_dlogit_kernel<<<ceil_div(T, 128), 128, 0, s>>>(w, gw, T, k, dl);
    } else {
        dx_kernel<<<T, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(da), dl, idx, WrT, H, k,
                                    static_cast<__nv_bfloat16*>(dX));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dl_scatter_kernel<<<ceil_div(T, 128), 128, 0, s>>>(dl, idx, T, E, k, dl_full);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dwr_partial_kernel<<<dim3(ceil_div(H, 512), kDwrSplits), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                                               dl_full, T, H, E, part);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dwr_reduce_kernel<<<ceil_div(H * E, 256), 256, 0, s>>>(part, H, E, dWr);
    }
    return cudaGetLastError();
}

}  // namespace mok
