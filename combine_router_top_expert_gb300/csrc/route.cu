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

namespace mok {

constexpr int kRouteTT = 16;       // tokens per CTA
constexpr int kRouteThreads = 256;
constexpr int kRouteChunk = 256;   // h values per pipeline chunk (32 lanes x 8)

// W_r [H, E] -> WrT [E, H] so each expert's weights are contiguous.
__global__ void transpose_wr_kernel(const float* __restrict__ W_r, float* __restrict__ WrT, int H, int E) {
    __shared__ float tile[32][33];
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

// 16-byte global -> shared copy that bypasses L1; `bytes` = 0 fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int bytes) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One CTA = kRouteTT tokens x all experts. Warp w owns experts
// eg + 4w .. eg + 4w + 3 of each 32-expert group eg; lane c owns summation
// chain c (h = 256*i + 8*c + m). The x and router-weight chunks of 256 h
// values stream through a double-buffered shared-memory pipeline (cp.async),
// so chunk i+1 is in flight while chunk i is multiplied. Dynamic shared
// memory:
//   xs [2][kRouteTT][256] bf16 | ws [2][32][256] f32 | lg [kRouteTT][E] f32 |
//   slog [kRouteTT][k] f32 | cnt [E] i32
__global__ void __launch_bounds__(kRouteThreads)
route_topk_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ WrT,
                  const float* __restrict__ bias, int T, int H, int E, int k,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ hist) {
    extern __shared__ __align__(16) unsigned char route_smem[];
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(route_smem);
    float* ws = reinterpret_cast<float*>(route_smem + 2 * kRouteTT * kRouteChunk * 2);
    float* lg = ws + 2 * 32 * kRouteChunk;
    float* slog = lg + kRouteTT * E;
    int32_t* cnt = reinterpret_cast<int32_t*>(slog + kRouteTT * k);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRouteTT;
    const int ntok = min(kRouteTT, T - t0);
    const int nchunks = ceil_div(H, kRouteChunk);

    for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0;

    // issue the copies of chunk c (expert group eg) into buffer b
    auto load_chunk = [&](int eg, int c, int b) {
        const int h0 = c * kRouteChunk;
        __nv_bfloat16* xb = xs + b * kRouteTT * kRouteChunk;
        float* wb = ws + b * 32 * kRouteChunk;
        for (int v = tid; v < kRouteTT * (kRouteChunk / 8); v += kRouteThreads) {
            const int t = v / (kRouteChunk / 8), c8 = (v % (kRouteChunk / 8)) * 8;
            const bool ok = t < ntok && h0 + c8 < H;
            const __nv_bfloat16* src = ok ? x + (int64_t)(t0 + t) * H + h0 + c8 : x;
            cp_async16(xb + t * kRouteChunk + c8, src, ok ? 16 : 0);
        }
        for (int v = tid; v < 32 * (kRouteChunk / 4); v += kRouteThreads) {
            const int e = v / (kRouteChunk / 4), c4 = (v % (kRouteChunk / 4)) * 4;
            const bool ok = eg + e < E && h0 + c4 < H;
            const float* src = ok ? WrT + (int64_t)(eg + e) * H + h0 + c4 : WrT;
            cp_async16(wb + e * kRouteChunk + c4, src, ok ? 16 : 0);
        }
        cp_async_commit();
    };

    for (int eg = 0; eg < E; eg += 32) {
        float acc[kRouteTT][4];
#pragma unroll
        for (int t = 0; t < kRouteTT; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[t][q] = 0.f;

        __syncthreads();  // buffers free (previous expert group done)
        load_chunk(eg, 0, 0);
        for (int c = 0; c < nchunks; ++c) {
            if (c + 1 < nchunks) {
                load_chunk(eg, c + 1, (c + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const int h0 = c * kRouteChunk;
            const __nv_bfloat16* xb = xs + (c & 1) * kRouteTT * kRouteChunk;
            const float* wb = ws + (c & 1) * 32 * kRouteChunk;
            if (h0 + 8 * lane < H) {
                float wv[4][8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 a = *reinterpret_cast<const float4*>(wb + (4 * warp + q) * kRouteChunk + 8 * lane);
                    float4 b = *reinterpret_cast<const float4*>(wb + (4 * warp + q) * kRouteChunk + 8 * lane + 4);
                    wv[q][0] = a.x; wv[q][1] = a.y; wv[q][2] = a.z; wv[q][3] = a.w;
                    wv[q][4] = b.x; wv[q][5] = b.y; wv[q][6] = b.z; wv[q][7] = b.w;
                }
#pragma unroll
                for (int t = 0; t < kRouteTT; ++t) {
                    uint4 xv = *reinterpret_cast<const uint4*>(xb + t * kRouteChunk + 8 * lane);
                    float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                                   bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int m = 0; m < 8; ++m) acc[t][q] = fmaf(xf[m], wv[q][m], acc[t][q]);
                }
            }
            __syncthreads();  // buffer (c & 1) may be refilled by the next iteration
        }
        // butterfly across the 32 chains, then the bias
#pragma unroll
        for (int t = 0; t < kRouteTT; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float s = acc[t][q];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) s = s + __shfl_xor_sync(0xffffffffu, s, off);
                int e = eg + 4 * warp + q;
                if (lane == 0 && e < E && t < ntok) lg[t * E + e] = bias ? s + bias[e] : s;
            }
    }
    __syncthreads();

    // top-k per token: warp w takes tokens w, w + 8, ...
    const int nq = (E + 31) / 32;
    for (int t = warp; t < ntok; t += kRouteThreads / 32) {
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
    for (int e = tid; e < E; e += kRouteThreads) hist[(int64_t)blockIdx.x * E + e] = cnt[e];
}

size_t route_topk_smem_bytes(int E, int k) {
    return (size_t)2 * kRouteTT * kRouteChunk * 2 + 2 * 32 * kRouteChunk * 4 + (size_t)kRouteTT * E * 4 +
           (size_t)kRouteTT * k * 4 + (size_t)E * 4;
}

// Counts, offsets and the stable (expert, token) permutation. CTA b handles
// the same kRouteTT tokens as route_topk_kernel's CTA b: its rows for expert e
// start at offsets[e] + (rows of e in CTAs < b).
__global__ void __launch_bounds__(kRouteThreads)
route_layout_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ hist, int T, int E,
                    int k, int nblocks, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ row_src, int32_t* __restrict__ slot_row) {
    __shared__ int32_t pre[kMaxE], tot[kMaxE], off[kMaxE + 1];
    __shared__ int32_t part[kRouteThreads];
    __shared__ int32_t part2[kRouteThreads];
    __shared__ unsigned char sel[kRouteTT][kMaxE];
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const int t0 = b * kRouteTT;
    const int ntok = min(kRouteTT, T - t0);

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
    for (int i = tid; i < kRouteTT * E; i += kRouteThreads) sel[i / E][i % E] = 0;
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

cudaError_t launch_transpose_wr(const float* W_r, float* WrT, int H, int E, cudaStream_t s) {
    transpose_wr_kernel<<<dim3(ceil_div(H, 32), ceil_div(E, 32)), dim3(32, 8), 0, s>>>(W_r, WrT, H, E);
    return cudaGetLastError();
}

size_t route_workspace_bytes(int T, int H, int E, int k) {
    (void)k;
    int nblocks = ceil_div(T, kRouteTT);
    return (size_t)kStatusBytes + align_up((int64_t)E * H * 4, 256) + align_up((int64_t)nblocks * E * 4, 256);
}

cudaError_t launch_route_layout(const void* x, const float* W_r, const float* bias, int T, int H, int E, int k,
                                int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                int32_t* row_src, int32_t* slot_row, void* ws, cudaStream_t s) {
    char* base = static_cast<char*>(ws) + kStatusBytes;
    float* WrT = reinterpret_cast<float*>(base);
    int32_t* hist = reinterpret_cast<int32_t*>(base + align_up((int64_t)E * H * 4, 256));
    int nblocks = ceil_div(T, kRouteTT);
    if (T == 0) {
        cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    }
    transpose_wr_kernel<<<dim3(ceil_div(H, 32), ceil_div(E, 32)), dim3(32, 8), 0, s>>>(W_r, WrT, H, E);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    size_t smem = route_topk_smem_bytes(E, k);
    if (smem > 48 * 1024) ensure_smem_attr(reinterpret_cast<const void*>(route_topk_kernel), (int)smem);
    route_topk_kernel<<<nblocks, kRouteThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(x), WrT, bias, T, H, E,
                                                        k, topk_idx, topk_w, hist);
    // the layout kernel must never run on top-k results that were not produced
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    route_layout_kernel<<<nblocks, kRouteThreads, 0, s>>>(topk_idx, hist, T, E, k, nblocks, counts, offsets,
                                                          row_src, slot_row);
    return cudaGetLastError();
}

}  // namespace mok
