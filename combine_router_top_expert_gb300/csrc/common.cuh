// common.cuh - shared definitions of the CUDA library (device + host).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "mok.h"

namespace mok {

// ---------------------------------------------------------------------------
// Sizes
// ---------------------------------------------------------------------------
constexpr int kTileM = 128;          // rows per tensor-core tile; expert segments pad to this
constexpr int kMaxE = 256;           // experts supported by the routing kernels
constexpr int kStatusBytes = 256;    // status block at the start of every workspace

inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows of the padded expert-contiguous layout, worst case over routings.
inline int64_t padded_rows_max(int64_t T, int64_t E, int64_t k) {
    return T * k + E * kTileM;
}

// ---------------------------------------------------------------------------
// Device status block (first 256 bytes of a workspace). code != 0 records the
// first failure of the last call; detail names where it happened.
// ---------------------------------------------------------------------------
struct StatusBlock {
    int32_t code;
    int32_t detail;
    int32_t abort;     // set once any CTA gives up; other CTAs stop waiting
    int32_t pad[61];
};
static_assert(sizeof(StatusBlock) == kStatusBytes, "status block size");

// Where a wait gave up (StatusBlock::detail).
enum WaitSite : int32_t {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaAccEmpty = 3,
    kSiteEpiAccFull = 4,
    kSiteDrain = 5,
    kSiteCounter = 6,
    kSiteRouterChunk = 7,
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_failure(StatusBlock* st, int32_t code, int32_t detail) {
    if (atomicCAS(&st->code, 0, code) == 0) st->detail = detail;
    atomicExch(&st->abort, 1);
}

__device__ __forceinline__ bool abort_requested(const StatusBlock* st) {
    return *((volatile const int32_t*)&st->abort) != 0;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched by launch_after (below)
// may become resident while the kernel before it on the stream is still
// running. pdl_wait() blocks until that kernel has completed and its memory
// writes are visible (a no-op for a plain launch), so everything before it
// may touch only shared memory, tensor memory, barriers and kernel
// parameters; pdl_allow_next() lets the next kernel on the stream start its
// own launch. The next kernel's CTAs take an SM only once every CTA of this
// grid has started, so a grid larger than one wave is never starved.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// kern<<<grid, block, smem, s>>>(args...) with the programmatic
// stream-serialization attribute (the kernel must call pdl_wait() before it
// reads or writes global memory that earlier work on the stream uses).
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                         Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------------------
// Numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
    return *reinterpret_cast<uint32_t*>(&p);
}

// E8M0 scale code of an MXFP8 block with largest magnitude amax (finite,
// >= 0): floor(log2(amax)) - 8 + 127, clamped at 0; read from the binary32
// exponent field, so no log2 is evaluated.
__device__ __forceinline__ uint32_t e8m0_code(float amax) {
    int eb = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    int c = eb - 8;
    return (uint32_t)(c < 0 ? 0 : c);
}

// 2^(127 - code): the exact reciprocal of the block scale.
__device__ __forceinline__ float e8m0_inv_scale(uint32_t code) {
    return __uint_as_float((254u - code) << 23);
}

// Two floats to two E4M3 bytes, round to nearest even, saturating; `a` lands
// in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
    __nv_fp8x2_storage_t r = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)r;
}

// Byte offset of the scale of (row r in a 128-row tile, 32-column block j in a
// 128-column block) inside that tile/block's 512-byte scale chunk. This is the
// order the tensor core reads block scales in after a 32x128b.warpx4 copy to
// tensor memory: row r lives in TMEM lane r % 32, column r / 32, byte j.
__host__ __device__ __forceinline__ int sf_chunk_offset(int r, int j) {
    return (r & 31) * 16 + (r >> 5) * 4 + j;
}

}  // namespace mok
