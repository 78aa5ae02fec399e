// noalloc.cu - routing whose scratch memory belongs to the library.
//
// mok_route_layout needs a caller-provided workspace (a transposed copy of
// the router weights and per-block expert histograms). Some callers cannot
// hand one over: code running where every device allocation has to go
// through a host framework's own allocator that they cannot reach, plugins
// loaded into a process whose device memory is already fully reserved, or
// hot paths that are forbidden from allocating at all. mok_route_layout_static
// serves them: it runs the same kernels with their scratch in a file-scope
// device array of fixed size (MOK_ROUTE_STATIC_SCRATCH_BYTES) that every GPU
// loading the library keeps until the process exits. It allocates nothing.
#include <mutex>

#include "common.cuh"
#include "moves.cuh"

namespace {

static_assert(MOK_ROUTE_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size");

// The scratch array. In host code this name is only a host-side stand-in for
// the device variable: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_route_scratch[MOK_ROUTE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

namespace mok {
cudaError_t route_static_scratch(void** out) { return scratch_address(out); }
}  // namespace mok

extern "C" mok_status mok_route_layout_static(const void* x, const float* W_r, const float* bias, int32_t T,
                                              int32_t H, int32_t E, int32_t k, int32_t* topk_idx, float* topk_w,
                                              int32_t* counts, int32_t* offsets, int32_t* row_src,
                                              int32_t* slot_row, mok_stream_t stream) {
    using namespace mok;
    if (T < 0 || H <= 0 || H % 8 || E < 1 || E > kMaxE || k < 1 || k > E) return MOK_ERR_INVALID;
    if ((int64_t)T * k >= (int64_t)1 << 30) return MOK_ERR_INVALID;
    if (!counts || !offsets || !W_r) return MOK_ERR_INVALID;
    if (T > 0 && (!x || !topk_idx || !topk_w || !row_src || !slot_row)) return MOK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(x) & 15) != 0) return MOK_ERR_INVALID;
    // the problem's scratch must fit the fixed array
    if (route_workspace_bytes(T, H, E, k) > (size_t)MOK_ROUTE_STATIC_SCRATCH_BYTES) return MOK_ERR_INVALID;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOK_ERR_CUDA;
    int dev = 0, major = 0, minor = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return MOK_ERR_CUDA;
    // Every kernel writes its scratch (transposed router weights, block
    // histograms) in full before reading it; the 256-byte status block at the
    // start of the array is cleared by the launch sequence itself, so a
    // router wait that gives up in this call is what mok_device_status(NULL,
    // ...) reports afterwards.
    cudaError_t e = launch_route_layout(x, W_r, bias, T, H, E, k, topk_idx, topk_w, counts, offsets, row_src,
                                        slot_row, scratch, (cudaStream_t)stream);
    return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
