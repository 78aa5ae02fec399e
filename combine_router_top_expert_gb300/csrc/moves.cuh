// moves.cuh - host launchers of the routing, data-movement and GEMM kernels.
#pragma once

#include "common.cuh"

namespace mok {

// gemm.cu: tensor map of a row-major [rows, cols] tensor read in
// unswizzled boxes of box_cols x box_rows (out-of-range elements read 0)
bool make_tmap_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int elem_bytes, int box_cols,
                    int box_rows);

// route.cu
size_t route_workspace_bytes(int T, int H, int E, int k);
cudaError_t launch_route_layout(const void* x, const float* W_r, const float* bias, int T, int H, int E, int k,
                                int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                int32_t* row_src, int32_t* slot_row, void* ws, cudaStream_t s);
// Test hook of the routing kernels' bounded waits (process-wide): withhold
// makes CTA 0 of the top-k kernel skip one copy so its wait runs out after
// timeout_ns (0: the default limit).
struct RouteTestHook {
    int withhold;
    uint64_t timeout_ns;
};
RouteTestHook route_test_hook();
void set_route_test_hook(int withhold, uint64_t timeout_ns);
// noalloc.cu: device address of the library's routing scratch array on the
// current device (its first 256 bytes are the status block of
// mok_route_layout_static)
cudaError_t route_static_scratch(void** out);
// W_r [H, E] -> `copies` identical copies of WrT [E, H], back to back.
cudaError_t launch_transpose_wr(const float* W_r, float* WrT, int H, int E, int copies, cudaStream_t s);

// moves.cu
// Gather rows into the padded expert-contiguous layout. BF16 with `wslot`:
// the rows are scale_src[t] * wslot[t*k+j] (reverse-combine of the backward).
cudaError_t launch_dispatch(bool mx, const void* x, int T, int H, int E, int k, const int32_t* counts,
                            const int32_t* offsets, const int32_t* row_src, void* A, uint8_t* A_sf,
                            const void* scale_src, const float* wslot, cudaStream_t s, bool zero_pads = true);
cudaError_t launch_combine(const void* partials, const float* w, const float* shared, void* out, int T, int H,
                           int k, cudaStream_t s);
// MXFP8 scales go per tile of sf_tile rows (128, or 224 for the down
// weights when H % 224 == 0: two 512-byte chunks per tile and K-chunk).
cudaError_t launch_pack(bool mx, const void* src0, const void* src1, int E, int K, int Nsrc, int il, void* dst,
                        uint8_t* dst_sf, int sf_tile, cudaStream_t s);
// stage 0: gw, dl; stage 1: dX, dW_r
cudaError_t launch_bwd_small(const void* dY, const void* partials, const float* w, const int32_t* idx,
                             const void* x, const float* WrT, const void* da, int T, int H, int E, int k, float* gw,
                             float* dl, float* dl_full, float* dwr_part, void* dX, float* dWr, int stage,
                             cudaStream_t s);
int64_t dwr_partial_floats(int H, int E);

// N-tile of the down GEMM; MXFP8 down weights keep their block scales per
// tile of this many rows.
inline int down_tile_n(int H, bool mx) {
    if (mx) return H % 256 == 0 ? 256 : H % 224 == 0 ? 224 : 128;
    return H % 256 == 0 ? 256 : 128;
}

// gemm.cu
// Raise a kernel's dynamic shared memory limit (per device) to at least `bytes`.
void ensure_smem_attr(const void* func, int bytes);

struct GemmCommon {
    StatusBlock* status;
    unsigned long long timeout_ns;
    int num_sms;
    int l2_prefetch;   // K blocks ahead at which the GEMM producers prefetch weight boxes into L2 (0: off)
    int cluster;   // 2: grouped GEMMs run as 2-SM CTA pairs (tcgen05 cta_group::2, B rows split
                   // between the two CTAs, no multicast loads; the BF16 default); 1: single CTAs
};
// Forward gate/up GEMM + SwiGLU. A: [rows, H] (bf16 or E4M3 + tile scales);
// packed B: [E * 2I, H] (interleaved gate/up per il = BN/2 columns).
// identity_rows > 0: A is a plain [identity_rows, H] matrix (shared expert;
// BF16 pairs then take ceil(identity_rows / 128) row tiles as for one expert).
cudaError_t gemm_gateup(bool mx, const void* A, const uint8_t* A_sf, const void* Bgu, const uint8_t* Bgu_sf,
                        int E, int H, int I, const int32_t* counts, int identity_rows, int64_t a_rows,
                        void* h, uint8_t* h_sf, void* gu_save, const GemmCommon& c, cudaStream_t s,
                        void* h_bf16 = nullptr);
// MXFP8 backward GEMMs (operands quantised along each GEMM's reduction
// dimension, scales in the tensor-core chunk order):
//   dgrad of the down projection: dh = dy W_down^T with dy [a_rows, H] and
//     W_down as [E*I, H], dSwiGLU epilogue (saved fp32 G|U) -> dG|dU bf16;
//   dgrad of gate/up: da = dG W_gate^T + dU W_up^T with dG|dU [a_rows, 2I] and
//     W_gate, W_up as [E*H, I], each row pushed to its slot;
//   weight gradients: out[e] = A^T B over expert e's token range, A given
//     transposed as [M, rows_pad] and B as [N, rows_pad] (tokens as K).
cudaError_t gemm_dgrad_h_mx(const void* dy_q, const uint8_t* dy_sf, const void* Wd_q, const uint8_t* Wd_sf, int E,
                            int H, int I, const int32_t* counts, int64_t a_rows, const void* gu, void* dgu,
                            const GemmCommon& c, cudaStream_t s);
cudaError_t gemm_dgrad_a_mx(const void* dgu_q, const uint8_t* dgu_sf, const void* Wg_q, const uint8_t* Wg_sf,
                            const void* Wu_q, const uint8_t* Wu_sf, int E, int H, int I, const int32_t* counts,
                            const int32_t* offsets, const int32_t* row_src, int64_t a_rows, void* da,
                            const GemmCommon& c, cudaStream_t s);
cudaError_t gemm_wgrad_mx(const void* AT_q, const uint8_t* AT_sf, int M, const void* BT_q, const uint8_t* BT_sf,
                          int N, int E, const int32_t* counts, int64_t rows_pad, void* out0, void* out1,
                          int split_col, const GemmCommon& c, cudaStream_t s);
// BF16 inference forward with the operands swapped (gemm_swap.cuh): weight
// rows as the M side of 2-SM pair tiles, token tiles of any multiple of 32
// rows as N. h [a_rows, I] (rows of the padded layout; only routed rows are
// written); down pushes each routed row to out[row_src[...]] (bf16).
// policy: SwapTilePolicy. Needs I % 128 == 0 and H % 256 == 0.
bool swap_supported(int H, int I);
cudaError_t gemm_gateup_swap(const void* A, const void* Bgu, int E, int H, int I, const int32_t* counts,
                             int64_t a_rows, void* h, int policy, const GemmCommon& c, cudaStream_t s);
cudaError_t gemm_down_swap(const void* h, const void* Bdn, int E, int H, int I, const int32_t* counts,
                           const int32_t* offsets, const int32_t* row_src, int64_t a_rows, void* out, int policy,
                           const GemmCommon& c, cudaStream_t s);
// Forward down GEMM; rows pushed to out[row_src[...]] (bf16) or, for
// identity_rows > 0, out[row] as f32.
// MXFP8 quantisation of each row of x [T, H] (the codes the dispatch writes):
// x_q [T, H] E4M3, x_sf [T, H/32] E8M0 bytes.
cudaError_t launch_quantize_rows(const void* x, int T, int H, void* x_q, void* x_sf, cudaStream_t s);
// Zero the pad rows of an MXFP8 expert-contiguous buffer of at most `rows`
// padded rows (codes 0, scale code 0), leaving the routed rows alone.
cudaError_t launch_zero_pad_rows_q(const int32_t* counts, int64_t rows, int E, int H, void* A, uint8_t* A_sf,
                                  cudaStream_t s);
// MXFP8 pull-dispatch in one token-major pass (each token quantised once,
// its k rows written from registers); pad rows are not written.
cudaError_t launch_dispatch_tokens(const void* x, int T, int H, int E, int k, const int32_t* topk_idx,
                                   const int32_t* slot_row, const int32_t* counts, const int32_t* offsets, void* A,
                                   uint8_t* A_sf, cudaStream_t s);
// MXFP8 quantisation of a row-major [R, K] BF16 matrix along K with scales in
// the tensor-core chunk order (R % 128 == 0, K % 128 == 0).
cudaError_t launch_quantize_rows_tiled(const void* src, int64_t R, int K, void* q, void* sf, cudaStream_t s);
// MXFP8 quantisation of the columns of a row-major [R, F] BF16 matrix along R
// (blocks of 32 rows), written transposed as a K-major [F, R] operand with
// chunk-ordered scales (R % 128 == 0, F % 128 == 0).
cudaError_t launch_quantize_cols_tiled(const void* src, int64_t R, int F, void* qT, void* sfT, cudaStream_t s);
// Both of the above from one read of the source (same bytes).
cudaError_t launch_quantize_rows_cols_tiled(const void* src, int64_t R, int F, void* q, void* sf, void* qT, void* sfT,
                                            cudaStream_t s);
// MXFP8 pull-dispatch of rows quantised by launch_quantize_rows (same bytes
// as launch_dispatch; pad rows left unwritten).
cudaError_t launch_dispatch_q(const void* x_q, const void* x_sf, int T, int H, int E, int k, const int32_t* counts,
                              const int32_t* offsets, const int32_t* row_src, void* A, uint8_t* A_sf,
                              cudaStream_t s);
cudaError_t gemm_down(bool mx, const void* h, const uint8_t* h_sf, const void* Bdn, const uint8_t* Bdn_sf, int E,
                      int H, int I, const int32_t* counts, const int32_t* offsets, const int32_t* row_src,
                      int identity_rows, int64_t a_rows, void* out, const GemmCommon& c, cudaStream_t s);
// dh = dy W_down^T with the dSwiGLU epilogue -> dGU [rows, 2I].
cudaError_t gemm_dgrad_h(const void* dy, const void* W_down, int E, int H, int I, const int32_t* counts,
                         int64_t a_rows, const void* gu, void* dgu, const GemmCommon& c, cudaStream_t s);
// da = dG W_gate^T + dU W_up^T, rows pushed to da[row_src[...]].
cudaError_t gemm_dgrad_a(const void* dgu, const void* W_gate, const void* W_up, int E, int H, int I,
                         const int32_t* counts, const int32_t* offsets, const int32_t* row_src, int64_t a_rows,
                         void* da, const GemmCommon& c, cudaStream_t s);
// out[e] = Aact_e^T B_e over each expert's padded rows; Aact [rows, M], B [rows, N].
cudaError_t gemm_wgrad(const void* Aact, int M, const void* B, int N, int E, const int32_t* counts, int64_t a_rows,
                       void* out0, void* out1, int split_col, const GemmCommon& c, cudaStream_t s);

}  // namespace mok
