/*
 * mok.h - C ABI of the GB300 (sm_103a) routed MoE layer library, libmok.so.
 *
 * The layer follows the pages on Cursor's "Mixture-of-Kittens" (MoK):
 *   [K-ja]  KuCoin (ja) "Cursor's MoK achieves 2.37x performance boost on
 *           NVIDIA GB300 NVL72", sections 01, 02, 03 (and the Filipino copy).
 *   [RW]    RuntimeWire "Cursor open-sources MoK MoE training kernel",
 *           "Rebuilding the MoE layer around communication".
 * A router picks k experts per token; per-expert counts and an
 * expert-contiguous placement feed a grouped GEMM ([K-ja] 01); tokens are
 * pulled to their experts, each expert runs a SwiGLU FFN, results are pushed
 * back to their tokens and summed with the routing weights ([K-ja] 02, 03), in
 * a fixed floating-point order so repeated runs are bitwise identical ([RW]).
 * On one GPU the pull-dispatch is a gather from local HBM.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated; the caller owns
 *     and allocates every buffer (inputs, outputs, packed weights, workspace,
 *     saved context). The library never allocates device memory.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronise the host, except
 *     mok_device_status and the *_host entry points, which say so.
 *   - Row-major layouts. BF16 tensors are raw IEEE bfloat16 (2 bytes).
 *   - Argument errors are detected on the host before any launch and return
 *     MOK_ERR_INVALID (nothing is enqueued). CUDA launch errors return
 *     MOK_ERR_CUDA. Problems found on the device (a bounded wait that ran out,
 *     a ring too small for one minibatch) are written to a status word in the
 *     workspace; read it with mok_device_status after the stream work ends.
 *   - No CPU fallback: without an sm_103a device every compute call returns
 *     MOK_ERR_CUDA.
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* mok_stream_t; /* cudaStream_t */

typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1 } mok_dtype;

typedef enum {
    MOK_OK = 0,
    MOK_ERR_INVALID = 1,     /* bad argument (host check) */
    MOK_ERR_CUDA = 2,        /* CUDA runtime/driver error */
    MOK_ERR_TIMEOUT = 3,     /* a device-side bounded wait gave up */
    MOK_ERR_CAPACITY = 4,    /* ring buffer smaller than one minibatch */
    MOK_ERR_UNSUPPORTED = 5  /* valid but not built (e.g. a backward with a shared expert) */
} mok_status;

/* Shapes of one layer. T tokens, hidden H, expert intermediate I, E routed
 * experts, top-k. dtype: operand type of the routed experts (MOK_BF16 or
 * MOK_MXFP8, E4M3 elements + one E8M0 scale per 32 elements along each GEMM's
 * reduction dimension). I_shared > 0 adds one BF16 shared expert (SwiGLU, I =
 * I_shared) applied to every token with weight 1 ([RW]: shared experts stay
 * BF16). Limits: 1 <= k <= E <= 256; H % 128 == 0; I % 128 == 0 or I == 64
 * (BF16); I % 128 == 0 (MXFP8); I_shared likewise; T >= 0, T*k < 2^30. */
typedef struct {
    int32_t T, H, I, E, k;
    int32_t dtype;
    int32_t I_shared;
} mok_problem;

/* Execution knobs. Zero-initialise for defaults. The megakernel's SM split,
 * minibatch size and ring size are explicit parameters, as the pages set
 * them per shape ([K-ja] 02 and 03). */
typedef struct {
    int32_t num_sms;          /* SMs the persistent kernels may use; 0 = all */
    int32_t timeout_ms;       /* limit of every device-side wait; 0 = 4000 */
    int32_t flags;            /* MOK_FLAG_* */
    int32_t mover_ctas;       /* megakernel: SMs that move tokens; 0 = 8 */
    int32_t minibatch_tokens; /* megakernel: most tokens per minibatch (default expert-tile cuts: at most
                                 minibatch_tokens * k rows, rounded up to a 128-row tile); 0 = as many as
                                 a ring region holds */
    int32_t ring_rows;        /* megakernel: ring token buffer rows, split in two regions;
                                 0 = two regions of mok_padded_rows_max rows each */
    int32_t reserved[2];
} mok_config;

/* Run the inference forward as the persistent megakernel (mover/compute
 * SM split, GPU-local counters, ring) instead of the stage kernels
 * (dispatch, grouped GEMMs, combine). */
#define MOK_FLAG_MEGAKERNEL 1
/* 2-SM CTA pairs for the staged grouped GEMMs (BF16 forward gate/up and
 * down, backward dgrad; MXFP8 gate/up): tcgen05 cta_group::2 MMAs of 256 rows
 * over two CTAs, each staging its own 128 A rows and half of the B rows
 * (MXFP8: its A rows' block scales and all B rows' scales). Results are
 * bit-identical to single-CTA kernels; an expert whose row count is an odd
 * number of 128-row tiles leaves half of its last pair idle. The BF16 GEMMs
 * run as pairs by default (measured faster); this flag also puts the MXFP8
 * gate/up GEMM on pairs (measured slower). The shared expert and the MXFP8
 * down GEMM always run single CTAs; the MXFP8 weight gradients always run as
 * pairs when the weight rows are a multiple of 256. */
#define MOK_FLAG_GEMM_PAIRS 2
/* Megakernel trace: the launch writes one record of eight uint64 per CTA
 * (CTA i at byte offset 256 + 64*i of the workspace): [0] role (0 mover,
 * 1 compute), [1] globaltimer at entry (ns), [2] start of its first unit of
 * work (mover: first minibatch; compute: first tile's loads, after its
 * counter wait), [3] end of its tile/move work, [4] exit, [5] ns spent
 * waiting on GPU-local counters (compute: tile inputs published; mover:
 * ring region free, less the weighted-sum chunks it took meanwhile), [6]
 * units done (tiles; minibatches), [7] ns in the weighted sums (mover: the
 * chunks taken while waiting plus the final pass after [3]). Costs a few
 * timer reads per tile. */
#define MOK_FLAG_TRACE 4
/* Megakernel minibatches as token ranges: each minibatch holds the rows of
 * a range of tokens, padded per expert to 128-row tiles, and its tokens'
 * weighted sums run as soon as its down tiles are done. By default a
 * minibatch is a run of consecutive 128-row tiles of the batch's
 * expert-contiguous layout (padded once per expert over the whole batch),
 * and a batch's weighted sums run once all of its minibatches are done. */
#define MOK_FLAG_MB_TOKEN_RANGES 8
/* The BF16 inference GEMMs run either on 128-row token tiles (the tokens as
 * the M side of the tensor-core tiles, each expert's rows padded to whole
 * tiles) or with the operands swapped: the weight rows as the M side of 2-SM
 * pair tiles (256 rows over two CTAs) and an expert's tokens cut into tiles
 * of 256 rows and one remainder tile (a multiple of 32 rows) as the N side,
 * so little tensor work is spent on padded rows and no CTA of a pair idles
 * (needs I % 128 == 0 and H % 256 == 0). The token tiles are the default
 * (measured as fast or faster from 512 to 1024 rows per expert), as 2-SM
 * pairs for BF16 (MOK_FLAG_GEMM_PAIRS); MOK_FLAG_SWAPPED_TILES selects the
 * swapped tiles, MOK_FLAG_ROW_TILES the token tiles on single CTAs. The
 * training forward (saved != NULL) and MXFP8 always use the token tiles. */
#define MOK_FLAG_ROW_TILES 16
#define MOK_FLAG_SWAPPED_TILES 128
/* Swapped-operand tiles: cut each expert's tokens into ceil(n/256) tiles of
 * about equal size (multiples of 32) instead of tiles of 256 rows plus one
 * remainder tile (the default; measured faster). */
#define MOK_FLAG_TOKEN_TILES_BALANCED 32
/* The grouped GEMMs' TMA producers prefetch each weight box into L2 several
 * K blocks ahead of its load (beyond the shared-memory ring, into the next
 * tile at a tile's end); this flag turns the prefetches off. */
#define MOK_FLAG_NO_L2_PREFETCH 64
/* Test hook: a mover withholds the publish of the last 8-row chunk of the
 * first minibatch, so the tiles waiting for it give up after timeout_ms and
 * the call reports MOK_ERR_TIMEOUT (exercises the bounded waits; never use
 * in production). */
#define MOK_FLAG_TEST_WITHHOLD_PUBLISH 256

/* ------------------------------------------------------------------------- */
/* Router, top-k and layout ([K-ja] 01: count each expert's tokens, place each */
/* token, keep each expert's tokens adjacent for the grouped GEMM).           */
/* ------------------------------------------------------------------------- */

/* Workspace bytes mok_route_layout needs (device memory, any content): a
 * 256-byte status block first (read it with mok_device_status), then the
 * router weights re-laid out in the order the kernel streams them (fp32,
 * padded to 256-wide h chunks and 32-expert groups; up to 4 MB of identical
 * copies), then per-block expert histograms. */
size_t mok_route_workspace_size(int32_t T, int32_t H, int32_t E, int32_t k);

/* logits[t,e] = sum_h x[t,h] * W_r[h,e] (+ bias[e]) in binary32, in this fixed
 * order: 32 partial fma chains, chain c over h = 256*i + 8*c + m (i = 0,1,..,
 * m = 0..7, h < H), combined by butterfly adds with offsets 16,8,4,2,1, then
 * the bias add. Top-k by (logit descending, expert ascending); slot j is the
 * j-th ranked expert; topk_w[t,j] = exp(l_j - l_0) / sum_i exp(l_i - l_0)
 * (the softmax over E renormalised over the selected experts).
 * counts[e] = routed rows of expert e; offsets = exclusive prefix sum (E+1
 * entries, unpadded); rows are ordered by (expert, token); row_src[row] =
 * t*k + j; slot_row[t*k + j] = row.
 *   x [T,H] bf16, W_r [H,E] f32, bias [E] f32 or NULL;
 *   outputs topk_idx [T,k] i32, topk_w [T,k] f32, counts [E] i32,
 *   offsets [E+1] i32, row_src [T*k] i32, slot_row [T*k] i32.
 * Logits must be finite (non-finite inputs give unspecified routing).
 * Requires H % 8 == 0, x 16-byte aligned, workspace 256-byte aligned.
 * Device-side waits are bounded: one that gives up is recorded in the
 * workspace's status block (mok_device_status: MOK_ERR_TIMEOUT) and the
 * outputs are then unspecified. */
mok_status mok_route_layout(const void* x, const float* W_r, const float* bias,
                            int32_t T, int32_t H, int32_t E, int32_t k,
                            int32_t* topk_idx, float* topk_w, int32_t* counts,
                            int32_t* offsets, int32_t* row_src, int32_t* slot_row,
                            void* workspace, size_t ws_bytes, mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Expert weights                                                              */
/* ------------------------------------------------------------------------- */

/* Bytes of the packed form of E experts' weights (dtype MOK_BF16/MOK_MXFP8). */
size_t mok_packed_weights_size(int32_t E, int32_t H, int32_t I, int32_t dtype);

/* One-time repacking of W_gate [E,H,I], W_up [E,H,I], W_down [E,I,H] (bf16,
 * device) into the K-major tile layout the tensor-core GEMMs read, with gate
 * and up columns interleaved per output tile (so one tile holds matching gate
 * and up columns for the fused SwiGLU), and for MXFP8 quantised to E4M3 with
 * E8M0 scales per 32 elements along H (gate/up) and along I (down). Runs on
 * `stream`; `packed` must hold mok_packed_weights_size bytes, 256-B aligned.
 * For the shared expert pass E = 1 and dtype MOK_BF16. */
mok_status mok_pack_weights(int32_t E, int32_t H, int32_t I, int32_t dtype,
                            const void* W_gate, const void* W_up, const void* W_down,
                            void* packed, size_t packed_bytes, mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Forward                                                                     */
/* ------------------------------------------------------------------------- */

/* Routing produced by mok_route_layout (device pointers). */
typedef struct {
    const int32_t* topk_idx;  /* [T,k] */
    const float* topk_w;      /* [T,k] */
    const int32_t* counts;    /* [E] */
    const int32_t* offsets;   /* [E+1] */
    const int32_t* row_src;   /* [T*k] */
    const int32_t* slot_row;  /* [T*k] */
} mok_routing;

typedef struct {
    const void* x;             /* [T,H] bf16 */
    const void* packed;        /* routed experts, from mok_pack_weights */
    const void* packed_shared; /* shared expert (E=1, BF16) or NULL; needs I_shared > 0 */
    mok_routing routing;
    void* out;                 /* [T,H] bf16 */
    void* saved;               /* NULL (inference) or mok_saved_size bytes kept for backward */
    void* workspace;           /* mok_workspace_size bytes, 256-B aligned */
    size_t ws_bytes;
} mok_fwd_args;

/* Workspace bytes of mok_moe_forward / mok_moe_backward for this problem
 * (either forward path, one batch). */
size_t mok_workspace_size(const mok_problem* p, const mok_config* cfg);
/* Workspace bytes of mok_moe_forward_batches for nbatch macro-batches. */
size_t mok_workspace_size_batches(const mok_problem* p, int32_t nbatch, const mok_config* cfg);
/* Bytes of the saved context (BF16 training forward only). */
size_t mok_saved_size(const mok_problem* p);

/* The layer forward: pull-gather (+MXFP8 quantisation) of each routed row
 * into expert-contiguous order, grouped gate/up GEMM with fused SwiGLU
 * (+MXFP8 quantisation of h), grouped down GEMM whose epilogue pushes each
 * row to its (token, slot) partial, then out[t] = bf16(sum_{j=0..k-1}
 * w[t,j] * y[t,j] (+ shared[t])) in fp32 with j ascending. Bitwise
 * deterministic, and the same bits on either path.
 * By default the stage kernels run in sequence on the stream. With
 * MOK_FLAG_MEGAKERNEL, inference (saved == NULL) runs the persistent
 * megakernel ([K-ja] 02) instead: one cooperative launch whose first
 * cfg->mover_ctas CTAs gather minibatches into a two-region ring while the
 * other CTAs run the tensor-core tiles; the two sides synchronise through
 * GPU-local counters only. It needs every SM of the device (the launch fails
 * with MOK_ERR_CUDA if they cannot all be resident) and tile widths that
 * divide H and 2I (256 for BF16, 128 for MXFP8); other shapes use the stage
 * kernels. The device status reports MOK_ERR_CAPACITY if a ring region
 * cannot hold the padded rows of 16 tokens. `saved` != NULL (training) keeps
 * the activations the backward needs: the gathered rows (BF16), the fp32
 * gate/up pre-activations, h (BF16) and the partials; MXFP8 training keeps
 * the same BF16 values and runs its GEMMs on MXFP8 copies in the workspace. */
mok_status mok_moe_forward(const mok_problem* p, const mok_fwd_args* a,
                           const mok_config* cfg, mok_stream_t stream);

/* Macro-batch streaming ([K-ja] 02, ring token buffer): nbatch <= 32
 * independent batches of p->T tokens each (a[b].x, a[b].routing, a[b].out),
 * the same weights (a[0].packed / packed_shared) and one workspace
 * (a[0].workspace, mok_workspace_size_batches bytes), through ONE megakernel
 * launch: minibatches of consecutive batches flow through the same ring, so
 * the weighted sums of batch b overlap the dispatch of batch b+1. The shared
 * expert (if any) runs as tensor-core GEMMs before the megakernel, for all
 * batches. Inference only (a[b].saved must be NULL). */
mok_status mok_moe_forward_batches(const mok_problem* p, int32_t nbatch, const mok_fwd_args* a,
                                   const mok_config* cfg, mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* The forward's stages as separate calls (same kernels), for tests and for   */
/* callers that interleave their own work.                                    */
/* ------------------------------------------------------------------------- */

/* Rows of the padded expert-contiguous layout the stages use: each expert's
 * segment starts on a multiple of 128 rows; pad rows hold zeros. */
int64_t mok_padded_rows_max(int32_t T, int32_t E, int32_t k);

/* Pull-dispatch: for every padded row of expert e at local index r < counts[e],
 * A[row] = Q(x[t]) with t*k+j = row_src[offsets[e]+r]; pad rows are zero.
 * BF16: A is [rows_max, H] bf16 and A_sf is unused (NULL).
 * MXFP8: A is [rows_max, H] E4M3 bytes and A_sf receives the E8M0 scales in
 * the tensor-core tile order: for row-tile rt (128 rows) and 128-column block
 * kc, a 512-byte chunk at ((rt * (H/128)) + kc) * 512 whose byte
 * (r % 32) * 16 + (r / 32) * 4 + (c / 32) % 4 holds the scale of row 128*rt+r,
 * 32-column block c/32 (c within the 128-column block). */
mok_status mok_dispatch(const mok_problem* p, const void* x, const mok_routing* r,
                        void* A, void* A_sf, mok_stream_t stream);

/* MXFP8 quantisation of every row of x [T, H] bf16 (H % 128 == 0), once per
 * token (the same rule as mok_dispatch): x_q [T, H] E4M3 bytes and x_sf
 * [T, H/32] E8M0 bytes, block b of row t at byte t*(H/32) + b. x_q 16-B and
 * x_sf 4-B aligned. The quantising half of the MXFP8 dispatch that
 * mok_moe_forward runs: each token is quantised once instead of k times. */
mok_status mok_quantize_rows(const void* x, int32_t T, int32_t H, void* x_q, void* x_sf,
                             mok_stream_t stream);

/* MXFP8 pull-dispatch of rows quantised by mok_quantize_rows: A and A_sf as
 * mok_dispatch writes them for routed rows (the same bytes); pad rows are
 * left unwritten (the forward never stores the GEMM rows they feed).
 * p->dtype must be MOK_MXFP8; A 16-B aligned. */
mok_status mok_dispatch_quantized(const mok_problem* p, const void* x_q, const void* x_sf,
                                  const mok_routing* r, void* A, void* A_sf, mok_stream_t stream);

/* MXFP8 pull-dispatch in one token-major pass, as mok_moe_forward runs it:
 * each token's row is quantised once (the rule of mok_quantize_rows) and its
 * codes and scale words are written to each of its k routed rows (the bytes
 * of mok_dispatch for routed rows); pad rows are left unwritten. Uses
 * topk_idx, slot_row, counts and offsets of the routing. p->dtype must be
 * MOK_MXFP8; x 16-B and A 32-B aligned. */
mok_status mok_dispatch_tokens(const mok_problem* p, const void* x, const mok_routing* r, void* A, void* A_sf,
                               mok_stream_t stream);

/* Grouped expert FFN on the dispatched rows: h = SwiGLU(A W_gate[e], A W_up[e])
 * (BF16 or MXFP8 as dtype), y = h W_down[e], y row pushed to partials[t*k+j]
 * ([T*k, H] bf16, unweighted). h/h_sf are caller scratch of
 * [rows_max, I] (bf16 or E4M3; h_sf uses the same tile order as A_sf with I
 * in place of H; MXFP8 only). A and h must be 1024-B aligned, partials
 * 32-B aligned (rows leave in 32-byte stores). `workspace`
 * supplies the 256-byte device status block (its first 256 bytes). */
mok_status mok_expert_ffn(const mok_problem* p, const void* A, const void* A_sf,
                          const void* packed, const mok_routing* r, void* h, void* h_sf,
                          void* partials, const mok_config* cfg, void* workspace,
                          mok_stream_t stream);

/* Fixed-order weighted sum: out[t] = bf16(sum_j topk_w[t,j] * partials[t*k+j]
 * (+ shared[t])), fp32, j ascending. shared: [T,H] f32 or NULL. */
mok_status mok_combine(const mok_problem* p, const void* partials, const float* topk_w,
                       const float* shared, void* out, mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Backward (BF16 and MXFP8)                                                    */
/* ------------------------------------------------------------------------- */

typedef struct {
    const void* x;          /* [T,H] bf16 (forward input) */
    const float* W_r;       /* [H,E] f32 */
    const void* W_gate;     /* [E,H,I] bf16, original layout */
    const void* W_up;       /* [E,H,I] bf16 */
    const void* W_down;     /* [E,I,H] bf16 */
    const void* packed;     /* the forward's packed weights */
    const void* dY;         /* [T,H] bf16 upstream gradient */
    mok_routing routing;
    const void* saved;      /* filled by the training forward */
    void* dX;               /* [T,H] bf16 */
    void* dW_gate;          /* [E,H,I] bf16 */
    void* dW_up;            /* [E,H,I] bf16 */
    void* dW_down;          /* [E,I,H] bf16 */
    float* dW_r;            /* [H,E] f32 */
    void* workspace;
    size_t ws_bytes;
    const void* packed_bwd; /* MXFP8: the weights' backward copies from mok_pack_weights_bwd, or NULL
                               (then they are made in each call, in the workspace); NULL for BF16 */
} mok_bwd_args;

/* Bytes of the MXFP8 backward's weight copies (0 unless dtype == MOK_MXFP8). */
size_t mok_packed_weights_bwd_size(int32_t E, int32_t H, int32_t I, int32_t dtype);

/* The MXFP8 backward's weight copies, made once per weight update like the
 * forward's packing: W_down [E,I,H] quantised along H (for dh = dy W_down^T)
 * and W_gate, W_up [E,H,I] along I (for da), E4M3 codes with E8M0 scales in
 * the tensor-core chunk order. packed_bwd: mok_packed_weights_bwd_size bytes,
 * 256-B aligned. */
mok_status mok_pack_weights_bwd(int32_t E, int32_t H, int32_t I, int32_t dtype, const void* W_gate,
                                const void* W_up, const void* W_down, void* packed_bwd, size_t bytes,
                                mok_stream_t stream);

/* Backward of the layer ([K-ja] 02: pull on reverse-combine, push on
 * reverse-dispatch). Reverse-combine pulls dy[row] = w[t,j] * dY[t] into
 * expert order and gw[t,j] = <dY[t], y[t,j]>; grouped dgrad GEMMs give
 * dh = dy W_down^T, dG = dh*U*silu'(G), dU = dh*silu(G),
 * da = dG W_gate^T + dU W_up^T, each da row pushed to its slot; grouped wgrad
 * GEMMs reduce over each expert's rows in row order (no split, no atomics):
 * dW_gate = A^T dG, dW_up = A^T dU, dW_down = h^T dy; router: dl_j =
 * w_j (gw_j - sum_i w_i gw_i), dW_r = x^T dl, and dX[t] = sum_j da[t,j] +
 * sum_j dl_j W_r[:, e_j] in fixed order. The bias gets no gradient.
 * Bitwise deterministic. dW_gate, dW_up and dW_down must be 16-B aligned
 * (written by TMA stores), workspace and saved 1024-B aligned.
 * MXFP8 (p->dtype == MOK_MXFP8, after an MXFP8 training forward; [K-ja] 03
 * and [RW] report an MXFP8 backward): every backward GEMM takes MXFP8
 * operands blocked by 32 along its own reduction dimension - dy and W_down
 * along H for dh, dG|dU and W_gate, W_up along I for da, and x, h, dy, dG,
 * dU along each expert's rows for the weight gradients (quantised from the
 * BF16 values, transposed so the tokens are the K dimension). The weights'
 * backward copies come from a->packed_bwd (mok_pack_weights_bwd), or are
 * quantised in the call into the workspace when it is NULL. A shared
 * expert (I_shared > 0) has no backward here: MOK_ERR_UNSUPPORTED. */
mok_status mok_moe_backward(const mok_problem* p, const mok_bwd_args* a,
                            const mok_config* cfg, mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Expert parallelism across ranks ([K-ja] 02: experts spread over GPUs, the  */
/* expert side pulls the token rows it needs, results are pushed back to the  */
/* tokens' slots; [RW] "Rebuilding the MoE layer around communication").      */
/* ------------------------------------------------------------------------- */

#define MOK_EP_MAX_RANKS 8

/* One rank's buffers as this process reaches them (device pointers usable in
 * this process: on one GPU ordinary allocations; across the GPUs of a node,
 * pointers that map the peer's allocation, e.g. opened CUDA IPC handles). */
typedef struct {
    const void* x;            /* [T, H] bf16: the rank's tokens */
    const int32_t* offsets;   /* [E+1]: the rank's routing layout over all E experts */
    const int32_t* row_src;   /* [T*k]: the rank's expert-ordered row -> slot t*k+j */
    void* partials;           /* [T*k, H] bf16: the rank's slot buffer (mok_ep_push writes it) */
    int32_t T;                /* the rank's tokens */
} mok_ep_peer;

/* Workspace bytes of mok_ep_dispatch (0 for invalid G, E). */
size_t mok_ep_workspace_size(int32_t G, int32_t E);

/* Rank `rank` of G owns experts [rank*E/G, (rank+1)*E/G) (E % G == 0). After
 * every rank routed its own tokens over all E experts (mok_route_layout) and
 * the per-rank counts were all-gathered into counts_all [G, E] int32 (device,
 * rank-major; the caller's collective also orders this call after every
 * rank's routing), this call
 *   - lays out the local experts' rows: local expert l gets counts_local[l] =
 *     sum_s counts_all[s][rank*E/G + l] rows, ordered by source rank s, then
 *     by the source's own layout order; offsets_local [E/G+1] (unpadded);
 *   - pulls each row from its source: A[padded row] = x_s[t] with t*k+j =
 *     row_src_s[offsets_s[e] + r], in the padded expert-contiguous layout of
 *     mok_dispatch (each local expert's segment starts on a 128-row
 *     boundary; pad rows are not written);
 *   - records src_rank[row] = s, src_slot[row] = t*k+j, ident[row] = row for
 *     the push and for the down GEMM's scatter.
 * Then run mok_expert_ffn with the local problem {T = rows_cap, k = 1,
 * E = E/G, H, I} and routing {counts_local, offsets_local, row_src = ident}
 * (the other routing pointers only need to be non-NULL), writing y rows in
 * local row order into `ys` (its partials), then mok_ep_push. peers: host
 * array of G entries (entry `rank` is this rank's own buffers). rows_cap >=
 * sum_s T_s*k + 128*E/G rows of A; src_rank, src_slot and ident hold
 * rows_cap entries. Rows whose source layout disagrees with counts_all are
 * skipped (src_rank -1). Plain loads only: no TMA or multicast touches peer
 * memory. */
mok_status mok_ep_dispatch(int32_t G, int32_t rank, int32_t H, int32_t E, int32_t k,
                           const mok_ep_peer* peers, const int32_t* counts_all, void* A,
                           int64_t rows_cap, int32_t* counts_local, int32_t* offsets_local,
                           int32_t* src_rank, int32_t* src_slot, int32_t* ident, void* workspace,
                           size_t ws_bytes, mok_stream_t stream);

/* Push-combine: every local row's result ys[row] ([rows_cap, H] bf16, local
 * row order; rows < offsets_local[E/G]) is stored into
 * peers[src_rank[row]].partials at slot src_slot[row] (plain 16-byte
 * stores; rows marked -1 by the dispatch are skipped). Once every rank's
 * push is done (the caller's barrier), each rank sums its own slots with
 * mok_combine. */
mok_status mok_ep_push(int32_t G, int32_t H, int32_t E, int32_t k, const mok_ep_peer* peers,
                       const void* ys, int64_t rows_cap, const int32_t* offsets_local,
                       const int32_t* src_rank, const int32_t* src_slot, mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Routing without a caller workspace. The pages have no counterpart: this    */
/* entry point exists for callers of this library that cannot allocate.       */
/* ------------------------------------------------------------------------- */

/* Size of the device scratch array owned by the library (8 MiB). Every GPU
 * that loads libmok.so holds one such array until the process exits. */
#define MOK_ROUTE_STATIC_SCRATCH_BYTES (8u << 20)

/* Same computation, arguments and outputs as mok_route_layout, minus the
 * workspace: the scratch (transposed router weights and per-block expert
 * histograms, mok_route_workspace_size bytes) lives in a file-scope device
 * array of MOK_ROUTE_STATIC_SCRATCH_BYTES inside the library. For callers that
 * cannot allocate device memory themselves - e.g. code that must route every
 * allocation through a host framework's allocator it cannot reach, plugins in
 * processes whose device memory is already fully reserved, or hot paths where
 * allocating is not allowed. It calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Problems whose scratch exceeds the array (mok_route_workspace_size(T, H,
 *     E, k) > MOK_ROUTE_STATIC_SCRATCH_BYTES; e.g. one copy of the re-laid
 *     router weights, about E*H*4 bytes, must fit) return MOK_ERR_INVALID;
 *     nothing is enqueued.
 *   - All calls on a device share that device's array, which keeps the last
 *     call's contents; the kernels overwrite every byte they read, so nothing
 *     needs clearing, but calls that overlap on the same GPU (e.g. issued on
 *     different streams without ordering) race on the array: order them on
 *     one stream or with events.
 *   - Device-side waits are bounded as in mok_route_layout. A wait that gives
 *     up is recorded in a 256-byte status block at the start of the array;
 *     read it with mok_device_status(NULL, stream, &detail, reset) after the
 *     call (MOK_ERR_TIMEOUT, detail 7: the routing outputs are then not the
 *     routing of x). Each call clears that block when it starts, and all
 *     calls on a device share it, so calls that overlap on the GPU also race
 *     on their error reports: read the status before the next call. */
mok_status mok_route_layout_static(const void* x, const float* W_r, const float* bias,
                                   int32_t T, int32_t H, int32_t E, int32_t k,
                                   int32_t* topk_idx, float* topk_w, int32_t* counts,
                                   int32_t* offsets, int32_t* row_src, int32_t* slot_row,
                                   mok_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Device status                                                               */
/* ------------------------------------------------------------------------- */

/* Synchronises `stream`, then returns the status the last call using
 * `workspace` recorded on the device (MOK_OK, MOK_ERR_TIMEOUT or
 * MOK_ERR_CAPACITY); *detail (if not NULL) receives a code naming the wait
 * that gave up. reset != 0 clears the word afterwards. workspace == NULL
 * reads the status of the last mok_route_layout_static call on the current
 * device (the status block of the library's routing scratch array). */
mok_status mok_device_status(const void* workspace, mok_stream_t stream, int32_t* detail,
                             int32_t reset);

/* Test hook of the routing kernels' bounded waits, for both routing entry
 * points: withhold_copy != 0 makes the first CTA of the top-k kernel skip one
 * of its bulk copies in every following routing call, so its wait runs out
 * after timeout_ms (0 = the default 4 s) and the call records
 * MOK_ERR_TIMEOUT with detail 7 in its status block; the tokens of that CTA
 * then get the lowest-index experts. withhold_copy = 0, timeout_ms = 0
 * restores normal routing. Process-wide and not thread-safe: tests only.
 * Returns MOK_ERR_INVALID for timeout_ms < 0. */
mok_status mok_route_test_hook(int32_t withhold_copy, int32_t timeout_ms);

/* Human-readable name of a status code (static string). */
const char* mok_status_string(mok_status s);

/* Library version string. */
const char* mok_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H */
