// plan.cuh - minibatch plan of the persistent forward megakernel.
//
// The pages (KuCoin article on MoK, section 02) hand tokens to the experts in
// minibatches: big enough that every compute SM gets work ("at least two full
// waves"), small enough that computing starts early, staged through a
// fixed-size ring token buffer that is reused as soon as its tokens have been
// consumed, with no CPU decision in the loop. On one GPU the plan is built on
// the device from the routing, so the host never waits for counts:
//   - the tokens of each macro-batch are cut, in order, into minibatches whose
//     padded expert-contiguous rows fit one half of the ring (ring regions
//     alternate between minibatches) and whose token count stays within the
//     configured maximum;
//   - for every (minibatch, expert): its rows (a contiguous sub-range of the
//     expert's segment of the batch's layout, because rows are ordered by
//     token within an expert), its padded offset inside the ring region, and
//     the prefix of its 128-row tiles;
//   - the compute phases in the order G1(0), G1(1), G2(0), G1(2), G2(1), ...,
//     G2(n-1) (gate/up GEMM of minibatch i+1 is queued before the down GEMM
//     of minibatch i), with the prefix of their tile counts.
#pragma once

#include "common.cuh"

namespace mok {

constexpr int kMaxMinibatches = 1024;
constexpr int kMaxBatches = 32;

struct MbInfo {
    int batch;    // macro-batch index
    int t0, t1;   // token range within the batch
    int rows;     // padded ring rows
    int mtiles;   // 128-row tiles (sum over experts)
    int region;   // ring / h region (0 or 1)
    int pad[2];
};

struct PlanHeader {
    int n_mb;          // minibatches
    int n_phase;       // compute phases
    int total_tiles;   // tiles over all phases
    int error;         // nonzero: a ring region cannot hold one token block
};

// Device plan, laid out in the workspace.
struct PlanView {
    PlanHeader* hdr;
    MbInfo* mb;           // [kMaxMinibatches]
    int* cnt;             // [kMaxMinibatches * E] rows of expert e in mb
    int* src0;            // [kMaxMinibatches * E] first index into the batch's row_src
    int* roff;            // [kMaxMinibatches * E] padded row offset inside the region
    int* mtoff;           // [kMaxMinibatches * (E + 1)] prefix of 128-row tiles
    int* phase_kind;      // [2 * kMaxMinibatches] 0 = gate/up, 1 = down
    int* phase_mb;        // [2 * kMaxMinibatches]
    int* phase_toff;      // [2 * kMaxMinibatches + 1]
};

inline size_t plan_bytes(int E) {
    size_t b = 256 + sizeof(MbInfo) * kMaxMinibatches;
    b += (size_t)kMaxMinibatches * E * 4 * 3;
    b += (size_t)kMaxMinibatches * (E + 1) * 4;
    b += (size_t)(2 * kMaxMinibatches) * 4 * 2 + (2 * kMaxMinibatches + 1) * 4;
    return (size_t)align_up((int64_t)b, 1024);
}

inline PlanView plan_view(void* base, int E) {
    char* p = static_cast<char*>(base);
    PlanView v;
    v.hdr = reinterpret_cast<PlanHeader*>(p); p += 256;
    v.mb = reinterpret_cast<MbInfo*>(p); p += sizeof(MbInfo) * kMaxMinibatches;
    v.cnt = reinterpret_cast<int*>(p); p += (size_t)kMaxMinibatches * E * 4;
    v.src0 = reinterpret_cast<int*>(p); p += (size_t)kMaxMinibatches * E * 4;
    v.roff = reinterpret_cast<int*>(p); p += (size_t)kMaxMinibatches * E * 4;
    v.mtoff = reinterpret_cast<int*>(p); p += (size_t)kMaxMinibatches * (E + 1) * 4;
    v.phase_kind = reinterpret_cast<int*>(p); p += (size_t)2 * kMaxMinibatches * 4;
    v.phase_mb = reinterpret_cast<int*>(p); p += (size_t)2 * kMaxMinibatches * 4;
    v.phase_toff = reinterpret_cast<int*>(p);
    return v;
}

// Everything one megakernel launch needs (host side).
struct MegaLaunch {
    bool mx;
    int E, H, I, k, T, nbatch;
    const void* x[kMaxBatches];
    const int32_t* offsets[kMaxBatches];
    const int32_t* row_src[kMaxBatches];
    const float* topk_w[kMaxBatches];
    void* partials[kMaxBatches];
    const float* shared[kMaxBatches];
    void* out[kMaxBatches];
    const void* gu;          // packed gate/up [E*2I, H]
    const void* dn;          // packed down [E*H, I]
    const uint8_t* gu_sf;
    const uint8_t* dn_sf;
    void* scratch;           // mega_scratch_bytes
    int region_rows;         // rows of each of the two ring regions (multiple of 128)
    int max_tokens;          // tokens per minibatch at most (tile cuts: rows <= max_tokens * k)
    bool tile_cuts;          // minibatches are runs of 128-row expert tiles (else token ranges)
    int n_movers;            // mover CTAs
    int grid;                // CTAs (<= SMs)
    int test_flags;          // MOK_FLAG_TEST_* bits
    unsigned long long* trace;   // MOK_FLAG_TRACE: one 8 x u64 record per CTA, else NULL
    StatusBlock* status;
    unsigned long long timeout_ns;
};

// The scratch starts with the trace records (kMegaTraceBytes), then the plan,
// counters, ring and h regions.
constexpr int kMegaTraceCtas = 1024;
constexpr size_t kMegaTraceBytes = (size_t)kMegaTraceCtas * 64;
size_t mega_scratch_bytes(int nbatch, int T, int H, int I, int E, int k, int region_rows, bool mx);
cudaError_t launch_mega(const MegaLaunch& L, cudaStream_t s);

}  // namespace mok
