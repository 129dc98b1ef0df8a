// Layouts and kernel parameter blocks shared by the host side and the kernels of the
// library (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/moestep.h"

namespace moe {

constexpr int kMaxRows = 64;         // rows per step
constexpr int kMaxK = 16;            // top-k
constexpr int kMaxE = 512;           // routed experts
constexpr int kTileRows = 8;         // route tile height
constexpr int kStepBytes = 128;      // K bytes per pipeline step (one 128-byte swizzle row)
constexpr int kBlockRows = 128;      // weight rows per MMA block (the MMA's M)
constexpr int kAtomBytes = 512;      // scale atom: 128 rows x 4 bytes
constexpr int kMaxGemmCtas = 160;    // GEMM grid cap (one CTA per SM); partial-sum slots are sized for it
constexpr int kPartialFloats = kMaxRows * kBlockRows;  // one partial sum of a unit piece
constexpr int kMaxPieces = 4;        // pieces of a unit cut in the dynamic pool
constexpr int kPoolSlot0 = 2 * kMaxGemmCtas;  // static ranges: 2 slots per CTA; then the pool's
// Partial-sum slots of a workspace: a single-GEMM launch uses [0, kPoolSlot0) for its
// static ranges and, with a counter-fed schedule, the pool's kMaxPieces per CTA after them;
// the one-launch FFN uses [0, kPoolSlot0) for gate_up and the next kPoolSlot0 for down.
__host__ __device__ inline int partial_slots(int schedule) {
    return kPoolSlot0 + (schedule == MOE_SCHED_STATIC ? kPoolSlot0 : kMaxPieces * kMaxGemmCtas);
}
constexpr int kGemmQueue = 16;       // work items in flight between a CTA's roles
constexpr int kMaxStages = 16;       // ring slots of the GEMM pipeline
constexpr int kDeferBytes = kMaxStages * 48;  // producer's deferred copies (shared memory)

__host__ __device__ inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

__host__ __device__ inline int64_t row_bytes(int fmt, int64_t K) {
    return fmt == MOE_FMT_BF16 ? 2 * K : (fmt == MOE_FMT_MXFP8 ? K : K / 2);
}
__host__ __device__ inline int64_t row_scales(int fmt, int64_t K) {
    return (fmt == MOE_FMT_MXFP8 || fmt == MOE_FMT_MXFP4) ? K / 32 : (fmt == MOE_FMT_NVFP4 ? K / 16 : 0);
}
// Scale atoms per 128-byte K step (MXFP8 1, MXFP4 2, NVFP4 4, BF16 0).
__host__ __device__ inline int atoms_per_step(int fmt) {
    return fmt == MOE_FMT_MXFP8 ? 1 : (fmt == MOE_FMT_MXFP4 ? 2 : (fmt == MOE_FMT_NVFP4 ? 4 : 0));
}
__host__ __device__ inline int steps_of(int fmt, int K) { return (int)(row_bytes(fmt, K) / kStepBytes); }
// Packed record: 128 rows x 128 B of codes plus the step's scale atoms.
__host__ __device__ inline int record_bytes(int fmt) {
    return kBlockRows * kStepBytes + atoms_per_step(fmt) * kAtomBytes;
}

// GEMM tensor-memory layout: two accumulator banks (one per MMA issuer), each holding
// nacc buffers of Mpad columns, then the scale factors of every pipeline stage
// (8 columns per scale atom). NVFP4 stages carry 4 atoms, so their banks are kept small.
constexpr int kGemmThreads = 352;  // 11 warps: copies, 2 MMA issuers, 4 epilogue, 4 scale copies
__host__ __device__ inline int acc_bank_cols(int atoms_max, int Mpad) {
    return atoms_max == 4 ? (2 * Mpad > 64 ? 2 * Mpad : 64) : 128;
}

// Group table entry written by the route kernel, one per selected routed expert.
struct Group {
    int32_t expert, rows, perm_off, row_off;  // row_off: padded rows before this group
};

// Workspace header (first 256 bytes of ws).
struct WsHeader {
    int32_t status;
    int32_t num_groups;  // routed groups
    int32_t num_tiles;
    int32_t pad0;
    int32_t err_info[4];
};

// Byte offsets of the workspace regions for a layer and a maximum row count.
struct WsLayout {
    size_t header, groups, logits, scores, topk_idx, topk_w, counts, perm, inv_perm, tiles, num_tiles;
    size_t xq, xs, xq_sh, xs_sh, hq, hs, y, cnt_gu, cnt_dn, partials, sched, gu_done, tcnt, total;
    int max_rows, P_max, G_max, T_max, U_gu, U_dn;
    size_t hq_routed_bytes, hs_routed_bytes;  // shared group's data / scales start here
};

// ---------------------------------------------------------------- kernel parameters
struct RouterParams {
    const uint16_t* x;        // bf16 [M, H]
    const uint16_t* wg;       // bf16 [E, H]
    const float* logits_in;   // [M, E] or null
    float* logits_out;        // [M, E] or null
    float* scores;            // [M, E]
    int M, H, E;
    int32_t* status;          // status word (MOE_ERR_TIMEOUT when a copy wait runs out)
    const uint8_t* l2_pf[2];  // bytes a later launch streams that do not depend on this one
    size_t l2_pf_bytes[2];    // (the shared expert's gate_up and down records): prefetched into L2
    uint64_t wait_ns;         // limit of each copy wait (kRouterWaitNs)
    uint32_t unreachable_tx;  // 0; a test of the timeout path makes the gate rows' barrier expect
                              // this many bytes more than its copies bring, so its wait runs out
};

constexpr uint64_t kRouterWaitNs = 2000000000ull;  // 2 s: limit of the router's copy waits

constexpr int kRouteThreads = 512;  // k_topk_route: 16 warps, one row each

struct TopkRouteParams {
    const float* scores;      // [M, E] (topk stage)
    const float* bias;        // [E] or null
    int32_t* topk_idx;        // [M, k]
    float* topk_w;            // [M, k]
    int M, E, k, renormalize, has_shared, do_topk, do_route;
    int topk_ctas;            // CTAs 0..topk_ctas-1 take the rows (one per warp); the last to finish routes
    int32_t* topk_arrivals;   // their arrival counter (self-resetting; used when topk_ctas > 1 and routing,
                              // or to clear router_status)
    int32_t* router_status;   // or null: a router timeout recorded here (no workspace) makes every row
                              // -1 ids / 0 weights; the last top-k CTA clears it
    float rsf;
    int32_t *counts, *perm, *inv_perm, *tiles, *num_tiles;
    Group* groups;
    WsHeader* hdr;
    // FC1 input quantisation into the tiled layout (CTAs topk_ctas.. of the launch)
    const uint16_t* x;        // bf16 [M, H]
    int H, fmt_r, fmt_s, quant_shared;
    uint8_t *xq, *xs, *xq_sh, *xs_sh;
    float gs_r, gs_s;
    // the last pf_ctas CTAs of the launch (0: none) prefetch these bytes into L2 (records a
    // later launch streams that do not depend on the routing), 128-byte lines spread over
    // their threads
    const uint8_t* l2_pf[2];
    size_t l2_pf_bytes[2];
    int pf_ctas;
};

// k_front: the router launch's and the top-k launch's parameters, plus the per-row-block
// arrival counters of the router CTAs ([ceil(M/8)], self-resetting); t.topk_arrivals counts
// the row blocks whose top-k is done.
struct FrontParams {
    RouterParams r;
    TopkRouteParams t;
    int32_t* rb_arrivals;
};

struct FinalizeParams {
    const float* y;           // [P, H]
    const float* topk_w;      // [M, k]
    const int32_t* inv_perm;  // [M*k + M]
    uint16_t* residual;       // bf16 [M, H]
    const uint16_t* gamma;
    uint16_t* out;
    uint8_t* outq;            // [M8, H] or null
    uint8_t* outs;            // [M8, H/32]
    int M, H, k, has_shared;
    float eps;
};

struct GemmClass {            // one weight class: routed experts or the shared expert
    int fmt;                  // weight / activation format
    const uint8_t* w;         // packed records
    const float* gs_w;        // NVFP4 per-expert global scales or null
    int MB, KS;               // 128-row blocks, 128-byte K steps
    const uint8_t* b;         // tiled B operand base (gate_up: xq; down: hq group region)
    const uint8_t* bs;        // its scales
    float gs_a;               // static global scale of the B operand (NVFP4) or 1
    float gs_out;             // gate_up: static global scale of the NVFP4 output or 1
    int out_fmt;              // gate_up: format of hq
    uint8_t* hq;              // gate_up output base for this class
    uint8_t* hs;
    int I;                    // gate_up: intermediate size of this class
};

struct GemmParams {
    int mode;                 // 0 gate_up, 1 down, 2 both in one launch (gate_up items first)
    int M, k, E, H, Mpad;
    GemmClass cls[2][2];      // [GEMM: 0 gate_up, 1 down][class: 0 routed, 1 shared]
    int has_shared;
    const int32_t* perm;
    const Group* groups;
    const WsHeader* hdr;
    float* y;                 // down output [P, H]
    int32_t* counters[2];     // per GEMM, per unit: pieces finished (self-resetting)
    float* partials[2];       // per GEMM: partial-sum slots (kPartialFloats each)
    int32_t* sched;           // [2]: next work item, CTAs finished (dynamic schedule, self-resetting)
    int32_t* gu_done;         // mode 2: gate_up units finished per group ([kMaxE]: shared expert),
                              // then CTAs finished at [kMaxE + 1] (self-resetting)
    int32_t* status;
    int stages, stage_bytes, a_off, sfa_off, b_off, sfb_off, atoms_max, sf_warps;
    int pool_units;           // units at the end of the list taken from the counter (-1: all)
    float swiglu_limit;       // > 0: clamped SwiGLU in the gate_up epilogue
    int prefetch_shared;      // 1: prefetch the shared expert's records into L2 before the wait
    uint64_t wait_ns;         // limit of every wait (2 s)
    int dep_extra;            // 0; 1 makes the down items' counter targets unreachable (a test
                              // of the timeout path, never set by the public calls)
};


struct PackParams {
    const uint8_t* codes;
    const uint8_t* scales;
    uint8_t* dst;
    int fmt, n_exp, rows, K, gate_up;  // gate_up: interleave gate/up halves per block
    int I;                              // gate_up: intermediate size
};

}  // namespace moe
