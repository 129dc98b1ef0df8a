/*
 * moestep.h - C ABI of the GB300 (sm_103a) small-M MoE decode/verify layer step.
 *
 * The step (1..64 rows) follows the MoE slots of the "SGLang-NVIDIA-Mega" README
 * (slot table of "What a covered DeepSeek-V4.1-Flash step runs": rows gate, moe,
 * shared_ll and hop_b; Qwen3.5 slot tables: rows route and mkm) and the routing pinned
 * by "sgl-nvidia-mega pull request 24" ("Modifications / Target spec": one expert
 * group, sigmoid scores, renormalised top-k). The routed sum takes a
 * routed_scaling_factor ("SGLang Spark GB10 Optimizations", "Key Optimizations 1").
 *
 *   a1 router GEMV      logits[m,e] = sum_h x[m,h] * Wg[e,h]         (bf16 in, fp32 out)
 *   a2 scoring / top-k  s = sigmoid(logit) (fp32 rounding of the double value);
 *                       key = s (+ bias[e]); top-k by key, ties to the lower index;
 *                       w_j = s_j / sum_j s_j * routed_scaling_factor
 *   a3 FC1 input quant  x -> MXFP8 (E4M3 + E8M0 per 32) or NVFP4 (E2M1 + E4M3 per 16
 *                       with a static fp32 global scale)
 *   a4 route            stable counting sort of the M*k (row, slot) pairs by expert into
 *                       8-row tiles; the shared expert is expert E with all M rows
 *   a5 gate_up          per selected expert: g = W_gate x, u = W_up x (block-scaled MMA),
 *                       h = silu(g) * u, requantised for FC2
 *   a6 down             y_pair = W_down h
 *   a7 finalize         residual' = bf16(residual + sum_j w_j y_j + y_shared);
 *                       out = bf16(RMSNorm(residual') * gamma); optional MXFP8 of out
 *
 * Conventions
 *  - Every call returns a moe_status and validates all of its arguments before it
 *    launches anything; a violation returns MOE_ERR_INVALID_ARG (a shape or pointer
 *    rule) or MOE_ERR_UNSUPPORTED (a format or size without a kernel), with the reason
 *    in moe_last_error_string() (thread-local). Nothing is launched in that case.
 *  - Calls are asynchronous on the given stream: no host synchronisation and no
 *    allocation inside (moe_get_status is the one call that synchronises).
 *  - All buffers are device memory owned by the caller (e.g. PyTorch tensors); the
 *    library owns no device memory. Pointers must be 16-byte aligned.
 *  - Device-side failures (a pipeline wait that exceeds its time limit, an expert id
 *    out of range) are recorded in the workspace status word; read it with
 *    moe_get_status. The kernels never trap.
 *  - A step's launches are chained with programmatic dependent launch and the whole
 *    moe_step may be captured into a CUDA graph.
 *
 * Formats and layouts
 *  - bf16 tensors are row-major; x and residual are [M, H]; Wg is [E, H]; gamma is [H].
 *  - Canonical expert weights (inputs of moe_pack_weights), per projection:
 *      codes  [n_exp][rows][row_bytes]  MXFP8: 1 byte/element (E4M3);
 *                                       NVFP4, MXFP4: 2 E2M1 elements/byte, low nibble =
 *                                       even element; BF16: 2 bytes/element
 *      scales [n_exp][rows][K/32] E8M0 (MXFP8, MXFP4) or [n_exp][rows][K/16] E4M3 (NVFP4)
 *      W13 rows: gate rows 0..I-1, then up rows I..2I-1, K = H.   W2 rows: H, K = I.
 *      NVFP4 global scales: fp32 [n_exp] per projection (passed to the GEMM calls).
 *  - Packed weights (outputs of moe_pack_weights): one record per (expert, 128-row
 *    block, 128-byte K step), records of one block contiguous. A record holds the
 *    block's 128 x 128 B codes in the 128-byte swizzled shared-memory image (16-byte
 *    chunk c of row r at chunk position c ^ (r & 7)), followed by its block scales as
 *    512-byte atoms (MXFP8: 1 atom of the four E8M0 scales of the step; MXFP4: 2 atoms of
 *    four E8M0 scales each, one per two 64-element MMA steps; NVFP4: 4 atoms of four E4M3
 *    scales each, one per 64-element MMA step), row r's four bytes at
 *    offset (r % 32) * 16 + (r / 32) * 4. W13 blocks interleave 64 gate rows and the
 *    64 matching up rows.
 *  - Tiled activations (xq, and the hidden activations of a selected expert): rows are
 *    padded to R_pad = round_up(rows, 16) with zeros; the row bytes are cut into
 *    128-byte K steps; step s holds R_pad rows x 128 B in the same swizzled image, then
 *    (scaled formats) the step's scale atoms laid out as for the weights (row r's bytes
 *    at (r % 32) * 16 + (r / 32) * 4 in each 512-byte atom) in a separate scale buffer.
 *    Sizes: moe_act_bytes / moe_act_scale_bytes.
 */
#ifndef MOESTEP_H
#define MOESTEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL is the legacy default stream */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_CUDA = 3,
    MOE_ERR_TIMEOUT = 4
} moe_status;

typedef enum { MOE_FMT_BF16 = 0, MOE_FMT_MXFP8 = 1, MOE_FMT_NVFP4 = 2, MOE_FMT_MXFP4 = 3 } moe_fmt;

typedef enum { MOE_W13 = 0, MOE_W2 = 1, MOE_SH13 = 2, MOE_SH2 = 3 } moe_proj;

/* How the expert GEMM launches hand their work to the CTAs (moe_layer_desc.gemm_schedule).
 * STATIC: the units' K steps are cut into equal contiguous ranges, one per CTA (the
 * default; the fastest on GB300). HYBRID: the last 2 units per CTA are taken from an
 * atomic counter by whichever CTA finishes its range first. DYNAMIC: every unit is taken
 * from the counter. All three are deterministic and agree with each other up to the fp32
 * summation order of a unit cut into pieces. The one-launch FFN always runs STATIC. */
typedef enum { MOE_SCHED_STATIC = 0, MOE_SCHED_HYBRID = 1, MOE_SCHED_DYNAMIC = 2 } moe_schedule;

/* One MoE layer. Limits: 1 <= k <= 16, k <= E <= 512; H % 256 == 0 and 1024 <= H <= 8192;
 * I, I_shared % 256 == 0 and 256 <= I <= 4096. w_fmt is MXFP8, NVFP4 or MXFP4; shared_fmt is
 * BF16, MXFP8, NVFP4 or MXFP4. gs_a1 / gs_a2 are the static NVFP4 global scales of the routed
 * experts' FC1 and FC2 inputs (gs_a1_shared / gs_a2_shared for the shared expert);
 * they are ignored for other formats. swiglu_limit > 0 selects the clamped SwiGLU of the
 * routed and the shared experts ("SGLang-NVIDIA-Mega" README, shared_ll row): the gate
 * is cut to min(g, L) and the up projection to clamp(u, -L, L) before silu(g) * u, with
 * L = swiglu_limit; 0 (or any value <= 0) is the plain SwiGLU; NaN is rejected.
 * Execution choices, fixed when the layer is set up (the pages' engines choose their
 * kernels and tactics at load, "SGLang-NVIDIA-Mega" README, Design): gemm_schedule is a
 * moe_schedule (0 = STATIC); ffn_launches is 0 or 1 for gate_up and down in one launch in
 * moe_step (the default), 2 for two launches; front_launches is 0 or 2 for the router
 * launch followed by the top-k / routing / quantisation launch (the default: on GB300 the
 * faster of the two), 1 for all four in one launch (the same bytes). A workspace serves
 * only descriptors whose moe_workspace_bytes it was sized with (the schedule changes the
 * size). */
typedef struct {
    int32_t H, E, k, I, I_shared;
    int32_t w_fmt, shared_fmt;
    int32_t has_shared, has_bias, renormalize, emit_next_mxfp8;
    float routed_scaling_factor, rms_eps;
    float gs_a1, gs_a2, gs_a1_shared, gs_a2_shared;
    float swiglu_limit;
    int32_t gemm_schedule, ffn_launches, front_launches;
} moe_layer_desc;

/* A packed projection: the moe_pack_weights output and, for NVFP4, the fp32 global
 * scale of each expert (NULL otherwise). */
typedef struct {
    const void* packed;
    const float* global_scale;
} moe_qweight;

/* Everything one moe_step reads and writes (device pointers). Intermediates live in
 * the workspace; moe_ws_view returns their addresses. */
typedef struct {
    const void* x;          /* bf16 [M, H] */
    const void* w_gate;     /* bf16 [E, H] */
    const float* bias;      /* fp32 [E] or NULL (selection bias, has_bias) */
    moe_qweight w13, w2;    /* routed experts */
    moe_qweight sh13, sh2;  /* shared expert (has_shared) */
    void* residual;         /* bf16 [M, H], read, then overwritten with residual + moe */
    const void* gamma;      /* bf16 [H] */
    void* out;              /* bf16 [M, H] */
    void* outq;             /* E4M3 [round_up(M,8), H] or NULL (emit_next_mxfp8) */
    void* outq_scales;      /* E8M0 [round_up(M,8), H/32] or NULL */
} moe_step_args;

/* Device addresses of the intermediates that moe_step keeps in the workspace. */
typedef struct {
    int32_t* status;        /* the device status word (moe_status value) */
    float* logits;          /* [M, E] */
    float* scores;          /* [M, E] sigmoid scores */
    int32_t* topk_idx;      /* [M, k] */
    float* topk_w;          /* [M, k] */
    int32_t* expert_counts; /* [E+1] */
    int32_t* perm;          /* [M*k + M] */
    int32_t* inv_perm;      /* [M*k + M] */
    int32_t* tiles;         /* [M*k + M + E + 1][3] */
    int32_t* num_tiles;     /* [1] */
    void* xq;               /* tiled routed FC1 input */
    void* xq_scales;
    void* xq_shared;        /* tiled shared FC1 input (same as xq when the formats agree) */
    void* xq_shared_scales;
    void* hq;               /* tiled FC2 inputs, one block per selected expert */
    void* hq_scales;
    float* y_pairs;         /* [M*k + M, H] fp32, rows in perm order */
} moe_ws_ptrs;

/* Reason for the last failure on this thread ("" if none). Owned by the library. */
const char* moe_last_error_string(void);

/* ---- sizes ------------------------------------------------------------------ */
/* Bytes of the packed image of projection `which` (all experts). 0 on bad input. */
size_t moe_packed_bytes(const moe_layer_desc* d, int which);
/* Bytes of a tiled activation of `rows` rows and K elements in `fmt` (codes / scales). */
size_t moe_act_bytes(int fmt, int rows, int K);
size_t moe_act_scale_bytes(int fmt, int rows, int K);
/* Bytes of the hidden-activation buffers (codes / scales) for up to max_rows rows. */
size_t moe_hq_bytes(const moe_layer_desc* d, int max_rows);
size_t moe_hq_scale_bytes(const moe_layer_desc* d, int max_rows);
/* Bytes of the workspace of a layer (sized for steps of up to 64 rows; tens of MB: the
 * largest parts are the fp32 per-pair FC2 rows and the stream-K partial sums). 0 on bad
 * input. One workspace serves one stream: calls that overlap on the GPU must not share it. */
size_t moe_workspace_bytes(const moe_layer_desc* d);

/* Zero a new workspace (status word, stream-K counters). Must run once before first use
 * and again after a step reported MOE_ERR_TIMEOUT. */
moe_status moe_workspace_init(const moe_layer_desc* d, void* ws, moe_stream_t stream);
/* Fill `out` with the addresses of the intermediates inside `ws`. Host-only. */
moe_status moe_ws_view(const moe_layer_desc* d, void* ws, moe_ws_ptrs* out);

/* ---- load time -------------------------------------------------------------- */
/* Repack one projection from the canonical layout (codes, scales; scales NULL for BF16)
 * into the streaming record layout above, for all experts of the projection (E for
 * W13/W2, 1 for SH13/SH2). dst holds moe_packed_bytes(d, which) bytes. The pages'
 * engines read routed weights from records derived at load ("sgl-nvidia-mega pull
 * request 24", Target spec, compact FC2 records); this is that step for these kernels. */
moe_status moe_pack_weights(const moe_layer_desc* d, int which, const void* codes, const void* scales,
                            void* dst, moe_stream_t stream);

/* ---- the step, call by call ---------------------------------------------------- */
/* a1 + a2 + a3. Router GEMV (skipped when logits_in != NULL), fp32 sigmoid through
 * double, optional selection bias, top-k with ties to the lower index, renormalised
 * weights; quantises x for the routed FC1 (xq, xq_scales, in w_fmt) and, when the
 * shared expert's format differs, for the shared FC1 (xq_sh, xq_sh_scales; BF16 has no
 * scales). x bf16 [M,H], w_gate bf16 [E,H], bias fp32 [E] | NULL, logits_in fp32 [M,E]
 * | NULL; outputs logits_out fp32 [M,E] | NULL, topk_idx int32 [M,k], topk_w fp32 [M,k].
 * The GEMV's copy waits are bounded: one that runs out (2 s) sets MOE_ERR_TIMEOUT in the
 * workspace status word and leaves the outputs unwritten.
 * [README: gate row; Qwen3.5 route row; PR24 Target spec] */
moe_status moe_router_topk(const moe_layer_desc* d, const void* x, const void* w_gate, const float* bias,
                           const float* logits_in, int M, float* logits_out, int32_t* topk_idx,
                           float* topk_w, void* xq, void* xq_scales, void* xq_sh, void* xq_sh_scales,
                           void* ws, moe_stream_t stream);

/* a4. Routes the M*k pairs of topk_idx (int32 [M,k], values in [0,E)) into 8-row tiles:
 * expert_counts [E+1] (the last entry is the shared expert's M, or 0), perm / inv_perm
 * [M*k + M] (pair id m*k+j; shared pair ids M*k+m), tiles [M*k+M+E+1][3] as (expert,
 * start in perm, rows 1..8), num_tiles [1]. Also writes the per-expert group table the
 * GEMM calls read from ws. Out-of-range ids set the status word to MOE_ERR_INVALID_ARG
 * and produce no tiles. [README: moe row: "an expert chosen by more than 8 rows takes
 * several tiles"] */
moe_status moe_route_tiles(const moe_layer_desc* d, const int32_t* topk_idx, int M, int32_t* tiles,
                           int32_t* num_tiles, int32_t* perm, int32_t* inv_perm, int32_t* expert_counts,
                           void* ws, moe_stream_t stream);

/* a5. For every expert group recorded in ws by moe_route_tiles: block-scaled FC1
 * (tcgen05, weights as the 128-row operand, the rows as N), SwiGLU and requantisation to
 * the FC2 input format, written as one tiled block per group into hq / hq_scales
 * (moe_hq_bytes / moe_hq_scale_bytes). xq / xq_sh are the tiled FC1 inputs from
 * moe_router_topk. [README: moe and shared_ll rows; Qwen3.5 mkm row] */
moe_status moe_expert_gate_up(const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13,
                              const void* xq, const void* xq_scales, const void* xq_sh,
                              const void* xq_sh_scales, const int32_t* perm, int M, void* hq,
                              void* hq_scales, void* ws, moe_stream_t stream);

/* a6. For every group: y = W_down h (block-scaled tcgen05), written fp32 to y_pairs
 * [M*k + M, H] at the pairs' perm positions (shared rows at M*k + m). */
moe_status moe_expert_down(const moe_layer_desc* d, const moe_qweight* w2, const moe_qweight* sh2,
                           const void* hq, const void* hq_scales, int M, float* y_pairs, void* ws,
                           moe_stream_t stream);

/* a5 + a6 in one launch: the same bytes in hq, hq_scales and y_pairs as
 * moe_expert_gate_up followed by moe_expert_down, with the arguments of both. A down unit
 * starts as soon as every FC1 unit of its group is done (per-group counters in ws, which
 * every launch leaves at zero), and its weight copies go out before that, so the FC2
 * weights stream while the last FC1 units finish. The grid is one CTA per SM and relies on
 * all of them being resident together; a wait that runs out (2 s) sets MOE_ERR_TIMEOUT in
 * the status word and the launch returns. moe_step uses this launch unless the layer's
 * ffn_launches is 2. [README: moe and shared_ll rows] */
moe_status moe_expert_ffn(const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13,
                          const moe_qweight* w2, const moe_qweight* sh2, const void* xq, const void* xq_scales,
                          const void* xq_sh, const void* xq_sh_scales, const int32_t* perm, int M, void* hq,
                          void* hq_scales, float* y_pairs, void* ws, moe_stream_t stream);

/* a7. moe[m] = sum_j topk_w[m,j] * y_pairs[inv_perm[m*k+j]] (j ascending) + shared row;
 * residual (bf16 [M,H], in place) = bf16(residual + moe); out = bf16(residual *
 * rsqrt(mean(residual^2) + eps) * gamma); outq / outq_scales (optional) = MXFP8 of out,
 * [round_up(M,8), H] and [round_up(M,8), H/32], padding rows zero. [README: hop_b row] */
moe_status moe_finalize_norm(const moe_layer_desc* d, const float* y_pairs, const float* topk_w,
                             const int32_t* inv_perm, int M, void* residual, const void* gamma, void* out,
                             void* outq, void* outq_scales, void* ws, moe_stream_t stream);

/* a1..a7 in four launches chained with programmatic dependent launch: the router GEMV, the
 * top-k / routing / FC1 input quantisation (whose extra CTAs also prefetch the shared
 * expert's weight records into L2), moe_expert_ffn (FC1 and FC2 in one launch), and the
 * finalize. The layer's front_launches = 1 runs the first two as one launch;
 * ffn_launches = 2 runs FC1 and FC2 as two launches. Intermediates in ws (see moe_ws_view).
 * M in [1, 64]. Capture-safe. */
moe_status moe_step(const moe_layer_desc* d, const moe_step_args* a, int M, void* ws, moe_stream_t stream);

/* The router step (a1 + a2 + a3, as moe_router_topk) for callers that cannot give the
 * library any device memory: a host framework that owns every allocation and offers
 * plugins no allocator, or a serving loop that must not allocate once running (an
 * allocation can synchronise the device or fail under memory pressure). The pages have no
 * counterpart: their engines allocate their buffers at load.
 *  - Takes no workspace and allocates nothing: its scratch (a 256-byte header and the
 *    scores of up to 64 rows x 512 experts in fp32: 131,328 bytes, 128 KiB + 256 B) is one
 *    fixed array inside the library, held by every GPU that loads the library until the
 *    process exits. Inputs and outputs are the caller's, exactly as for moe_router_topk,
 *    and the results are the same, for every layer moe_router_topk accepts.
 *  - The first call on a device looks up the array's device address (with that device
 *    current); make that first call before any stream capture.
 *  - Every call uses the same array and it keeps the last call's contents (each call
 *    clears the counters it needs at zero). Calls that overlap on the GPU race: issue them
 *    on one stream, or order them.
 *  - Device-side status has no workspace to go to. If a router copy wait runs out (2 s),
 *    the call writes -1 expert ids and zero weights for every row instead of results, and
 *    leaves the scratch ready for the next call. Host-side errors are returned as usual. */
moe_status moe_router_topk_noalloc(const moe_layer_desc* d, const void* x, const void* w_gate, const float* bias,
                                   const float* logits_in, int M, float* logits_out, int32_t* topk_idx,
                                   float* topk_w, void* xq, void* xq_scales, void* xq_sh, void* xq_sh_scales,
                                   moe_stream_t stream);

/* Synchronises `stream` and reads the workspace status word into *dev_status. */
moe_status moe_get_status(void* ws, moe_stream_t stream, int* dev_status);

#ifdef __cplusplus
}
#endif
#endif /* MOESTEP_H */
