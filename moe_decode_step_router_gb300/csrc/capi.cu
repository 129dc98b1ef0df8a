// Host side of the C ABI declared in include/moestep.h: argument validation, workspace
// layout, launch configuration and the programmatic-dependent-launch chain.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace moe {
__global__ void k_router(RouterParams p);
__global__ void k_router_rows(RouterParams p);
__global__ void k_topk_route(TopkRouteParams p);
__global__ void k_front(FrontParams f);
__global__ void k_finalize(FinalizeParams p);
__global__ void k_pack(PackParams p);
__global__ void k_expert_gemm(const __grid_constant__ GemmParams p);
}  // namespace moe

using namespace moe;

namespace {

thread_local std::string g_err;

moe_status fail(moe_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

moe_status ok() {
    g_err.clear();
    return MOE_OK;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, ...)                                            \
    do {                                                              \
        if (!(cond)) return fail(MOE_ERR_INVALID_ARG, __VA_ARGS__);   \
    } while (0)
#define REQUIRE_PTR(p, name)                                                         \
    do {                                                                             \
        if (!(p)) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);              \
        if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)
#define OPT_PTR(p, name)                                                             \
    do {                                                                             \
        if ((p) && !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

moe_status check_desc(const moe_layer_desc* d) {
    if (!d) return fail(MOE_ERR_INVALID_ARG, "layer descriptor is NULL");
    REQUIRE(d->H >= 1024 && d->H <= 8192 && d->H % 256 == 0, "H=%d: need 1024 <= H <= 8192, H %% 256 == 0", d->H);
    REQUIRE(d->E >= 1 && d->E <= kMaxE, "E=%d: need 1 <= E <= %d", d->E, kMaxE);
    REQUIRE(d->k >= 1 && d->k <= kMaxK && d->k <= d->E, "k=%d: need 1 <= k <= min(16, E)", d->k);
    REQUIRE(d->I >= 256 && d->I <= 4096 && d->I % 256 == 0, "I=%d: need 256 <= I <= 4096, I %% 256 == 0", d->I);
    if (d->w_fmt != MOE_FMT_MXFP8 && d->w_fmt != MOE_FMT_NVFP4 && d->w_fmt != MOE_FMT_MXFP4)
        return fail(MOE_ERR_UNSUPPORTED, "routed weight format %d has no kernel (MXFP8=1, NVFP4=2, MXFP4=3)",
                    d->w_fmt);
    if (d->has_shared) {
        REQUIRE(d->I_shared >= 256 && d->I_shared <= 4096 && d->I_shared % 256 == 0,
                "I_shared=%d: need 256 <= I_shared <= 4096, %% 256 == 0", d->I_shared);
        if (d->shared_fmt < MOE_FMT_BF16 || d->shared_fmt > MOE_FMT_MXFP4)
            return fail(MOE_ERR_UNSUPPORTED, "shared weight format %d has no kernel", d->shared_fmt);
    }
    REQUIRE(d->routed_scaling_factor == d->routed_scaling_factor, "routed_scaling_factor is NaN");
    REQUIRE(d->rms_eps >= 0.0f, "rms_eps must be >= 0");
    REQUIRE(d->swiglu_limit == d->swiglu_limit, "swiglu_limit must not be NaN");
    REQUIRE(d->gemm_schedule >= MOE_SCHED_STATIC && d->gemm_schedule <= MOE_SCHED_DYNAMIC,
            "gemm_schedule=%d: need 0 (static), 1 (hybrid) or 2 (dynamic)", d->gemm_schedule);
    REQUIRE(d->ffn_launches >= 0 && d->ffn_launches <= 2, "ffn_launches=%d: need 0, 1 or 2", d->ffn_launches);
    REQUIRE(d->front_launches >= 0 && d->front_launches <= 2, "front_launches=%d: need 0, 1 or 2",
            d->front_launches);
    if (d->w_fmt == MOE_FMT_NVFP4) REQUIRE(d->gs_a1 > 0.0f && d->gs_a2 > 0.0f, "NVFP4 needs gs_a1, gs_a2 > 0");
    if (d->has_shared && d->shared_fmt == MOE_FMT_NVFP4)
        REQUIRE(d->gs_a1_shared > 0.0f && d->gs_a2_shared > 0.0f, "NVFP4 shared needs gs_a1_shared, gs_a2_shared > 0");
    return MOE_OK;
}

int shared_fmt_of(const moe_layer_desc* d) { return d->has_shared ? d->shared_fmt : d->w_fmt; }
bool separate_shared_input(const moe_layer_desc* d) { return d->has_shared && d->shared_fmt != d->w_fmt; }

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

size_t act_bytes(int fmt, int rows, int K) { return (size_t)round_up(rows, 16) * row_bytes(fmt, K); }
size_t act_scale_bytes(int fmt, int K) { return (size_t)steps_of(fmt, K) * atoms_per_step(fmt) * kAtomBytes; }

// Routed part of the hidden buffers for up to `rows` rows; the shared block follows it.
size_t hq_routed(const moe_layer_desc* d, int rows) {
    const int P = rows * d->k, G = P < d->E ? P : d->E;
    return al256((size_t)(P + 15 * G) * row_bytes(d->w_fmt, d->I));
}
size_t hs_routed(const moe_layer_desc* d, int rows) {
    const int P = rows * d->k, G = P < d->E ? P : d->E;
    return al256((size_t)G * act_scale_bytes(d->w_fmt, d->I));
}
size_t hq_total(const moe_layer_desc* d, int rows) {
    return hq_routed(d, rows) + (d->has_shared ? al256(act_bytes(d->shared_fmt, rows, d->I_shared)) : 0);
}
size_t hs_total(const moe_layer_desc* d, int rows) {
    return hs_routed(d, rows) + (d->has_shared ? al256(act_scale_bytes(d->shared_fmt, d->I_shared)) + 256 : 256);
}

WsLayout layout(const moe_layer_desc* d) {
    const int max_rows = kMaxRows;
    WsLayout L{};
    L.max_rows = max_rows;
    L.P_max = max_rows * d->k + max_rows;
    L.G_max = (max_rows * d->k < d->E) ? max_rows * d->k : d->E;
    L.T_max = L.P_max + d->E + 1;
    const int Ish = d->has_shared ? d->I_shared : 256;
    L.U_gu = L.G_max * (2 * d->I / kBlockRows) + 2 * Ish / kBlockRows;
    L.U_dn = L.G_max * (d->H / kBlockRows) + d->H / kBlockRows;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t r = o;
        o = al256(o + bytes);
        return r;
    };
    L.header = take(256);
    L.groups = take(sizeof(Group) * (size_t)L.G_max);
    L.logits = take(4ull * max_rows * d->E);
    L.scores = take(4ull * max_rows * d->E);
    L.topk_idx = take(4ull * max_rows * d->k);
    L.topk_w = take(4ull * max_rows * d->k);
    L.counts = take(4ull * (d->E + 1));
    L.perm = take(4ull * L.P_max);
    L.inv_perm = take(4ull * L.P_max);
    L.tiles = take(12ull * L.T_max);
    L.num_tiles = take(4);
    L.xq = take(act_bytes(d->w_fmt, max_rows, d->H));
    L.xs = take(act_scale_bytes(d->w_fmt, d->H) + 256);
    if (separate_shared_input(d)) {
        L.xq_sh = take(act_bytes(d->shared_fmt, max_rows, d->H));
        L.xs_sh = take(act_scale_bytes(d->shared_fmt, d->H) + 256);
    } else {
        L.xq_sh = L.xq;
        L.xs_sh = L.xs;
    }
    L.hq_routed_bytes = hq_routed(d, max_rows);
    L.hs_routed_bytes = hs_routed(d, max_rows);
    L.hq = take(hq_total(d, max_rows));
    L.hs = take(hs_total(d, max_rows));
    L.y = take(4ull * L.P_max * d->H);
    L.cnt_gu = take(4ull * L.U_gu);
    L.cnt_dn = take(4ull * L.U_dn);
    L.partials = take(4ull * partial_slots(d->gemm_schedule) * kPartialFloats);
    L.sched = take(4ull * 4);  // gate_up and down: next work item, CTAs finished
    L.gu_done = take(4ull * (kMaxE + 2));  // one launch for both GEMMs: per-group gate_up units done
    L.tcnt = take(64);  // arrival counters: [0] top-k CTAs / row blocks, [4 ..) router CTAs per row block
    L.total = o;
    return L;
}

struct DevInfo {
    int dev = -1, sms = 0, smem_optin = 0;
    bool gemm_attr_set = false;
    bool router_rows_attr_set = false;
    bool front_attr_set = false;
};
thread_local DevInfo g_dev;

moe_status dev_info(DevInfo** out) {
    int dev;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (g_dev.dev != dev) {
        g_dev = DevInfo{};
        g_dev.dev = dev;
        e = cudaDeviceGetAttribute(&g_dev.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        e = cudaDeviceGetAttribute(&g_dev.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3) {
            g_dev.dev = -1;
            return fail(MOE_ERR_UNSUPPORTED, "device %d is sm_%d%d; the kernels are built for sm_103a", dev, major,
                        minor);
        }
    }
    *out = &g_dev;
    return MOE_OK;
}

// Launch with programmatic stream serialisation (the kernel may start before its
// predecessor on the stream finishes; it waits in griddepcontrol.wait).
template <typename Kern, typename Arg>
moe_status launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Arg& arg,
                      const char* name, bool cooperative = false) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // blocks that wait on one another: all of them resident at once, or no launch
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, arg);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return MOE_OK;
}

// ------------------------------------------------------------------ launch helpers
RouterParams router_params(const moe_layer_desc* d, const void* x, const void* w_gate, const float* logits_in, int M,
                           float* logits_out, float* scores, int32_t* status, const void* l2_pf = nullptr,
                           size_t l2_pf_bytes = 0, const void* l2_pf2 = nullptr, size_t l2_pf2_bytes = 0) {
    RouterParams p{};
    p.status = status;
    p.wait_ns = kRouterWaitNs;
    p.unreachable_tx = 0;
    p.l2_pf[0] = static_cast<const uint8_t*>(l2_pf);
    p.l2_pf_bytes[0] = l2_pf_bytes;
    p.l2_pf[1] = static_cast<const uint8_t*>(l2_pf2);
    p.l2_pf_bytes[1] = l2_pf2_bytes;
    p.x = static_cast<const uint16_t*>(x);
    p.wg = static_cast<const uint16_t*>(w_gate);
    p.logits_in = logits_in;
    p.logits_out = logits_out;
    p.scores = scores;
    p.M = M;
    p.H = d->H;
    p.E = d->E;
    return p;
}

// Dynamic shared memory of a router CTA: its 4 gate rows and up to 8 x rows of H bf16, each
// padded by 8 elements ((4 + 8) * (H + 8) * 2 <= 192.2 KB).
size_t router_smem(const moe_layer_desc* d, int M) { return (size_t)(4 + (M < 8 ? M : 8)) * (d->H + 8) * 2; }

moe_status launch_router(const moe_layer_desc* d, const void* x, const void* w_gate, const float* logits_in, int M,
                         float* logits_out, float* scores, int32_t* status, cudaStream_t st,
                         const void* l2_pf = nullptr, size_t l2_pf_bytes = 0, const void* l2_pf2 = nullptr,
                         size_t l2_pf2_bytes = 0, uint64_t wait_ns = kRouterWaitNs, uint32_t unreachable_tx = 0) {
    RouterParams p = router_params(d, x, w_gate, logits_in, M, logits_out, scores, status, l2_pf, l2_pf_bytes, l2_pf2,
                                   l2_pf2_bytes);
    p.wait_ns = wait_ns;
    p.unreachable_tx = unreachable_tx;
    DevInfo* di;
    moe_status s = dev_info(&di);
    if (s != MOE_OK) return s;
    // the GEMV: CTAs of 4 experts x 8 rows over the whole of H (512 threads, as in k_front,
    // so both give the same logits), x rows and gate rows in shared memory (plus ~2 KB of
    // static shared memory)
    if (!logits_in) {
        if (!di->router_rows_attr_set) {
            cudaError_t e = cudaFuncSetAttribute(k_router_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 di->smem_optin - 4096);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(k_router_rows)");
            di->router_rows_attr_set = true;
        }
        return launch_pdl(k_router_rows, dim3((d->E + 3) / 4, (M + 7) / 8), dim3(kRouteThreads), router_smem(d, M),
                          st, p, "k_router_rows launch");
    }
    // the logits are given: scores only
    return launch_pdl(k_router, dim3((M * d->E + 255) / 256), dim3(256), 0, st, p, "k_router launch");
}

// CTAs of a step's top-k launch that prefetch the shared expert's records into L2.
constexpr int kTopkPrefetchCtas = 64;

// FC1 input quantisation arguments, carried by the top-k launch (CTAs 1..).
struct QuantArgs {
    const void* x = nullptr;
    void *xq = nullptr, *xs = nullptr, *xq_sh = nullptr, *xs_sh = nullptr;
    // router step without a workspace: where the router records a timeout, and the top-k
    // CTAs' arrival counter that decides which of them clears it
    int32_t *router_status = nullptr, *arrivals = nullptr;
};

int quant_units_host(int fmt, int M, int H) {
    const int Mpad = round_up(M, 16);
    return (fmt == MOE_FMT_MXFP8 || fmt == MOE_FMT_MXFP4) ? Mpad * (H / 32)
                                                          : (fmt == MOE_FMT_NVFP4 ? Mpad * (H / 16) : Mpad * (H / 8));
}

TopkRouteParams topk_params(const moe_layer_desc* d, const WsLayout& L, uint8_t* ws, int M, const float* scores,
                            const float* bias, int32_t* topk_idx, float* topk_w, int do_topk, int do_route,
                            int32_t* counts, int32_t* perm, int32_t* inv_perm, int32_t* tiles, int32_t* num_tiles,
                            const QuantArgs& qa, int* qctas_out) {
    TopkRouteParams p{};
    p.scores = scores;
    p.bias = d->has_bias ? bias : nullptr;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.M = M;
    p.E = d->E;
    p.k = d->k;
    p.renormalize = d->renormalize;
    p.has_shared = d->has_shared;
    p.do_topk = do_topk;
    p.do_route = do_route;
    p.rsf = d->routed_scaling_factor;
    p.counts = counts;
    p.perm = perm;
    p.inv_perm = inv_perm;
    p.tiles = tiles;
    p.num_tiles = num_tiles;
    p.groups = reinterpret_cast<Group*>(ws + L.groups);
    p.hdr = reinterpret_cast<WsHeader*>(ws + L.header);
    // one row per warp: ceil(M / 16) CTAs of 16 warps take the top-k
    p.topk_ctas = do_topk ? (M + kRouteThreads / 32 - 1) / (kRouteThreads / 32) : 1;
    p.topk_arrivals = (p.topk_ctas > 1 && do_route) ? reinterpret_cast<int32_t*>(ws + L.tcnt) : nullptr;
    if (qa.router_status) {
        p.router_status = qa.router_status;
        p.topk_arrivals = qa.arrivals;
    }
    int qctas = 0;
    if (qa.x) {
        p.x = static_cast<const uint16_t*>(qa.x);
        p.H = d->H;
        p.fmt_r = d->w_fmt;
        p.fmt_s = shared_fmt_of(d);
        p.quant_shared = separate_shared_input(d) ? 1 : 0;
        p.xq = static_cast<uint8_t*>(qa.xq);
        p.xs = static_cast<uint8_t*>(qa.xs);
        p.xq_sh = static_cast<uint8_t*>(qa.xq_sh);
        p.xs_sh = static_cast<uint8_t*>(qa.xs_sh);
        p.gs_r = d->w_fmt == MOE_FMT_NVFP4 ? d->gs_a1 : 1.0f;
        p.gs_s = (d->has_shared && d->shared_fmt == MOE_FMT_NVFP4) ? d->gs_a1_shared : 1.0f;
        int units = quant_units_host(p.fmt_r, M, d->H);
        if (p.quant_shared && quant_units_host(p.fmt_s, M, d->H) > units) units = quant_units_host(p.fmt_s, M, d->H);
        qctas = (units + kRouteThreads - 1) / kRouteThreads;
    }
    *qctas_out = qctas;
    return p;
}

moe_status launch_topk_route(const moe_layer_desc* d, const WsLayout& L, uint8_t* ws, int M, const float* scores,
                             const float* bias, int32_t* topk_idx, float* topk_w, int do_topk, int do_route,
                             int32_t* counts, int32_t* perm, int32_t* inv_perm, int32_t* tiles, int32_t* num_tiles,
                             cudaStream_t st, const QuantArgs& qa = QuantArgs()) {
    int qctas = 0;
    const TopkRouteParams p = topk_params(d, L, ws, M, scores, bias, topk_idx, topk_w, do_topk, do_route, counts,
                                          perm, inv_perm, tiles, num_tiles, qa, &qctas);
    return launch_pdl(k_topk_route, dim3(p.topk_ctas + qctas), dim3(kRouteThreads), 0, st, p,
                      "k_topk_route launch");
}

// Router, top-k, routing and quantisation as one launch (k_front): the router CTAs of
// k_router_rows, then the quantisation CTAs of k_topk_route. Its arrival counters sit in
// the workspace's arrival region: [0] row blocks done, [4 .. 4 + ceil(M/8)) router CTAs
// done per row block (all self-resetting).
moe_status launch_front(const moe_layer_desc* d, const RouterParams& r, const TopkRouteParams& t, int qctas,
                        const WsLayout& L, uint8_t* ws, int M, cudaStream_t st) {
    DevInfo* di;
    moe_status s = dev_info(&di);
    if (s != MOE_OK) return s;
    if (!di->front_attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_front, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             di->smem_optin - 16384);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(k_front)");
        di->front_attr_set = true;
    }
    FrontParams f{};
    f.r = r;
    f.t = t;
    int32_t* arrivals = reinterpret_cast<int32_t*>(ws + L.tcnt);
    f.t.topk_arrivals = arrivals;
    f.rb_arrivals = arrivals + 4;
    const int nr = ((d->E + 3) / 4) * ((M + 7) / 8);
    return launch_pdl(k_front, dim3(nr + qctas), dim3(kRouteThreads), router_smem(d, M), st, f, "k_front launch");
}

struct GemmBuffers {
    const void *xq, *xs, *xq_sh, *xs_sh;  // gate_up inputs
    void *hq, *hs;                         // gate_up outputs / down inputs
    float* y;
    const int32_t* perm;
};

// Units at the end of a GEMM launch's list that CTAs take from a shared counter once they
// have finished their equal static range (the layer's gemm_schedule). STATIC (the default)
// takes none: on GB300 the counter-fed items stream measurably slower than the static
// ranges. HYBRID puts 2 units per CTA in the pool, DYNAMIC all of them. Every schedule
// agrees with the definition of the step within the tolerance of the fp32 accumulation,
// and each is deterministic.
int gemm_pool_units(int schedule, int grid) {
    if (schedule == MOE_SCHED_DYNAMIC) return -1;
    if (schedule == MOE_SCHED_HYBRID) return 2 * grid;
    return 0;
}

// Weight classes of one GEMM (0 gate_up, 1 down): routed experts and the shared expert.
void gemm_classes(int g, const moe_layer_desc* d, const moe_qweight* wr, const moe_qweight* ws_,
                  const GemmBuffers& b, int M, GemmClass* cls) {
    const size_t hqr = hq_routed(d, M), hsr = hs_routed(d, M);
    for (int c = 0; c < 2; ++c) {
        GemmClass& C = cls[c];
        const bool sh = c == 1;
        if (sh && !d->has_shared) {
            C.fmt = d->w_fmt;
            C.MB = 1;
            C.KS = 1;
            continue;
        }
        const moe_qweight* w = sh ? ws_ : wr;
        C.fmt = sh ? d->shared_fmt : d->w_fmt;
        C.w = static_cast<const uint8_t*>(w->packed);
        C.gs_w = C.fmt == MOE_FMT_NVFP4 ? w->global_scale : nullptr;
        const int I = sh ? d->I_shared : d->I;
        C.I = I;
        C.out_fmt = C.fmt;
        const float gs1 = sh ? d->gs_a1_shared : d->gs_a1, gs2 = sh ? d->gs_a2_shared : d->gs_a2;
        if (g == 0) {
            C.MB = 2 * I / kBlockRows;
            C.KS = steps_of(C.fmt, d->H);
            C.b = static_cast<const uint8_t*>(sh ? b.xq_sh : b.xq);
            C.bs = static_cast<const uint8_t*>(sh ? b.xs_sh : b.xs);
            C.gs_a = C.fmt == MOE_FMT_NVFP4 ? gs1 : 1.0f;
            C.gs_out = C.fmt == MOE_FMT_NVFP4 ? gs2 : 1.0f;
            C.hq = static_cast<uint8_t*>(b.hq) + (sh ? hqr : 0);
            C.hs = static_cast<uint8_t*>(b.hs) + (sh ? hsr : 0);
        } else {
            C.MB = d->H / kBlockRows;
            C.KS = steps_of(C.fmt, I);
            C.b = static_cast<const uint8_t*>(b.hq) + (sh ? hqr : 0);
            C.bs = static_cast<const uint8_t*>(b.hs) + (sh ? hsr : 0);
            C.gs_a = C.fmt == MOE_FMT_NVFP4 ? gs2 : 1.0f;
            C.gs_out = 1.0f;
        }
    }
}

// One expert-GEMM launch: mode 0 gate_up, 1 down, 2 both (gate_up items first; a down item
// waits in the kernel until its group's gate_up units are done).
constexpr uint64_t kGemmWaitNs = 2000000000ull;  // 2 s: limit of every wait in the GEMM kernel

moe_status launch_gemm(int mode, const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13,
                       const moe_qweight* w2, const moe_qweight* sh2, const GemmBuffers& b, int M, const WsLayout& L,
                       uint8_t* ws, cudaStream_t st, bool prefetch_shared = true, uint64_t wait_ns = kGemmWaitNs,
                       int dep_extra = 0) {
    DevInfo* di;
    moe_status s = dev_info(&di);
    if (s != MOE_OK) return s;
    GemmParams p{};
    p.mode = mode;
    p.M = M;
    p.k = d->k;
    p.E = d->E;
    p.H = d->H;
    p.Mpad = round_up(M, 16);
    p.has_shared = d->has_shared;
    p.perm = b.perm;
    p.groups = reinterpret_cast<const Group*>(ws + L.groups);
    p.hdr = reinterpret_cast<const WsHeader*>(ws + L.header);
    p.y = b.y;
    p.counters[0] = reinterpret_cast<int32_t*>(ws + L.cnt_gu);
    p.counters[1] = reinterpret_cast<int32_t*>(ws + L.cnt_dn);
    float* part = reinterpret_cast<float*>(ws + L.partials);
    p.partials[0] = part;
    // in one launch both GEMMs cut units at once: down uses the pool's slots (no pool then)
    p.partials[1] = mode == 2 ? part + (size_t)kPoolSlot0 * kPartialFloats : part;
    p.sched = reinterpret_cast<int32_t*>(ws + L.sched) + 2 * (mode == 1 ? 1 : 0);
    p.gu_done = reinterpret_cast<int32_t*>(ws + L.gu_done);
    p.swiglu_limit = d->swiglu_limit > 0.0f ? d->swiglu_limit : 0.0f;
    p.prefetch_shared = prefetch_shared ? 1 : 0;
    p.wait_ns = wait_ns;
    p.dep_extra = dep_extra;

    p.pool_units = mode == 2 ? 0 : gemm_pool_units(d->gemm_schedule, di->sms < kMaxGemmCtas ? di->sms : kMaxGemmCtas);
    p.status = reinterpret_cast<int32_t*>(ws + L.header);
    if (mode != 1) gemm_classes(0, d, w13, sh13, b, M, p.cls[0]);
    if (mode != 0) gemm_classes(1, d, w2, sh2, b, M, p.cls[1]);
    const int g0 = mode == 1 ? 1 : 0;
    int am = 0;
    for (int g = g0; g <= (mode == 0 ? 0 : 1); ++g)
        for (int c = 0; c < 2; ++c) am = atoms_per_step(p.cls[g][c].fmt) > am ? atoms_per_step(p.cls[g][c].fmt) : am;
    p.atoms_max = am;
    // NVFP4 stages carry 8 scale copies; issuing them from two extra warps keeps the MMA
    // issuers' streams short. MXFP8-only launches copy in the issuers (one hop less).
    p.sf_warps = am == 4 ? 1 : 0;
    p.a_off = 0;
    p.sfa_off = kBlockRows * kStepBytes;
    p.b_off = round_up(p.sfa_off + am * kAtomBytes, 1024);
    p.sfb_off = p.b_off + p.Mpad * kStepBytes;
    p.stage_bytes = round_up(p.sfb_off + am * kAtomBytes, 1024);
    // alignment, epilogue staging, work-item queue, deferred copies, barriers and flags (1 KB covers those
    // not counted per stage)
    const int fixed = 1024 + p.Mpad * kBlockRows * 4 + kGemmQueue * 64 + kDeferBytes + 1024;
    int S = (di->smem_optin - fixed) / (p.stage_bytes + 24);  // + full/empty/ready barriers
    const int tmem_cap = am ? (512 - 2 * acc_bank_cols(am, p.Mpad)) / (8 * am) : 16;
    if (S > tmem_cap) S = tmem_cap;
    if (S > kMaxStages) S = kMaxStages;
    S &= ~1;  // even ring: items start on even slots
    if (S < 2) return fail(MOE_ERR_UNSUPPORTED, "not enough shared memory for the GEMM pipeline");
    p.stages = S;
    const size_t smem = (size_t)fixed + (size_t)S * p.stage_bytes + 24 * S;
    if (!di->gemm_attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_expert_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             di->smem_optin);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(k_expert_gemm)");
        di->gemm_attr_set = true;
    }
    int grid = di->sms;
    if (grid > kMaxGemmCtas) grid = kMaxGemmCtas;
    return launch_pdl(k_expert_gemm, dim3(grid), dim3(kGemmThreads), smem, st, p,
                      mode == 0 ? "k_expert_gemm(gate_up) launch"
                                : (mode == 1 ? "k_expert_gemm(down) launch" : "k_expert_gemm(gate_up+down) launch"),
                      mode == 2);
}

FinalizeParams finalize_params(const moe_layer_desc* d, const float* y, const float* topk_w, const int32_t* inv_perm,
                               int M, void* residual, const void* gamma, void* out, void* outq, void* outs) {
    FinalizeParams p{};
    p.y = y;
    p.topk_w = topk_w;
    p.inv_perm = inv_perm;
    p.residual = static_cast<uint16_t*>(residual);
    p.gamma = static_cast<const uint16_t*>(gamma);
    p.out = static_cast<uint16_t*>(out);
    p.outq = static_cast<uint8_t*>(outq);
    p.outs = static_cast<uint8_t*>(outs);
    p.M = M;
    p.H = d->H;
    p.k = d->k;
    p.has_shared = d->has_shared;
    p.eps = d->rms_eps;
    return p;
}

moe_status launch_finalize(const moe_layer_desc* d, const float* y, const float* topk_w, const int32_t* inv_perm,
                           int M, void* residual, const void* gamma, void* out, void* outq, void* outs,
                           cudaStream_t st) {
    const FinalizeParams p = finalize_params(d, y, topk_w, inv_perm, M, residual, gamma, out, outq, outs);
    const int rows = outq ? round_up(M, 8) : M;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(8, rows);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 8;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_finalize, p);
    if (e != cudaSuccess) return cuda_fail(e, "k_finalize launch");
    return MOE_OK;
}

moe_status check_qweight(const moe_qweight* w, int fmt, const char* name) {
    if (!w) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
    if (!w->packed || !aligned16(w->packed)) return fail(MOE_ERR_INVALID_ARG, "%s.packed is NULL or unaligned", name);
    if (fmt == MOE_FMT_NVFP4 && !w->global_scale)
        return fail(MOE_ERR_INVALID_ARG, "%s.global_scale is required for NVFP4", name);
    return MOE_OK;
}

}  // namespace

// ================================================================== C ABI
namespace {

// Arguments of the FC1 call (moe_expert_gate_up, and the first half of moe_expert_ffn).
moe_status gate_up_buffers(const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13, const void* xq,
                           const void* xq_scales, const void* xq_sh, const void* xq_sh_scales, const int32_t* perm,
                           int M, void* hq, void* hq_scales, void* ws, GemmBuffers& b) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    if ((s = check_qweight(w13, d->w_fmt, "w13")) != MOE_OK) return s;
    if (d->has_shared && (s = check_qweight(sh13, d->shared_fmt, "sh13")) != MOE_OK) return s;
    REQUIRE_PTR(xq, "xq");
    REQUIRE_PTR(xq_scales, "xq_scales");
    if (separate_shared_input(d)) {
        REQUIRE_PTR(xq_sh, "xq_sh");
        if (d->shared_fmt != MOE_FMT_BF16) REQUIRE_PTR(xq_sh_scales, "xq_sh_scales");
    }
    REQUIRE_PTR(perm, "perm");
    REQUIRE_PTR(hq, "hq");
    REQUIRE_PTR(hq_scales, "hq_scales");
    REQUIRE_PTR(ws, "ws");
    b.xq = xq;
    b.xs = xq_scales;
    b.xq_sh = separate_shared_input(d) ? xq_sh : xq;
    b.xs_sh = separate_shared_input(d) ? xq_sh_scales : xq_scales;
    b.hq = hq;
    b.hs = hq_scales;
    b.perm = perm;
    return MOE_OK;
}

// Arguments of the FC2 call (moe_expert_down, and the second half of moe_expert_ffn).
moe_status down_buffers(const moe_layer_desc* d, const moe_qweight* w2, const moe_qweight* sh2, const void* hq,
                        const void* hq_scales, int M, float* y_pairs, void* ws, GemmBuffers& b) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    if ((s = check_qweight(w2, d->w_fmt, "w2")) != MOE_OK) return s;
    if (d->has_shared && (s = check_qweight(sh2, d->shared_fmt, "sh2")) != MOE_OK) return s;
    REQUIRE_PTR(hq, "hq");
    REQUIRE_PTR(hq_scales, "hq_scales");
    REQUIRE_PTR(y_pairs, "y_pairs");
    REQUIRE_PTR(ws, "ws");
    b.hq = const_cast<void*>(hq);
    b.hs = const_cast<void*>(hq_scales);
    b.y = y_pairs;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_last_error_string(void) { return g_err.c_str(); }

size_t moe_packed_bytes(const moe_layer_desc* d, int which) {
    if (check_desc(d) != MOE_OK) return 0;
    int fmt, rows, K, n;
    switch (which) {
        case MOE_W13: fmt = d->w_fmt; rows = 2 * d->I; K = d->H; n = d->E; break;
        case MOE_W2: fmt = d->w_fmt; rows = d->H; K = d->I; n = d->E; break;
        case MOE_SH13: if (!d->has_shared) return 0; fmt = d->shared_fmt; rows = 2 * d->I_shared; K = d->H; n = 1; break;
        case MOE_SH2: if (!d->has_shared) return 0; fmt = d->shared_fmt; rows = d->H; K = d->I_shared; n = 1; break;
        default: return 0;
    }
    return (size_t)n * (rows / kBlockRows) * steps_of(fmt, K) * record_bytes(fmt);
}

size_t moe_act_bytes(int fmt, int rows, int K) {
    if (fmt < 0 || fmt > 3 || rows < 1 || rows > kMaxRows || K <= 0 || row_bytes(fmt, K) % kStepBytes) return 0;
    return act_bytes(fmt, rows, K);
}
size_t moe_act_scale_bytes(int fmt, int rows, int K) {
    if (fmt < 0 || fmt > 3 || rows < 1 || rows > kMaxRows || K <= 0 || row_bytes(fmt, K) % kStepBytes) return 0;
    return act_scale_bytes(fmt, K);
}
size_t moe_hq_bytes(const moe_layer_desc* d, int max_rows) {
    if (check_desc(d) != MOE_OK || max_rows < 1 || max_rows > kMaxRows) return 0;
    return hq_total(d, max_rows);
}
size_t moe_hq_scale_bytes(const moe_layer_desc* d, int max_rows) {
    if (check_desc(d) != MOE_OK || max_rows < 1 || max_rows > kMaxRows) return 0;
    return hs_total(d, max_rows);
}
size_t moe_workspace_bytes(const moe_layer_desc* d) {
    if (check_desc(d) != MOE_OK) return 0;
    return layout(d).total;
}

moe_status moe_workspace_init(const moe_layer_desc* d, void* ws, moe_stream_t stream) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws, "ws");
    const WsLayout L = layout(d);
    cudaError_t e = cudaMemsetAsync(ws, 0, L.total, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(ws)");
    return ok();
}

moe_status moe_ws_view(const moe_layer_desc* d, void* ws, moe_ws_ptrs* out) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws, "ws");
    REQUIRE(out != nullptr, "out is NULL");
    const WsLayout L = layout(d);
    uint8_t* w = static_cast<uint8_t*>(ws);
    out->status = reinterpret_cast<int32_t*>(w + L.header);
    out->logits = reinterpret_cast<float*>(w + L.logits);
    out->scores = reinterpret_cast<float*>(w + L.scores);
    out->topk_idx = reinterpret_cast<int32_t*>(w + L.topk_idx);
    out->topk_w = reinterpret_cast<float*>(w + L.topk_w);
    out->expert_counts = reinterpret_cast<int32_t*>(w + L.counts);
    out->perm = reinterpret_cast<int32_t*>(w + L.perm);
    out->inv_perm = reinterpret_cast<int32_t*>(w + L.inv_perm);
    out->tiles = reinterpret_cast<int32_t*>(w + L.tiles);
    out->num_tiles = reinterpret_cast<int32_t*>(w + L.num_tiles);
    out->xq = w + L.xq;
    out->xq_scales = w + L.xs;
    out->xq_shared = w + L.xq_sh;
    out->xq_shared_scales = w + L.xs_sh;
    out->hq = w + L.hq;
    out->hq_scales = w + L.hs;
    out->y_pairs = reinterpret_cast<float*>(w + L.y);
    return ok();
}

moe_status moe_pack_weights(const moe_layer_desc* d, int which, const void* codes, const void* scales, void* dst,
                            moe_stream_t stream) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(which >= 0 && which <= 3, "which=%d: need 0..3", which);
    REQUIRE(d->has_shared || which < 2, "shared projection requested but has_shared == 0");
    PackParams p{};
    const bool sh = which >= 2;
    p.fmt = sh ? d->shared_fmt : d->w_fmt;
    p.n_exp = sh ? 1 : d->E;
    const int I = sh ? d->I_shared : d->I;
    p.gate_up = (which == MOE_W13 || which == MOE_SH13) ? 1 : 0;
    p.rows = p.gate_up ? 2 * I : d->H;
    p.K = p.gate_up ? d->H : I;
    p.I = I;
    REQUIRE_PTR(codes, "codes");
    REQUIRE_PTR(dst, "dst");
    if (p.fmt != MOE_FMT_BF16) REQUIRE_PTR(scales, "scales");
    p.codes = static_cast<const uint8_t*>(codes);
    p.scales = static_cast<const uint8_t*>(scales);
    p.dst = static_cast<uint8_t*>(dst);
    k_pack<<<1024, 256, 0, (cudaStream_t)stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "k_pack launch");
    return ok();
}

moe_status moe_router_topk(const moe_layer_desc* d, const void* x, const void* w_gate, const float* bias,
                           const float* logits_in, int M, float* logits_out, int32_t* topk_idx, float* topk_w,
                           void* xq, void* xq_scales, void* xq_sh, void* xq_sh_scales, void* ws,
                           moe_stream_t stream) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    REQUIRE_PTR(x, "x");
    if (!logits_in) REQUIRE_PTR(w_gate, "w_gate");
    OPT_PTR(logits_in, "logits_in");
    OPT_PTR(logits_out, "logits_out");
    if (d->has_bias) REQUIRE_PTR(bias, "bias");
    REQUIRE_PTR(topk_idx, "topk_idx");
    REQUIRE_PTR(topk_w, "topk_w");
    REQUIRE_PTR(xq, "xq");
    REQUIRE_PTR(xq_scales, "xq_scales");
    if (separate_shared_input(d)) {
        REQUIRE_PTR(xq_sh, "xq_sh");
        if (d->shared_fmt != MOE_FMT_BF16) REQUIRE_PTR(xq_sh_scales, "xq_sh_scales");
    }
    REQUIRE_PTR(ws, "ws");
    const WsLayout L = layout(d);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* scores = reinterpret_cast<float*>(w + L.scores);
    cudaStream_t st = (cudaStream_t)stream;
    s = launch_router(d, x, w_gate, logits_in, M, logits_out, scores, reinterpret_cast<int32_t*>(w + L.header), st);
    if (s != MOE_OK) return s;
    QuantArgs qa;
    qa.x = x;
    qa.xq = xq;
    qa.xs = xq_scales;
    qa.xq_sh = xq_sh;
    qa.xs_sh = xq_sh_scales;
    s = launch_topk_route(d, L, w, M, scores, bias, topk_idx, topk_w, 1, 0, nullptr, nullptr, nullptr, nullptr,
                          nullptr, st, qa);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_route_tiles(const moe_layer_desc* d, const int32_t* topk_idx, int M, int32_t* tiles,
                           int32_t* num_tiles, int32_t* perm, int32_t* inv_perm, int32_t* expert_counts, void* ws,
                           moe_stream_t stream) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    REQUIRE_PTR(topk_idx, "topk_idx");
    REQUIRE_PTR(tiles, "tiles");
    REQUIRE_PTR(num_tiles, "num_tiles");
    REQUIRE_PTR(perm, "perm");
    REQUIRE_PTR(inv_perm, "inv_perm");
    REQUIRE_PTR(expert_counts, "expert_counts");
    REQUIRE_PTR(ws, "ws");
    const WsLayout L = layout(d);
    s = launch_topk_route(d, L, static_cast<uint8_t*>(ws), M, nullptr, nullptr, const_cast<int32_t*>(topk_idx),
                          nullptr, 0, 1, expert_counts, perm, inv_perm, tiles, num_tiles, (cudaStream_t)stream);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_expert_gate_up(const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13,
                              const void* xq, const void* xq_scales, const void* xq_sh, const void* xq_sh_scales,
                              const int32_t* perm, int M, void* hq, void* hq_scales, void* ws,
                              moe_stream_t stream) {
    GemmBuffers b{};
    moe_status s = gate_up_buffers(d, w13, sh13, xq, xq_scales, xq_sh, xq_sh_scales, perm, M, hq, hq_scales, ws, b);
    if (s != MOE_OK) return s;
    s = launch_gemm(0, d, w13, sh13, nullptr, nullptr, b, M, layout(d), static_cast<uint8_t*>(ws),
                    (cudaStream_t)stream);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_expert_down(const moe_layer_desc* d, const moe_qweight* w2, const moe_qweight* sh2, const void* hq,
                           const void* hq_scales, int M, float* y_pairs, void* ws, moe_stream_t stream) {
    GemmBuffers b{};
    moe_status s = down_buffers(d, w2, sh2, hq, hq_scales, M, y_pairs, ws, b);
    if (s != MOE_OK) return s;
    s = launch_gemm(1, d, nullptr, nullptr, w2, sh2, b, M, layout(d), static_cast<uint8_t*>(ws),
                    (cudaStream_t)stream);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_expert_ffn(const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13,
                          const moe_qweight* w2, const moe_qweight* sh2, const void* xq, const void* xq_scales,
                          const void* xq_sh, const void* xq_sh_scales, const int32_t* perm, int M, void* hq,
                          void* hq_scales, float* y_pairs, void* ws, moe_stream_t stream) {
    GemmBuffers b{};
    moe_status s = gate_up_buffers(d, w13, sh13, xq, xq_scales, xq_sh, xq_sh_scales, perm, M, hq, hq_scales, ws, b);
    if (s != MOE_OK) return s;
    if ((s = down_buffers(d, w2, sh2, hq, hq_scales, M, y_pairs, ws, b)) != MOE_OK) return s;
    s = launch_gemm(2, d, w13, sh13, w2, sh2, b, M, layout(d), static_cast<uint8_t*>(ws), (cudaStream_t)stream);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_finalize_norm(const moe_layer_desc* d, const float* y_pairs, const float* topk_w,
                             const int32_t* inv_perm, int M, void* residual, const void* gamma, void* out,
                             void* outq, void* outq_scales, void* ws, moe_stream_t stream) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    REQUIRE_PTR(y_pairs, "y_pairs");
    REQUIRE_PTR(topk_w, "topk_w");
    REQUIRE_PTR(inv_perm, "inv_perm");
    REQUIRE_PTR(residual, "residual");
    REQUIRE_PTR(gamma, "gamma");
    REQUIRE_PTR(out, "out");
    REQUIRE((outq == nullptr) == (outq_scales == nullptr), "outq and outq_scales must both be given or both NULL");
    OPT_PTR(outq, "outq");
    OPT_PTR(outq_scales, "outq_scales");
    (void)ws;
    s = launch_finalize(d, y_pairs, topk_w, inv_perm, M, residual, gamma, out, outq, outq_scales,
                        (cudaStream_t)stream);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_step(const moe_layer_desc* d, const moe_step_args* a, int M, void* ws, moe_stream_t stream) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(a != nullptr, "args is NULL");
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    REQUIRE_PTR(a->x, "x");
    REQUIRE_PTR(a->w_gate, "w_gate");
    if (d->has_bias) REQUIRE_PTR(a->bias, "bias");
    if ((s = check_qweight(&a->w13, d->w_fmt, "w13")) != MOE_OK) return s;
    if ((s = check_qweight(&a->w2, d->w_fmt, "w2")) != MOE_OK) return s;
    if (d->has_shared) {
        if ((s = check_qweight(&a->sh13, d->shared_fmt, "sh13")) != MOE_OK) return s;
        if ((s = check_qweight(&a->sh2, d->shared_fmt, "sh2")) != MOE_OK) return s;
    }
    REQUIRE_PTR(a->residual, "residual");
    REQUIRE_PTR(a->gamma, "gamma");
    REQUIRE_PTR(a->out, "out");
    if (d->emit_next_mxfp8) {
        REQUIRE_PTR(a->outq, "outq");
        REQUIRE_PTR(a->outq_scales, "outq_scales");
    }
    REQUIRE_PTR(ws, "ws");
    const WsLayout L = layout(d);
    uint8_t* w = static_cast<uint8_t*>(ws);
    cudaStream_t st = (cudaStream_t)stream;
    float* logits = reinterpret_cast<float*>(w + L.logits);
    float* scores = reinterpret_cast<float*>(w + L.scores);
    int32_t* topk_idx = reinterpret_cast<int32_t*>(w + L.topk_idx);
    float* topk_w = reinterpret_cast<float*>(w + L.topk_w);
    int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);
    int32_t* inv_perm = reinterpret_cast<int32_t*>(w + L.inv_perm);
    // the shared expert's records do not depend on the routing: the router launch prefetches
    // them into L2 while the front end runs (the GEMM launch then does not)
    const size_t sh13_bytes = d->has_shared ? (size_t)(2 * d->I_shared / kBlockRows) *
                                                  steps_of(d->shared_fmt, d->H) * record_bytes(d->shared_fmt)
                                            : 0;
    const size_t sh2_bytes = d->has_shared ? (size_t)(d->H / kBlockRows) * steps_of(d->shared_fmt, d->I_shared) *
                                                 record_bytes(d->shared_fmt)
                                           : 0;
    const void* sh13_w = d->has_shared ? a->sh13.packed : nullptr;
    const void* sh2_w = d->has_shared ? a->sh2.packed : nullptr;
    QuantArgs qa;
    qa.x = a->x;
    qa.xq = w + L.xq;
    qa.xs = w + L.xs;
    qa.xq_sh = w + L.xq_sh;
    qa.xs_sh = w + L.xs_sh;
    // one front launch: its router CTAs prefetch the shared expert; two launches: the top-k
    // launch's extra CTAs do (the router CTAs then leave as soon as their logits are out)
    const bool one_front = d->front_launches == 1;
    const RouterParams rp = router_params(d, a->x, a->w_gate, nullptr, M, logits, scores,
                                          reinterpret_cast<int32_t*>(w + L.header), sh13_w, sh13_bytes, sh2_w,
                                          sh2_bytes);
    int qctas = 0;
    const TopkRouteParams tp = topk_params(d, L, w, M, scores, a->bias, topk_idx, topk_w, 1, 1,
                                           reinterpret_cast<int32_t*>(w + L.counts), perm, inv_perm,
                                           reinterpret_cast<int32_t*>(w + L.tiles),
                                           reinterpret_cast<int32_t*>(w + L.num_tiles), qa, &qctas);
    if (one_front) {
        s = launch_front(d, rp, tp, qctas, L, w, M, st);
        if (s != MOE_OK) return s;
    } else {
        s = launch_router(d, a->x, a->w_gate, nullptr, M, logits, scores, reinterpret_cast<int32_t*>(w + L.header), st);
        if (s != MOE_OK) return s;
        TopkRouteParams tpp = tp;
        if (d->has_shared) {
            tpp.l2_pf[0] = static_cast<const uint8_t*>(sh13_w);
            tpp.l2_pf_bytes[0] = sh13_bytes;
            tpp.l2_pf[1] = static_cast<const uint8_t*>(sh2_w);
            tpp.l2_pf_bytes[1] = sh2_bytes;
            tpp.pf_ctas = kTopkPrefetchCtas;
        }
        s = launch_pdl(k_topk_route, dim3(tpp.topk_ctas + qctas + tpp.pf_ctas), dim3(kRouteThreads), 0, st, tpp,
                       "k_topk_route launch");
        if (s != MOE_OK) return s;
    }
    GemmBuffers b{};
    b.xq = w + L.xq;
    b.xs = w + L.xs;
    b.xq_sh = w + L.xq_sh;
    b.xs_sh = w + L.xs_sh;
    b.hq = w + L.hq;
    b.hs = w + L.hs;
    b.y = reinterpret_cast<float*>(w + L.y);
    b.perm = perm;
    void* outq = d->emit_next_mxfp8 ? a->outq : nullptr;
    void* outs = d->emit_next_mxfp8 ? a->outq_scales : nullptr;
    if (d->ffn_launches != 2) {
        s = launch_gemm(2, d, &a->w13, &a->sh13, &a->w2, &a->sh2, b, M, L, w, st, false);
        if (s != MOE_OK) return s;
    } else {
        s = launch_gemm(0, d, &a->w13, &a->sh13, nullptr, nullptr, b, M, L, w, st, false);
        if (s != MOE_OK) return s;
        s = launch_gemm(1, d, nullptr, nullptr, &a->w2, &a->sh2, b, M, L, w, st);
        if (s != MOE_OK) return s;
    }
    s = launch_finalize(d, b.y, topk_w, inv_perm, M, a->residual, a->gamma, a->out, outq, outs, st);
    if (s != MOE_OK) return s;
    return ok();
}

// ------------------------------------------------------------------------------------
// Router step without a caller workspace (moe_router_topk_noalloc).
//
// Some callers cannot give the library device memory: a host framework that owns every
// allocation and hands plugins no allocator, or a serving loop that must not allocate once
// it is running (an allocation can synchronise the device or fail under memory pressure).
// For them the router step keeps its scratch (the scores) in one fixed array in the
// library's own device memory, allocated when the library is loaded and held by every GPU
// that loads it until the process exits.
//
// Layout: [256 B header: router status word, top-k arrival counter][scores 64 x 512 fp32].
constexpr size_t kNaHeader = 0, kNaArrivals = 16, kNaScores = 256;
constexpr size_t kNoAllocScratchBytes = kNaScores + 4ull * kMaxRows * kMaxE;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array per device, looked up once per device (with that device
// current) on its first call; the host-side name of the array is not a device address.
static uint8_t* noalloc_scratch(moe_status* st) {
    static std::mutex mu;
    static uint8_t* addr[128] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= 128) {
        *st = fail(MOE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            *st = cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
            return nullptr;
        }
        addr[dev] = static_cast<uint8_t*>(ptr);
    }
    *st = MOE_OK;
    return addr[dev];
}

// wait_ns and unreachable_tx: the router's copy waits (kRouterWaitNs and 0 but in the test of
// the timeout path below).
static moe_status router_topk_noalloc(const moe_layer_desc* d, const void* x, const void* w_gate, const float* bias,
                                      const float* logits_in, int M, float* logits_out, int32_t* topk_idx,
                                      float* topk_w, void* xq, void* xq_scales, void* xq_sh, void* xq_sh_scales,
                                      moe_stream_t stream, uint64_t wait_ns, uint32_t unreachable_tx) {
    moe_status s = check_desc(d);
    if (s != MOE_OK) return s;
    REQUIRE(M >= 1 && M <= kMaxRows, "M=%d: need 1..%d", M, kMaxRows);
    REQUIRE_PTR(x, "x");
    if (!logits_in) REQUIRE_PTR(w_gate, "w_gate");
    OPT_PTR(logits_in, "logits_in");
    OPT_PTR(logits_out, "logits_out");
    if (d->has_bias) REQUIRE_PTR(bias, "bias");
    REQUIRE_PTR(topk_idx, "topk_idx");
    REQUIRE_PTR(topk_w, "topk_w");
    REQUIRE_PTR(xq, "xq");
    REQUIRE_PTR(xq_scales, "xq_scales");
    if (separate_shared_input(d)) {
        REQUIRE_PTR(xq_sh, "xq_sh");
        if (d->shared_fmt != MOE_FMT_BF16) REQUIRE_PTR(xq_sh_scales, "xq_sh_scales");
    }
    uint8_t* scratch = noalloc_scratch(&s);
    if (!scratch) return s;
    // scratch regions as a workspace layout for the shared launch helpers (the top-k-only
    // launch reads no group table and no arrival counter)
    WsLayout L{};
    L.header = kNaHeader;
    L.groups = kNaHeader;
    cudaStream_t st = (cudaStream_t)stream;
    float* scores = reinterpret_cast<float*>(scratch + kNaScores);
    s = launch_router(d, x, w_gate, logits_in, M, logits_out, scores, reinterpret_cast<int32_t*>(scratch + kNaHeader),
                      st, nullptr, 0, nullptr, 0, wait_ns, unreachable_tx);
    if (s != MOE_OK) return s;
    QuantArgs qa;
    qa.x = x;
    qa.xq = xq;
    qa.xs = xq_scales;
    qa.xq_sh = xq_sh;
    qa.xs_sh = xq_sh_scales;
    qa.router_status = reinterpret_cast<int32_t*>(scratch + kNaHeader);
    qa.arrivals = reinterpret_cast<int32_t*>(scratch + kNaArrivals);
    s = launch_topk_route(d, L, scratch, M, scores, bias, topk_idx, topk_w, 1, 0, nullptr, nullptr, nullptr, nullptr,
                          nullptr, st, qa);
    if (s != MOE_OK) return s;
    return ok();
}

extern "C" moe_status moe_router_topk_noalloc(const moe_layer_desc* d, const void* x, const void* w_gate,
                                              const float* bias, const float* logits_in, int M, float* logits_out,
                                              int32_t* topk_idx, float* topk_w, void* xq, void* xq_scales,
                                              void* xq_sh, void* xq_sh_scales, moe_stream_t stream) {
    return router_topk_noalloc(d, x, w_gate, bias, logits_in, M, logits_out, topk_idx, topk_w, xq, xq_scales, xq_sh,
                               xq_sh_scales, stream, kRouterWaitNs, 0);
}

// Test of the allocation-free router's timeout path, not part of the public ABI (the header
// does not declare it): moe_router_topk_noalloc with the router GEMV's gate-row barrier
// expecting 16 bytes that no copy brings and its copy waits limited to wait_ns, so every
// router CTA gives up after wait_ns, records the timeout in the scratch header, waits for its
// real copies and returns without writing scores; the top-k launch then gives every row -1
// ids and zero weights and clears the record. Needs w_gate (no logits_in).
moe_status moe_internal_router_noalloc_unreachable_wait(const moe_layer_desc* d, const void* x, const void* w_gate,
                                                        const float* bias, int M, float* logits_out,
                                                        int32_t* topk_idx, float* topk_w, void* xq, void* xq_scales,
                                                        void* xq_sh, void* xq_sh_scales, uint64_t wait_ns,
                                                        moe_stream_t stream) {
    REQUIRE(wait_ns >= 1000000ull && wait_ns <= kRouterWaitNs, "wait_ns=%llu: need 1 ms .. 2 s",
            (unsigned long long)wait_ns);
    REQUIRE_PTR(w_gate, "w_gate");
    return router_topk_noalloc(d, x, w_gate, bias, nullptr, M, logits_out, topk_idx, topk_w, xq, xq_scales, xq_sh,
                               xq_sh_scales, stream, wait_ns, 16);
}

// Test of the GEMM's timeout path, not part of the public ABI (the header does not declare
// it): moe_expert_ffn with every down item's counter target one above what the FC1 units
// can reach and all waits limited to wait_ns, so the producers give up after wait_ns, record
// MOE_ERR_TIMEOUT in the workspace status word, and every CTA drains its copies and MMAs,
// frees its tensor memory and returns. The workspace then needs moe_workspace_init.
moe_status moe_internal_ffn_unreachable_wait(const moe_layer_desc* d, const moe_qweight* w13, const moe_qweight* sh13,
                                             const moe_qweight* w2, const moe_qweight* sh2, const void* xq,
                                             const void* xq_scales, const void* xq_sh, const void* xq_sh_scales,
                                             const int32_t* perm, int M, void* hq, void* hq_scales, float* y_pairs,
                                             void* ws, uint64_t wait_ns, moe_stream_t stream) {
    GemmBuffers b{};
    moe_status s = gate_up_buffers(d, w13, sh13, xq, xq_scales, xq_sh, xq_sh_scales, perm, M, hq, hq_scales, ws, b);
    if (s != MOE_OK) return s;
    if ((s = down_buffers(d, w2, sh2, hq, hq_scales, M, y_pairs, ws, b)) != MOE_OK) return s;
    REQUIRE(wait_ns >= 1000000ull && wait_ns <= kGemmWaitNs, "wait_ns=%llu: need 1 ms .. 2 s",
            (unsigned long long)wait_ns);
    s = launch_gemm(2, d, w13, sh13, w2, sh2, b, M, layout(d), static_cast<uint8_t*>(ws), (cudaStream_t)stream, true,
                    wait_ns, 1);
    if (s != MOE_OK) return s;
    return ok();
}

moe_status moe_get_status(void* ws, moe_stream_t stream, int* dev_status) {
    REQUIRE_PTR(ws, "ws");
    REQUIRE(dev_status != nullptr, "dev_status is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    *dev_status = v;
    return ok();
}

}  // extern "C"
