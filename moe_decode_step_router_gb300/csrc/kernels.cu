// Router, route, finalize and packing kernels of the MoE step (sm_103a).
//
// Sources: "SGLang-NVIDIA-Mega" README, slot table of "What a covered DeepSeek-V4.1-Flash
// step runs" (rows gate: one router per row, sigmoid top-k; moe: route kernel and 8-row
// tiles; shared_ll: one-pass MXFP8 quant of the expert input into its row-tile layout;
// hop_b: top-k finalize, shared-expert add, RMSNorm, next input's MXFP8 scales per 8-row
// tile) and Qwen3.5 slot table (row route: router GEMM and NVFP4 quantisation of the MoE
// input in one launch); "sgl-nvidia-mega pull request 24", "Modifications / Target spec"
// (one expert group, sigmoid scores, renormalised top-k).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "finalize.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------------------------
// FC1 input quantisation into the tiled layout. Unit = one scale block (MXFP8, MXFP4: 32
// elements, NVFP4: 16) or one 16-byte chunk (BF16) of one padded row; rows >= M are zero.
__device__ void quant_unit(const uint16_t* __restrict__ x, int M, int H, int Mpad, int fmt, float gs, uint8_t* xq,
                           uint8_t* xs, int u) {
    if (fmt == MOE_FMT_MXFP8) {
        const int nb = H / 32, m = u / nb, bi = u % nb;
        float v[32];
        if (m < M) {
            const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)m * H + 32 * bi);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 w = __ldg(src + i);
                v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
                v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
                v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
                v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const int e = mx_exponent(amax);
        const float sc = exp2_int(-e);
        uint32_t wd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo = e4m3x2(__fmul_rn(v[4 * i + 1], sc), __fmul_rn(v[4 * i + 0], sc));
            uint32_t hi = e4m3x2(__fmul_rn(v[4 * i + 3], sc), __fmul_rn(v[4 * i + 2], sc));
            wd[i] = lo | (hi << 16);
        }
        const int s = bi / 4, c0 = 2 * (bi % 4);
        uint8_t* row = xq + (size_t)s * Mpad * kStepBytes + (size_t)m * kStepBytes;
        *reinterpret_cast<uint4*>(row + ((c0 ^ (m & 7)) * 16)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (m & 7)) * 16)) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
        xs[(size_t)s * kAtomBytes + (m % 32) * 16 + (m / 32) * 4 + (bi % 4)] = (uint8_t)(e + 127);
    } else if (fmt == MOE_FMT_MXFP4) {
        const int nb = H / 32, m = u / nb, bi = u % nb;
        float v[32];
        if (m < M) {
            const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)m * H + 32 * bi);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 w = __ldg(src + i);
                v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
                v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
                v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
                v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const int e = mx4_exponent(amax);
        const float sc = exp2_int(-e);
        uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i)
            wd[i / 4] |= (uint32_t)e2m1x2(__fmul_rn(v[2 * i + 1], sc), __fmul_rn(v[2 * i], sc)) << (8 * (i % 4));
        // a 256-element step holds 8 blocks of 16 bytes each
        const int s = bi / 8, c = bi % 8;
        uint8_t* row = xq + (size_t)s * Mpad * kStepBytes + (size_t)m * kStepBytes;
        *reinterpret_cast<uint4*>(row + ((c ^ (m & 7)) * 16)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        xs[(size_t)s * 2 * kAtomBytes + (c / 4) * kAtomBytes + (m % 32) * 16 + (m / 32) * 4 + (c % 4)] =
            (uint8_t)(e + 127);
    } else if (fmt == MOE_FMT_NVFP4) {
        const int nb = H / 16, m = u / nb, bi = u % nb;
        float v[16];
        if (m < M) {
            const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)m * H + 16 * bi);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint4 w = __ldg(src + i);
                v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
                v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
                v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
                v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const uint8_t s8 = nv_scale(amax, gs);
        const float dsc = e4m3_to_f32(s8);
        const float denom = __fmul_rn(dsc, gs);
        uint32_t wd[2] = {0u, 0u};
        if (dsc != 0.0f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t b = e2m1x2(__fdiv_rn(v[2 * i + 1], denom), __fdiv_rn(v[2 * i], denom));
                wd[i / 4] |= b << (8 * (i % 4));
            }
        }
        const int s = bi / 16, b16 = bi % 16, c = b16 / 2;
        uint8_t* row = xq + (size_t)s * Mpad * kStepBytes + (size_t)m * kStepBytes;
        *reinterpret_cast<uint2*>(row + ((c ^ (m & 7)) * 16) + (b16 % 2) * 8) = make_uint2(wd[0], wd[1]);
        xs[(size_t)s * 4 * kAtomBytes + (b16 / 4) * kAtomBytes + (m % 32) * 16 + (m / 32) * 4 + (b16 % 4)] = s8;
    } else {  // BF16: 16-byte chunks copied into the swizzled image
        const int nc = H / 8, m = u / nc, ci = u % nc;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (m < M) w = __ldg(reinterpret_cast<const uint4*>(x + (size_t)m * H + 8 * ci));
        const int s = ci / 8, c = ci % 8;
        uint8_t* row = xq + (size_t)s * Mpad * kStepBytes + (size_t)m * kStepBytes;
        *reinterpret_cast<uint4*>(row + ((c ^ (m & 7)) * 16)) = w;
    }
}

__device__ __forceinline__ int quant_units(int fmt, int Mpad, int H) {
    return (fmt == MOE_FMT_MXFP8 || fmt == MOE_FMT_MXFP4) ? Mpad * (H / 32)
                                                          : (fmt == MOE_FMT_NVFP4 ? Mpad * (H / 16) : Mpad * (H / 8));
}

// ------------------------------------------------------------------------------------
// One 128-byte line into L2 (no data returned, no copy engine involved).
__device__ __forceinline__ void prefetch_line_l2(const void* src) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(src) : "memory");
}

// a2 with the logits given (moe_router_topk with logits_in): the fp32 sigmoid score,
// evaluated in double and rounded once, as after the GEMV below.
constexpr int kRouterThreads = 256;

__global__ void __launch_bounds__(kRouterThreads) k_router(RouterParams p) {
    pdl_wait();
    const int n = p.M * p.E;
    for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < n; q += gridDim.x * blockDim.x) {
        const float lg = p.logits_in[q];
        p.scores[q] = (float)(1.0 / (1.0 + exp(-(double)lg)));
        if (p.logits_out) p.logits_out[q] = lg;
    }
    pdl_trigger();
}

// ------------------------------------------------------------------------------------
// a1 with no partial sums leaving the CTA: CTA (i, j) takes experts EPC i .. EPC i + EPC - 1
// and rows R j .. R j + R - 1 over the whole of H. Their gate rows are copied into shared
// memory (one bulk copy per row) before the dependency wait (they do not depend on earlier
// launches), the x rows (one bulk copy per row) after it; rows are kRouterRowPad elements
// apart beyond H, so that the fragment loads below hit 32 different banks.
// The dot products run on the tensor cores as bf16 x bf16 -> fp32 products of 16-wide K
// chunks (mma.sync m16n8k16): A holds the EPC gate rows (rows EPC..15 zero), B the R x rows
// (one per column), so D's rows 0..EPC-1 are this CTA's logits. Warp w takes the K chunks
// w, w + NW, ..., alternating between two accumulators; thread l then adds, for output
// l = expert * R + row, the two accumulators of every warp in warp order. The order of every
// addition is fixed: the logits are deterministic, and the same in both launches that run
// this (k_router_rows and k_front, both at NW = 16). The score is the same fp32 sigmoid as in
// k_router (evaluated in double, rounded once).
// (ei, rj): this CTA's expert group and row block; CTA cta of nct takes its share of the L2
// prefetch (k_front only; in the two-launch front the top-k launch prefetches). Returns false
// when a copy wait ran out (recorded in the status word; nothing is written).
constexpr int kRouterRowPad = 8;  // bf16 elements between the end of a row and the next row

// D += A B for one m16n8k16 tile: bf16 inputs, fp32 accumulators (register layouts of the
// PTX ISA's mma fragments).
__device__ __forceinline__ void mma_bf16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int EPC, int R, int NW>
__device__ __forceinline__ bool router_rows(const RouterParams& p, int ei, int rj, int cta, int nct) {
    static_assert(EPC * R == 32, "one output per lane");
    static_assert(EPC <= 8 && R == 8, "A rows 0..EPC-1 and B columns 0..7 of one m16n8k16 tile");
    extern __shared__ __align__(16) uint16_t rrs[];
    __shared__ float red[NW][32];
    __shared__ __align__(8) uint64_t rbar[2];  // gate rows, x rows
    __shared__ int s_never;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int H = p.H, E = p.E;
    const int e0 = ei * EPC, m0 = rj * R;
    const int M = min(R, p.M - m0);          // rows of this CTA
    const int LD = H + kRouterRowPad;        // shared-memory row stride (elements)
    uint16_t* wsm = rrs;                     // [EPC][LD]
    uint16_t* xsm = rrs + (size_t)EPC * LD;  // [M][LD]: rows m0 ..
    const uint32_t bar_w = smem_u32(&rbar[0]), bar_x = smem_u32(&rbar[1]);
    if (threadIdx.x == 0) {
        s_never = 0;
        mbar_init(bar_w, 1);
        mbar_init(bar_x, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_w, (uint32_t)(EPC * H * 2) + p.unreachable_tx);
        for (int r = 0; r < EPC; ++r)
            bulk_g2s(smem_u32(wsm + (size_t)r * LD), p.wg + (size_t)min(e0 + r, E - 1) * H, (uint32_t)(H * 2), bar_w);
    }
    __syncthreads();  // the barriers are initialised before anyone waits on them
    if (threadIdx.x == 32) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (!p.l2_pf[r]) continue;
            const size_t share = (p.l2_pf_bytes[r] / (size_t)nct + 15) & ~(size_t)15;
            const size_t b0 = (size_t)cta * share, b1 = b0 + share < p.l2_pf_bytes[r] ? b0 + share : p.l2_pf_bytes[r];
            for (size_t o = b0; o < b1; o += 65536)
                prefetch_l2(p.l2_pf[r] + o, (uint32_t)(b1 - o < 65536 ? b1 - o : 65536));
        }
    }
    pdl_wait();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar_x, (uint32_t)(M * H * 2));
        for (int m = 0; m < M; ++m)
            bulk_g2s(smem_u32(xsm + (size_t)m * LD), p.x + (size_t)(m0 + m) * H, (uint32_t)(H * 2), bar_x);
    }
    bool ok = mbar_wait_bounded(bar_w, 0, &s_never, p.wait_ns);
    ok = mbar_wait_bounded(bar_x, 0, &s_never, p.wait_ns) && ok;
    if (!__syncthreads_and(ok)) {
        // a copy did not land in time: record it, give the copies one more bounded wait so
        // that none still writes shared memory when the CTA leaves, and produce nothing
        // (bytes a test asked for that no copy brings are counted first, so that this wait
        // ends exactly when the real copies have landed)
        if (threadIdx.x == 0) {
            if (p.status) atomicCAS(p.status, 0, (int)MOE_ERR_TIMEOUT);
            if (p.unreachable_tx) mbar_complete_tx(bar_w, p.unreachable_tx);
        }
        mbar_wait_bounded(bar_w, 0, &s_never, p.wait_ns / 2);
        mbar_wait_bounded(bar_x, 0, &s_never, p.wait_ns / 2);
        return false;
    }
    // fragments: lane (g = lane / 4, t = lane % 4) holds A rows g (and g + 8: zero) at columns
    // 2t, 2t + 1 and 2t + 8, 2t + 9 of the chunk, B column g at the same K, and D rows g,
    // g + 8 at columns 2t, 2t + 1
    const int g = lane >> 2, t = lane & 3;
    const bool a_live = g < EPC, b_live = g < M;
    const uint32_t* wrow = reinterpret_cast<const uint32_t*>(wsm + (size_t)(a_live ? g : 0) * LD) + t;
    const uint32_t* xrow = reinterpret_cast<const uint32_t*>(xsm + (size_t)(b_live ? g : 0) * LD) + t;
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};  // chunks w + 2 i NW / w + (2 i + 1) NW
    auto chunk = [&](int kc, float* d) {
        const int o = kc * 8;  // 32-bit words before the chunk
        const uint32_t a0 = a_live ? wrow[o] : 0u, a2 = a_live ? wrow[o + 4] : 0u;
        const uint32_t b0 = b_live ? xrow[o] : 0u, b1 = b_live ? xrow[o + 4] : 0u;
        mma_bf16_16816(d, a0, 0u, a2, 0u, b0, b1);
    };
    const int KC = H / 16;
    int kc = warp;
    for (; kc + NW < KC; kc += 2 * NW) {
        chunk(kc, d0);
        chunk(kc + NW, d1);
    }
    if (kc < KC) chunk(kc, d0);
    pdl_trigger();  // let the top-k launch get scheduled while the sums are added
    if (a_live) {
        red[warp][g * R + 2 * t] = d0[0] + d1[0];
        red[warp][g * R + 2 * t + 1] = d0[1] + d1[1];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int e = e0 + threadIdx.x / R, m = threadIdx.x % R;
        float lg = red[0][threadIdx.x];
#pragma unroll
        for (int w = 1; w < NW; ++w) lg += red[w][threadIdx.x];
        if (m < M && e < E) {
            p.scores[(size_t)(m0 + m) * E + e] = (float)(1.0 / (1.0 + exp(-(double)lg)));
            if (p.logits_out) p.logits_out[(size_t)(m0 + m) * E + e] = lg;
        }
    }
    return true;
}

__global__ void __launch_bounds__(kRouteThreads) k_router_rows(RouterParams p) {
    router_rows<4, 8, kRouteThreads / 32>(p, blockIdx.x, blockIdx.y, blockIdx.y * gridDim.x + blockIdx.x,
                                          gridDim.x * gridDim.y);
}

// ------------------------------------------------------------------------------------
// a2 + a4: top-k of the selection key (score + bias) with ties to the lower expert index
// and renormalised weights (fp32, within a few ulps of the exact value), one row per warp
// over the first ceil(M / 16) CTAs; the last of them to finish then runs the stable counting
// sort of the (row, slot) pairs into 8-row tiles and the per-expert group table.

// Order-preserving map of an fp32 key to u32: a larger key gives a larger integer; every
// finite key maps above 0, which marks taken or absent experts.
__device__ __forceinline__ uint32_t key_u32(float f) {
    const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));  // -0 -> +0: equal keys tie
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void block_scan4(int4 v, int4* out_excl, int4* total, int4* sh_warp) {
    // inclusive warp scan
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int4 s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int a = __shfl_up_sync(0xffffffffu, s.x, o), b = __shfl_up_sync(0xffffffffu, s.y, o);
        int c = __shfl_up_sync(0xffffffffu, s.z, o), d = __shfl_up_sync(0xffffffffu, s.w, o);
        if (lane >= o) { s.x += a; s.y += b; s.z += c; s.w += d; }
    }
    if (lane == 31) sh_warp[warp] = s;
    __syncthreads();
    if (warp == 0) {
        int4 t = (lane < (int)(blockDim.x / 32)) ? sh_warp[lane] : make_int4(0, 0, 0, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int a = __shfl_up_sync(0xffffffffu, t.x, o), b = __shfl_up_sync(0xffffffffu, t.y, o);
            int c = __shfl_up_sync(0xffffffffu, t.z, o), d = __shfl_up_sync(0xffffffffu, t.w, o);
            if (lane >= o) { t.x += a; t.y += b; t.z += c; t.w += d; }
        }
        sh_warp[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    int4 base = (warp > 0) ? sh_warp[warp - 1] : make_int4(0, 0, 0, 0);
    *out_excl = make_int4(base.x + s.x - v.x, base.y + s.y - v.y, base.z + s.z - v.z, base.w + s.w - v.w);
    *total = sh_warp[blockDim.x / 32 - 1];
    __syncthreads();
}

// a2: the top-k of row m by one warp (the warp's lanes hold experts lane + 32 i); writes
// topk_idx / topk_w of the row and, when s_topk is given, the ids into it too.
// The lane's bias values (a layer constant, so a launch may load them before its dependency
// wait): experts lane + 32 i, clamped.
__device__ __forceinline__ void topk_bias(const TopkRouteParams& p, int lane, float bi[kMaxE / 32]) {
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) bi[i] = __ldg(p.bias + min(lane + 32 * i, p.E - 1));
}

// bias_pre: the lane's bias values when the caller has loaded them (topk_bias), else null.
__device__ __forceinline__ void topk_row(const TopkRouteParams& p, int m, int lane, int* s_topk,
                                         const float* bias_pre = nullptr) {
    const int E = p.E, k = p.k;
    // keys as order-preserving u32 (0 = taken / absent); lane owns e = lane + 32 i
    uint32_t ku[kMaxE / 32];
    float sc[kMaxE / 32], bi[kMaxE / 32];
    // unconditional (clamped) loads of the row's scores and of the bias, all in flight
    // before the first use
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) sc[i] = __ldcg(p.scores + (size_t)m * E + min(lane + 32 * i, E - 1));
    if (p.bias) {
        if (bias_pre) {
#pragma unroll
            for (int i = 0; i < kMaxE / 32; ++i) bi[i] = bias_pre[i];
        } else {
            topk_bias(p, lane, bi);
        }
    }
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const bool valid = lane + 32 * i < E;
        ku[i] = valid ? key_u32(p.bias ? __fadd_rn(sc[i], bi[i]) : sc[i]) : 0u;
        if (!valid) sc[i] = 0.0f;
    }
    // Lane-local order: larger key first, lower index among equal keys. Each lane keeps its
    // first element in that order (best) and the one after it (second); a lane whose best is
    // taken promotes its second, and scans its keys again only when it has no second left
    // (from its second win on), for the elements after the one just taken. So most rounds
    // cost one max reduction, one ballot and two shuffles, not a scan.
    uint32_t lb = 0u, l2 = 0u;
    int li = 0, i2 = 0;
    float ls = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        if (ku[i] > lb) {
            l2 = lb; i2 = li; s2 = ls;
            lb = ku[i]; li = i; ls = sc[i];
        } else if (ku[i] > l2) {
            l2 = ku[i]; i2 = i; s2 = sc[i];
        }
    }
    bool has2 = true;
    int my_idx = 0;
    float my_sc = 0.0f;
    float ssum = 0.0f;  // fp32 in slot order: FP64 is ~50x slower than fp32 on this part
    // Each round: one max reduction and one ballot find the winning lane (a tie between
    // lanes, which needs the lower expert id, takes one more reduction); the winner moves on
    // to its next element while the others read its id and score.
    for (int j = 0; j < k; ++j) {
        const uint32_t wmax = __reduce_max_sync(0xffffffffu, lb);
        const uint32_t bal = __ballot_sync(0xffffffffu, lb == wmax);
        int wl;
        if ((bal & (bal - 1u)) == 0u) {
            wl = __ffs(bal) - 1;
        } else {
            const uint32_t cand = (lb == wmax) ? (uint32_t)(lane + 32 * li) : 0xffffffffu;
            wl = (int)(__reduce_min_sync(0xffffffffu, cand) & 31u);
        }
        const int wsl = __shfl_sync(0xffffffffu, li, wl);
        const float wsc = __shfl_sync(0xffffffffu, ls, wl);
        if (lane == wl) {
            if (has2) {
                lb = l2; li = i2; ls = s2;
                has2 = false;
            } else {
                // the elements after the taken one (key lt, index lti) in the lane's order
                const uint32_t lt = lb;
                const int lti = li;
                lb = 0u; l2 = 0u; li = 0; i2 = 0; ls = 0.0f; s2 = 0.0f;
#pragma unroll
                for (int i = 0; i < kMaxE / 32; ++i) {
                    const uint32_t kv = (ku[i] < lt || (ku[i] == lt && i > lti)) ? ku[i] : 0u;
                    if (kv > lb) {
                        l2 = lb; i2 = li; s2 = ls;
                        lb = kv; li = i; ls = sc[i];
                    } else if (kv > l2) {
                        l2 = kv; i2 = i; s2 = sc[i];
                    }
                }
                has2 = true;
            }
        }
        ssum = __fadd_rn(ssum, wsc);
        if (lane == j) { my_idx = wl + 32 * wsl; my_sc = wsc; }
    }
    if (lane < k) {
        p.topk_idx[(size_t)m * k + lane] = my_idx;
        if (s_topk) s_topk[m * k + lane] = my_idx;
        p.topk_w[(size_t)m * k + lane] =
            p.renormalize ? __fmul_rn(__fdiv_rn(my_sc, ssum), p.rsf) : __fmul_rn(my_sc, p.rsf);
    }
}

// Shared memory of the routing CTA.
struct RouteSmem {
    unsigned long long sel[kMaxE + 1];  // per expert: bit m set when row m selected it
    int s_off[kMaxE + 2];               // per expert: first position in perm
    int4 sh_warp[32];
    int s_bad;
};

// a4 by one CTA of kRouteThreads threads: the stable counting sort of the M*k selections
// into 8-row tiles, perm / inv_perm and the group table. own_topk: the selections, when
// this CTA made them all (shared memory); else they are read through L2.
__device__ void route_all(const TopkRouteParams& p, const int* own_topk, RouteSmem& rs) {
    const int M = p.M, E = p.E, k = p.k;
    unsigned long long* sel = rs.sel;
    int* s_off = rs.s_off;
    const int P = M * k;
    if (threadIdx.x == 0) rs.s_bad = 0;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) sel[e] = 0ull;
    __syncthreads();
    for (int q = threadIdx.x; q < P; q += blockDim.x) {
        const int e = own_topk ? own_topk[q] : __ldcg(p.topk_idx + q);
        if (e < 0 || e >= E) {
            rs.s_bad = 1;
        } else {
            atomicOr(&sel[e], 1ull << (q / k));
        }
    }
    __syncthreads();
    if (rs.s_bad) {
        if (threadIdx.x == 0) {
            atomicCAS(&p.hdr->status, 0, (int)MOE_ERR_INVALID_ARG);
            p.hdr->num_groups = 0;
            p.hdr->num_tiles = 0;
            *p.num_tiles = 0;
        }
        return;
    }
    // two experts per thread (E + 1 <= 513 <= 2 * blockDim): pairs, tiles, group flag,
    // padded rows; one block-wide exclusive scan over the per-thread sums
    auto vals = [&](int e) {
        int c = 0;
        if (e < E) c = __popcll(sel[e]);
        else if (e == E) c = p.has_shared ? M : 0;
        if (e > E) return make_int4(0, 0, 0, 0);
        return make_int4(c, (c + kTileRows - 1) / kTileRows, (e < E && c > 0) ? 1 : 0, (e < E) ? round_up(c, 16) : 0);
    };
    const int e0 = 2 * threadIdx.x;
    const int4 v0 = vals(e0), v1 = vals(e0 + 1);
    int4 ex, tot;
    block_scan4(make_int4(v0.x + v1.x, v0.y + v1.y, v0.z + v1.z, v0.w + v1.w), &ex, &tot, rs.sh_warp);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = e0 + h;
        const int4 v = h ? v1 : v0;
        const int4 x0 = h ? make_int4(ex.x + v0.x, ex.y + v0.y, ex.z + v0.z, ex.w + v0.w) : ex;
        if (e <= E) {
            const int c = v.x;
            p.counts[e] = c;
            for (int t = 0; t < v.y; ++t) {
                int32_t* tp = p.tiles + 3 * (x0.y + t);
                tp[0] = e;
                tp[1] = x0.x + kTileRows * t;
                tp[2] = min(kTileRows, c - kTileRows * t);
            }
            if (v.z) p.groups[x0.z] = Group{e, c, x0.x, x0.w};
            s_off[e] = x0.x;
        }
    }
    if (threadIdx.x == 0) {
        *p.num_tiles = tot.y;
        p.hdr->num_tiles = tot.y;
        p.hdr->num_groups = tot.z;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < P; q += blockDim.x) {
        const int ee = own_topk ? own_topk[q] : __ldcg(p.topk_idx + q), m = q / k;
        const unsigned long long below = (m == 0) ? 0ull : (sel[ee] & ((1ull << m) - 1ull));
        const int pos = s_off[ee] + __popcll(below);
        p.perm[pos] = q;
        p.inv_perm[q] = pos;
    }
    if (p.has_shared)
        for (int m = threadIdx.x; m < M; m += blockDim.x) {
            p.perm[P + m] = P + m;
            p.inv_perm[P + m] = P + m;
        }
}

// a3: the FC1 input quantisation, spread over CTAs [0, ncta) of a group (cta: this one).
__device__ void quant_all(const TopkRouteParams& p, int cta, int ncta) {
    const int Mpad = round_up(p.M, 16);
    const int nthreads = ncta * blockDim.x, tid = cta * blockDim.x + threadIdx.x;
    const int nr = quant_units(p.fmt_r, Mpad, p.H);
    for (int u = tid; u < nr; u += nthreads) quant_unit(p.x, p.M, p.H, Mpad, p.fmt_r, p.gs_r, p.xq, p.xs, u);
    if (p.quant_shared) {
        const int ns = quant_units(p.fmt_s, Mpad, p.H);
        for (int u = tid; u < ns; u += nthreads) quant_unit(p.x, p.M, p.H, Mpad, p.fmt_s, p.gs_s, p.xq_sh, p.xs_sh, u);
    }
}

__global__ void __launch_bounds__(kRouteThreads) k_topk_route(TopkRouteParams p) {
    __shared__ RouteSmem rs;
    __shared__ int s_topk[kMaxRows * kMaxK];  // this CTA's selections, when it also routes
    __shared__ int s_last;
    const int npf = p.pf_ctas;
    if ((int)blockIdx.x >= (int)gridDim.x - npf) {
        // L2 prefetch of records a later launch streams: they depend on no earlier launch, so
        // these CTAs do not wait for the router, and they are done (line prefetches leave the
        // SM at once) long before the routing CTA, whose end the next launch waits for; HBM
        // is otherwise idle while the front end runs
        const int cta = blockIdx.x - (gridDim.x - npf);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (!p.l2_pf[r]) continue;
            const size_t share = (p.l2_pf_bytes[r] / (size_t)npf + 127) & ~(size_t)127;
            const size_t b0 = (size_t)cta * share, b1 = b0 + share < p.l2_pf_bytes[r] ? b0 + share : p.l2_pf_bytes[r];
            for (size_t o = b0 + 128 * (size_t)threadIdx.x; o < b1; o += 128 * (size_t)blockDim.x)
                prefetch_line_l2(p.l2_pf[r] + o);
        }
        return;
    }
    // the top-k CTAs' bias values are a layer constant: loaded while the dependency wait runs
    float bias_r[kMaxE / 32];
    const bool pre_bias = p.bias && p.do_topk && (int)blockIdx.x < p.topk_ctas;
    if (pre_bias) topk_bias(p, threadIdx.x % 32, bias_r);
    pdl_wait();
    pdl_trigger();  // the GEMM's CTAs may take the other SMs and wait there
    const int tk = p.topk_ctas;
    if ((int)blockIdx.x >= tk) {  // the CTAs after the top-k ones quantise x
        quant_all(p, blockIdx.x - tk, gridDim.x - tk - npf);
        return;
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int M = p.M, k = p.k;
    // without a workspace a router timeout has no status word to go to: its scores were
    // never written, so every row gets -1 ids and zero weights instead of stale results
    const bool router_failed = p.router_status && __ldcg(p.router_status) != 0;
    if (p.do_topk && router_failed) {
        for (int q = (int)blockIdx.x * blockDim.x + threadIdx.x; q < M * k; q += tk * blockDim.x) {
            p.topk_idx[q] = -1;
            p.topk_w[q] = 0.0f;
        }
    }
    if (p.router_status) {
        // the last top-k CTA to read the record clears it for the next call
        __syncthreads();
        if (threadIdx.x == 0) {
            bool last = true;
            if (tk > 1) {
                __threadfence();
                last = atomicAdd(p.topk_arrivals, 1) == tk - 1;
                if (last) *p.topk_arrivals = 0;
            }
            if (last && router_failed) *p.router_status = 0;
        }
        if (router_failed) return;
    }
    if (p.do_topk) {
        for (int m = (int)blockIdx.x * (kRouteThreads / 32) + warp; m < M; m += tk * (kRouteThreads / 32))
            topk_row(p, m, lane, s_topk, pre_bias ? bias_r : nullptr);
        __syncthreads();
    }
    if (!p.do_route) return;
    if (tk > 1) {
        // the last top-k CTA to finish routes every row (the others' rows through L2)
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int old = atomicAdd(p.topk_arrivals, 1);
            s_last = (old == tk - 1) ? 1 : 0;
            if (s_last) *p.topk_arrivals = 0;  // every CTA has arrived: ready for the next launch
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
    }
    route_all(p, (p.do_topk && tk == 1) ? s_topk : nullptr, rs);
}

// ------------------------------------------------------------------------------------
// a1 + a2 + a3 + a4 in one launch (Qwen3.5 slot table of the "SGLang-NVIDIA-Mega" README,
// row route: the router GEMM and the quantisation of the MoE input in one launch; here the
// top-k and the routing join them). CTAs [0, nE * nRB) are the router's (CTA i: expert
// group i % nE, row block i / nE, as k_router_rows); the last of a row block's router CTAs
// to finish takes that block's rows' top-k (one warp per row), and the last row block to
// finish routes every row; the CTAs after the router ones quantise x. No CTA waits for
// another (arrival counters only), so the launch needs no co-residency, and its logits,
// selections and routing are the bytes of the router launch followed by the top-k launch.
__global__ void __launch_bounds__(kRouteThreads, 1) k_front(FrontParams f) {
    __shared__ RouteSmem rs;
    __shared__ int s_topk[kMaxRows * kMaxK];
    __shared__ int s_last;
    const RouterParams& r = f.r;
    const TopkRouteParams& t = f.t;
    const int nE = (r.E + 3) / 4, nRB = (r.M + 7) / 8, nr = nE * nRB;
    if ((int)blockIdx.x >= nr) {
        pdl_wait();
        pdl_trigger();
        quant_all(t, blockIdx.x - nr, gridDim.x - nr);
        return;
    }
    const int rj = blockIdx.x / nE;
    if (!router_rows<4, 8, kRouteThreads / 32>(r, blockIdx.x % nE, rj, blockIdx.x, nr)) return;
    // the last router CTA of the row block takes its rows' top-k (the other CTAs' scores
    // through L2)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int old = atomicAdd(f.rb_arrivals + rj, 1);
        s_last = (old == nE - 1) ? 1 : 0;
        if (s_last) f.rb_arrivals[rj] = 0;  // every CTA of the block has arrived
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, m = 8 * rj + warp;
    if (warp < 8 && m < r.M) topk_row(t, m, lane, s_topk);
    __threadfence();  // this block's selections, before its arrival below
    __syncthreads();
    if (nRB > 1) {
        // the last row block to finish routes every row
        if (threadIdx.x == 0) {
            const int old = atomicAdd(t.topk_arrivals, 1);
            s_last = (old == nRB - 1) ? 1 : 0;
            if (s_last) *t.topk_arrivals = 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
    }
    route_all(t, nRB == 1 ? s_topk : nullptr, rs);
}

// ------------------------------------------------------------------------------------
// a7 as its own launch: one cluster of kFinSlices CTAs per row (finalize.cuh), the slices'
// sums of squares exchanged over distributed shared memory and added in rank order
// (deterministic).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of a cluster barrier, for an arrival long before the wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// v into the copy of *local in the shared memory of the cluster's CTA `rank`.
__device__ __forceinline__ void dsmem_st(float* local, uint32_t rank, float v) {
    uint32_t a = smem_u32(local), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

__global__ void __launch_bounds__(kFinThreads) k_finalize(FinalizeParams p) {
    __shared__ FinSmem fs;
    const int m = blockIdx.y, s = (int)cluster_rank();
    if (m >= p.M) {  // padding rows of the 8-row output tiles (written by no earlier launch)
        pdl_wait();
        pdl_trigger();
        fin_pad_row(p, m, s);
        cluster_sync();
        return;
    }
    // every CTA of the cluster has started once this barrier completes (waited on before
    // the first store into another CTA's shared memory)
    cluster_arrive_relaxed();
    // everything but the FC2 rows, before the wait for the FC2 launch
    const FinPre pre = fin_preload(p, m, s, fs);
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    float hv[4];
    fin_combine(p, m, s, pre, hv, fs);
    cluster_wait();
    // this slice's sum of squares into slot s of every CTA of the cluster (thread 0 wrote
    // fs.part); after the barrier each CTA holds all of them and no CTA touches another's
    // shared memory again
    if (threadIdx.x == 0)
        for (int rk = 0; rk < kFinSlices; ++rk) dsmem_st(&fs.parts[s], (uint32_t)rk, fs.part);
    cluster_sync();
    float tot = 0.0f;
#pragma unroll
    for (int rk = 0; rk < kFinSlices; ++rk) tot += fs.parts[rk];
    fin_output(p, m, s, pre, hv, tot);
}

// ------------------------------------------------------------------------------------
// Load-time repack of one projection into streaming records (see the ABI header).
__global__ void k_pack(PackParams p) {
    const int KS = steps_of(p.fmt, p.K), A = atoms_per_step(p.fmt), MB = p.rows / kBlockRows;
    const size_t REC = record_bytes(p.fmt);
    const int64_t rb = row_bytes(p.fmt, p.K), rs = row_scales(p.fmt, p.K);
    const size_t nrec = (size_t)p.n_exp * MB * KS;
    // work item: (record, row, 16-byte chunk) for codes and (record, row, atom) for scales
    const size_t per_rec = (size_t)kBlockRows * 8 + (size_t)kBlockRows * A;
    const size_t total = nrec * per_rec;
    for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < total; w += (size_t)gridDim.x * blockDim.x) {
        const size_t rec = w / per_rec;
        const int item = (int)(w % per_rec);
        const int s = (int)(rec % KS);
        const int b = (int)((rec / KS) % MB);
        const int e = (int)(rec / ((size_t)KS * MB));
        int r, c = 0, a = 0;
        const bool is_code = item < kBlockRows * 8;
        if (is_code) {
            r = item / 8;
            c = item % 8;
        } else {
            r = (item - kBlockRows * 8) / A;
            a = (item - kBlockRows * 8) % A;
        }
        int src_row;
        if (p.gate_up) src_row = (r < 64) ? (64 * b + r) : (p.I + 64 * b + (r - 64));
        else src_row = kBlockRows * b + r;
        uint8_t* dst = p.dst + rec * REC;
        if (is_code) {
            const uint4 v = *reinterpret_cast<const uint4*>(p.codes + ((size_t)e * p.rows + src_row) * rb +
                                                            (size_t)s * kStepBytes + 16 * c);
            *reinterpret_cast<uint4*>(dst + r * kStepBytes + ((c ^ (r & 7)) * 16)) = v;
        } else {
            const uint8_t* sp = p.scales + ((size_t)e * p.rows + src_row) * rs + (size_t)s * 4 * A + 4 * a;
            uint8_t* dp = dst + kBlockRows * kStepBytes + a * kAtomBytes + (r % 32) * 16 + (r / 32) * 4;
            dp[0] = sp[0];
            dp[1] = sp[1];
            dp[2] = sp[2];
            dp[3] = sp[3];
        }
    }
}

}  // namespace moe
