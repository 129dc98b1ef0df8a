// a7, the arithmetic of one (row, H slice) task: weighted combine in fixed slot order +
// shared row + residual (bf16) + RMSNorm, optional MXFP8 of the output per 32 along H
// ("SGLang-NVIDIA-Mega" README, slot table, row hop_b: top-k finalize, shared-expert add,
// RMSNorm, the next input's MXFP8 scales per 8-row tile).
//
// A row is cut into kFinSlices contiguous slices; a slice is handled by kFinThreads threads
// of one CTA, 4 consecutive elements (one float4 of each y row) each; k_finalize runs one
// 8-CTA cluster per row: every CTA pushes its slice's sum of squares into all the cluster's
// CTAs over distributed shared memory, and each adds them in slice order.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "quant.cuh"

namespace moe {

constexpr int kFinThreads = 256;
constexpr int kFinSlices = 8;

struct FinSmem {
    float red[kFinThreads / 32];
    float part;               // this slice's sum of squares (thread 0 writes it)
    float parts[kFinSlices];  // every slice's sum of squares, pushed here by the cluster's CTAs
    float w_s[kMaxK];
    int pos_s[kMaxK + 1];
};

__device__ __forceinline__ float fin_bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float fin_bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Rows M .. round_up(M, 8) - 1 of the next layer's MXFP8 input are zero (slice s).
__device__ __forceinline__ void fin_pad_row(const FinalizeParams& p, int m, int s) {
    const int H = p.H, slice = H / kFinSlices, n = s * slice + 4 * (int)threadIdx.x;
    if (threadIdx.x < kFinThreads && 4 * (int)threadIdx.x < slice) {
        *reinterpret_cast<uint32_t*>(p.outq + (size_t)m * H + n) = 0u;
        if ((n % 32) == 0) p.outs[(size_t)m * (H / 32) + n / 32] = 0;
    }
}

// What a (row m < M, slice s) task reads besides the FC2 rows: the row's pair positions
// and weights (into fs; the caller synchronises before fin_combine) and this thread's
// residual and gamma elements. None of it is written by the FC2 launch, so a launch that
// follows it may read this before its dependency wait (all of it comes from launches that
// had finished before the FC2 launch passed its own wait, or from before the step).
struct FinPre {
    uint2 rr, gg;  // residual, gamma: 4 bf16 each
};
__device__ __forceinline__ FinPre fin_preload(const FinalizeParams& p, int m, int s, FinSmem& fs) {
    const int H = p.H, k = p.k, P = p.M * k;
    const int slice = H / kFinSlices, n = s * slice + 4 * (int)threadIdx.x;
    const bool act = threadIdx.x < kFinThreads && 4 * (int)threadIdx.x < slice;
    // slots beyond k read slot k-1's row (an L2 hit) with weight 0, so every FC2-row load is
    // unconditional and all of them are in flight before the first FMA
    if (threadIdx.x < kMaxK) {
        const int j = min((int)threadIdx.x, k - 1);
        fs.pos_s[threadIdx.x] = __ldcg(p.inv_perm + m * k + j);
        fs.w_s[threadIdx.x] = (int)threadIdx.x < k ? __ldcg(p.topk_w + m * k + j) : 0.0f;
    }
    if (threadIdx.x == kMaxK) fs.pos_s[kMaxK] = p.has_shared ? __ldcg(p.inv_perm + P + m) : -1;
    FinPre pre{make_uint2(0u, 0u), make_uint2(0u, 0u)};
    if (act) {
        pre.rr = __ldcg(reinterpret_cast<const uint2*>(p.residual + (size_t)m * H + n));
        pre.gg = __ldg(reinterpret_cast<const uint2*>(p.gamma + n));
    }
    return pre;
}

// Combine + residual of slice s of row m (m < M), after fin_preload and a barrier: writes
// the new residual, leaves the bf16 values in hv and this slice's sum of their squares in
// fs.part (thread 0 writes it; the caller synchronises before reading it). Every thread of
// the CTA calls this (it holds __syncthreads); threads at or above kFinThreads take no
// elements.
__device__ __forceinline__ void fin_combine(const FinalizeParams& p, int m, int s, const FinPre& pre, float hv[4],
                                            FinSmem& fs) {
    const int H = p.H, k = p.k;
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int slice = H / kFinSlices, n = s * slice + 4 * (int)threadIdx.x;
    const bool act = threadIdx.x < kFinThreads && 4 * (int)threadIdx.x < slice;
    hv[0] = hv[1] = hv[2] = hv[3] = 0.0f;
    float ss = 0.0f;
    if (act) {
        float4 yv[kMaxK + 1];
        const int psh = fs.pos_s[kMaxK];
        const int kl = (k + 3) & ~3;  // slots loaded: k rounded up to 4 (the rest weigh 0)
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
            if ((j & 3) == 0 && j >= kl) break;
            else yv[j] = __ldcg(reinterpret_cast<const float4*>(p.y + (size_t)fs.pos_s[j] * H + n));
        yv[kMaxK] = __ldcg(reinterpret_cast<const float4*>(p.y + (size_t)max(psh, fs.pos_s[0]) * H + n));
        const uint2 rr = pre.rr;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {  // fixed slot order; FMAs only, no load below this point
                const float w = fs.w_s[j];
                acc[0] = fmaf(w, yv[j].x, acc[0]);
                acc[1] = fmaf(w, yv[j].y, acc[1]);
                acc[2] = fmaf(w, yv[j].z, acc[2]);
                acc[3] = fmaf(w, yv[j].w, acc[3]);
            }
        }
        if (psh >= 0) {
            acc[0] = __fadd_rn(acc[0], yv[kMaxK].x);
            acc[1] = __fadd_rn(acc[1], yv[kMaxK].y);
            acc[2] = __fadd_rn(acc[2], yv[kMaxK].z);
            acc[3] = __fadd_rn(acc[3], yv[kMaxK].w);
        }
        const float r[4] = {fin_bf16_lo(rr.x), fin_bf16_hi(rr.x), fin_bf16_lo(rr.y), fin_bf16_hi(rr.y)};
        uint32_t hb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat16 b = __float2bfloat16_rn(__fadd_rn(r[i], acc[i]));
            hb[i] = __bfloat16_as_ushort(b);
            hv[i] = __bfloat162float(b);
            ss = fmaf(hv[i], hv[i], ss);
        }
        *reinterpret_cast<uint2*>(p.residual + (size_t)m * H + n) = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0 && warp < kFinThreads / 32) fs.red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
#pragma unroll
        for (int i = 0; i < kFinThreads / 32; ++i) t += fs.red[i];
        fs.part = t;
    }
}

// RMSNorm of slice s of row m from the row's sum of squares tot (the slices' sums added in
// slice order, starting from 0): out, and the next layer's MXFP8 input when asked for.
__device__ __forceinline__ void fin_output(const FinalizeParams& p, int m, int s, const FinPre& pre, const float hv[4],
                                           float tot) {
    const int H = p.H, slice = H / kFinSlices, n = s * slice + 4 * (int)threadIdx.x;
    const bool act = threadIdx.x < kFinThreads && 4 * (int)threadIdx.x < slice;
    // the lanes of this warp that hold elements: whole 8-lane groups (a slice is a multiple
    // of 32 elements), so the MXFP8 block maximum below shuffles among active lanes only
    const uint32_t amask = __ballot_sync(0xffffffffu, act);
    const float rstd = rsqrtf(tot / (float)H + p.eps);
    if (!act) return;
    const uint2 gg = pre.gg;
    const float g[4] = {fin_bf16_lo(gg.x), fin_bf16_hi(gg.x), fin_bf16_lo(gg.y), fin_bf16_hi(gg.y)};
    uint32_t ob[4];
    float of[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 b = __float2bfloat16_rn(hv[i] * rstd * g[i]);
        ob[i] = __bfloat16_as_ushort(b);
        of[i] = __bfloat162float(b);
    }
    *reinterpret_cast<uint2*>(p.out + (size_t)m * H + n) = make_uint2(ob[0] | (ob[1] << 16), ob[2] | (ob[3] << 16));
    if (p.outq) {
        // a 32-element MX block = 8 consecutive lanes x 4 elements
        float amax = fmaxf(fmaxf(fabsf(of[0]), fabsf(of[1])), fmaxf(fabsf(of[2]), fabsf(of[3])));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(amask, amax, o, 8));
        const int e = mx_exponent(amax);
        const float sc = exp2_int(-e);
        const uint32_t lo = e4m3x2(__fmul_rn(of[1], sc), __fmul_rn(of[0], sc));
        const uint32_t hi = e4m3x2(__fmul_rn(of[3], sc), __fmul_rn(of[2], sc));
        *reinterpret_cast<uint32_t*>(p.outq + (size_t)m * H + n) = lo | (hi << 16);
        if ((n % 32) == 0) p.outs[(size_t)m * (H / 32) + n / 32] = (uint8_t)(e + 127);
    }
}

}  // namespace moe
