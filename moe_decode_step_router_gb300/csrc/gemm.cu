// Expert GEMMs of the MoE step on the 5th-generation tensor cores (sm_103a).
//
// "SGLang-NVIDIA-Mega" README, slot table of "What a covered DeepSeek-V4.1-Flash step
// runs", row moe: a route kernel and a pair of block-scaled tcgen05 GEMMs with 8-row
// tiles; row shared_ll: SwiGLU between the shared expert's GEMMs; Qwen3.5 slot table,
// row mkm: FC1, SwiGLU, NVFP4 requantisation and FC2. "sgl-nvidia-mega pull request 24",
// Target spec: the engines stream weights from records derived at load, and every map
// of the same rows gives the same bytes.
//
// Design (swap-AB): the expert weight is the MMA's A operand (M = 128 weight rows), the
// step's rows are N (padded to a multiple of 16). A unit is one (expert group, 128-row
// weight block); its K loop runs over 128-byte steps. The launch is persistent (one CTA
// per SM). The units, in order, are handed out as work items in two parts:
//  - static: the steps of all but the last units are cut into equal contiguous ranges, one
//    per CTA (stream-K), so every SM streams the same number of bytes;
//  - pool (none by default): a CTA that has finished its range takes items of the last
//    units from an atomic counter (whole units first, the final ones cut into up to four
//    pieces), so SMs that get more memory bandwidth than others take more of the pool.
// A unit cut into pieces is summed by the CTA that finishes the last piece, in piece order.
// Item boundaries depend only on the routing and every item starts on an even ring slot,
// so the arithmetic of each output is fixed whichever CTA computes it.
//
// A launch runs gate_up (mode 0), down (mode 1) or both (mode 2, moe_expert_ffn). In mode 2
// every CTA takes its static range of gate_up's units, then its range of down's, cut as the
// two launches cut them (so the bytes are the same). The gate_up epilogue that completes a
// unit counts it in its group's counter; a down item's weight copies go out at once and its
// activation copies wait, in ring order, until its group's counter is complete. The grid
// waits on itself, so mode 2 is a cooperative launch; every wait is bounded.
//
// Roles: warp 0 lane 0 takes the work items, publishes them to the other roles through a
// shared-memory queue and issues the bulk copies (weight record + activation tile + its
// scales) into a ring of shared-memory stages. Two MMA issuers (lane 0 of warps 1 and 6)
// consume the even and the odd ring slots, each accumulating into its own TMEM bank: at
// 8-64 rows one thread's tcgen05 issue rate, not the tensor pipe, caps the bytes a CTA
// can consume, and two issuers double that cap. In launches with NVFP4 weights (4 scale
// atoms per operand and step) warps 7..10 copy the stages' A and B block scales into
// tensor memory, two atoms each; otherwise each issuer copies the scales of its slots.
// Either way a slot's scale columns always have the same writer. Warps 2..5 add the two
// banks and run the epilogue (gate_up: SwiGLU + requantisation into the tiled FC2 input;
// down: fp32 rows in perm order).
#include <climits>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {

constexpr uint32_t kTmemCols = 512;
constexpr int kMaxAcc = 8;  // up to 8 accumulator buffers per bank

// One work item as published to the CTA's roles: the steps [ka, kb) of one unit with the
// facts of its group, and where its partial sum goes when the unit is cut into pieces.
struct WorkItem {
    int cls;  // 2 * GEMM (0 gate_up, 1 down) + class (0 routed, 1 shared); -1 end of the CTA's work
    int b, ka, kb;
    int rot;  // the steps are taken in the order ka + (rot + j) % (kb - ka), j = 0, 1, ...
    int expert, rows, perm_off, row_off, gidx;
    int unit;                     // unit id (piece counter index)
    int np;                       // pieces of the unit (1: the item is the whole unit)
    int s0, sb, sstride, myslot;  // partial slots: piece 0 in s0, piece pc > 0 in sb + pc * sstride
};
static_assert(sizeof(WorkItem) == 64, "queue entries are 64 bytes");

__device__ __forceinline__ int4 ld_group(const Group* gp) {
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(gp));
    return v;
}

// Position in the ring of shared-memory stages: slot and the parity of its lap. The ring
// length is even and every item starts on an even slot (an item of odd length is followed
// by one empty "bubble" slot), so step j of an item always sits in a slot of parity j % 2.
struct Ring {
    int st;
    uint32_t ph;
    int S;  // even, >= 2
    __device__ __forceinline__ void adv1() {
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }
    }
};

// Static part: this CTA's contiguous range of the steps of units [0, U0) (routed units in
// group order, then the shared expert's units). The position is advanced incrementally (no
// divisions after the start) and each group record is loaded one group ahead.
struct Walker {
    const Group* groups;
    long long T_r, T, t, t1;
    int gemm, ngroups, MB0, KS0, MB1, KS1, M, ktop;
    int cls, g, b, k;  // position of step t
    int4 cur, nxt;     // records of groups g and g + 1
    // Steps of units [0, U0) of GEMM gm.
    __device__ static long long steps_before(const GemmParams& p, int gm, int ngroups, int U0) {
        const int NRU = ngroups * p.cls[gm][0].MB;
        return U0 <= NRU ? (long long)U0 * p.cls[gm][0].KS
                         : (long long)NRU * p.cls[gm][0].KS + (long long)(U0 - NRU) * p.cls[gm][1].KS;
    }
    __device__ void init(const GemmParams& p, int gm, int ngroups_, int G, int c, int U0) {
        groups = p.groups;
        gemm = gm;
        ngroups = ngroups_;
        MB0 = p.cls[gm][0].MB;
        KS0 = p.cls[gm][0].KS;
        MB1 = p.cls[gm][1].MB;
        KS1 = p.cls[gm][1].KS;
        M = p.M;
        ktop = p.k;
        T_r = (long long)ngroups * MB0 * KS0;
        T = steps_before(p, gm, ngroups, U0);
        t = t1 = 0;
        if (c >= G || T == 0) return;
        seek((long long)c * T / G, (long long)(c + 1) * T / G);
    }
    // The walk [ta, tb): position of step ta, with the records of its group and the next.
    __device__ void seek(long long ta, long long tb) {
        t = ta;
        t1 = tb;
        if (t < T_r) {
            const long long u = t / KS0;
            cls = 0;
            g = (int)(u / MB0);
            b = (int)(u - (long long)g * MB0);
            k = (int)(t - u * KS0);
            cur = ld_group(groups + g);
            nxt = ld_group(groups + (g + 1 < ngroups ? g + 1 : g));
        } else {
            const long long tt = t - T_r;
            cls = 1;
            g = ngroups;
            b = (int)(tt / KS1);
            k = (int)(tt - (long long)b * KS1);
        }
    }
    __device__ long long start(long long c, int G) const { return c * T / G; }
    __device__ int cta_of(long long step, int G) const { return (int)(((step + 1) * G - 1) / T); }
    // The next segment of the range (with its stream-K piece facts), or false at its end.
    __device__ __forceinline__ bool next(WorkItem& w, int G, int c) {
        if (t >= t1) return false;
        const int KS = cls ? KS1 : KS0;
        w.cls = 2 * gemm + cls;
        w.b = b;
        w.rot = 0;
        w.ka = k;
        const long long room = t1 - t;
        w.kb = room < (long long)(KS - k) ? k + (int)room : KS;
        const long long us = t - k;  // first step of the unit
        if (cls == 0) {
            w.unit = g * MB0 + b;
            w.expert = cur.x;
            w.rows = cur.y;
            w.perm_off = cur.z;
            w.row_off = cur.w;
            w.gidx = g;
        } else {
            w.unit = ngroups * MB0 + b;
            w.expert = 0;
            w.rows = M;
            w.perm_off = M * ktop;
            w.row_off = 0;
            w.gidx = 0;
        }
        w.np = 1;
        if (w.ka != 0 || w.kb != KS) {
            // the unit is cut between CTAs c_first..c_last; each CTA has two slots (for
            // the unit its range starts in and the one it ends in)
            const int c_first = cta_of(us, G), c_last = cta_of(us + KS - 1, G);
            w.np = c_last - c_first + 1;
            w.s0 = 2 * c_first + (start(c_first, G) < us ? 1 : 0);
            w.sb = 2 * c_first;
            w.sstride = 2;
            w.myslot = 2 * c + ((c == c_first && start(c, G) < us) ? 1 : 0);
        }
        t += w.kb - w.ka;
        k = w.kb;
        if (k == KS) {
            k = 0;
            if (++b == (cls ? MB1 : MB0)) {
                b = 0;
                if (cls == 0) {
                    if (++g == ngroups) {
                        cls = 1;
                    } else {
                        cur = nxt;
                        nxt = ld_group(groups + (g + 1 < ngroups ? g + 1 : g));
                    }
                }
            }
        }
        return true;
    }
};

// Dynamic schedule: the units in order (routed units in group order, then the shared
// expert's) are handed out by a counter. The first Uh units go whole, Cu consecutive units
// per grab (at least 32 steps, so the counter's round trip hides behind the copies); the
// last Ut = min(U, CTAs) units go one per grab, cut into P = clamp(KS / 8, 1, 4) pieces.
// Head grab w takes chunk (w % G) * R + w / G (R = ceil(Nh / G); indices past the head
// are skipped): the G grabs in flight at any time read G regions spread over the weights,
// each region in order, as the static ranges do, which HBM serves faster than G
// neighbouring chunks.
struct DynList {
    int NRU, U, U0, Uh, Urt, Ust, P0, P1, Cu, Nh, R, Wh, W, G;
    int gemm, MB0, KS0, KS1, M, ktop;
    // The pool of GEMM gm: units [U0_, U).
    __device__ void init(const GemmParams& p, int gm, int ngroups, int G_, int U0_) {
        G = G_;
        U0 = U0_;
        gemm = gm;
        MB0 = p.cls[gm][0].MB;
        KS0 = p.cls[gm][0].KS;
        KS1 = p.cls[gm][1].KS;
        M = p.M;
        ktop = p.k;
        NRU = ngroups * MB0;
        const int Ush = p.has_shared ? p.cls[gm][1].MB : 0;
        U = NRU + Ush;
        const int Up = U - U0;
        const int Ut = Up < G ? Up : G;
        Uh = Up - Ut;
        Ust = Ut < Ush ? Ut : Ush;
        Urt = Ut - Ust;
        P0 = min(max(KS0 / 8, 1), kMaxPieces);
        P1 = min(max(KS1 / 8, 1), kMaxPieces);
        Cu = (32 + KS0 - 1) / KS0;
        Nh = (Uh + Cu - 1) / Cu;
        R = (Nh + G - 1) / G;
        Wh = R * G;
        W = Wh + Urt * P0 + Ust * P1;
    }
    // Grab w < W: units [ub, ue), whole (P = 1, ti = -1) or piece pc of P of tail unit ti;
    // ub == ue for a skipped head index.
    __device__ __forceinline__ void grab(int w, int& ub, int& ue, int& pc, int& P, int& ti) const {
        if (w < Wh) {
            const int ch = (w % G) * R + w / G;
            ub = ch * Cu;
            if (ub > Uh) ub = Uh;
            ue = ub + Cu < Uh ? ub + Cu : Uh;
            ub += U0;
            ue += U0;
            pc = 0;
            P = 1;
            ti = -1;
            return;
        }
        const int i = w - Wh;
        if (i < Urt * P0) {
            ti = i / P0;
            pc = i - ti * P0;
            P = P0;
        } else {
            const int j = i - Urt * P0;
            const int q = j / P1;
            ti = Urt + q;
            pc = j - q * P1;
            P = P1;
        }
        ub = U0 + Uh + ti;
        ue = ub + 1;
    }
    __device__ __forceinline__ int group_of(int u) const { return u < NRU ? u / MB0 : -1; }
    // Item of unit u (piece pc of P, tail index ti) with the record grp of its group
    // (ignored for the shared expert).
    __device__ __forceinline__ void item(int u, int pc, int P, int ti, int4 grp, WorkItem& it) const {
        const bool routed = u < NRU;
        const int KS = routed ? KS0 : KS1;
        it.cls = 2 * gemm + (routed ? 0 : 1);
        it.unit = u;
        if (routed) {
            const int g = u / MB0;
            it.b = u - g * MB0;
            it.expert = grp.x;
            it.rows = grp.y;
            it.perm_off = grp.z;
            it.row_off = grp.w;
            it.gidx = g;
        } else {
            it.b = u - NRU;
            it.expert = 0;
            it.rows = M;
            it.perm_off = M * ktop;
            it.row_off = 0;
            it.gidx = 0;
        }
        it.np = P;
        it.ka = pc * KS / P;
        it.kb = (pc + 1) * KS / P;
        // CTAs that run at the same time work on neighbouring units; starting each unit's
        // K loop at a different step keeps them off the same activation tile (one L2 slice)
        it.rot = u % (it.kb - it.ka);
        if (P > 1) {
            it.s0 = it.sb = kPoolSlot0 + kMaxPieces * ti;
            it.sstride = 1;
            it.myslot = kPoolSlot0 + kMaxPieces * ti + pc;
        }
    }
};

// One ring slot whose activation copies wait for the gate_up counter `dep` (both GEMMs in
// one launch): sources, the slot's shared address and full barrier, bytes, its ring
// position and its item's queue index.
struct Deferred {
    const uint8_t* b;
    const uint8_t* s;
    uint32_t stage, fb, bb, sb;
    int pos, q, dep;
};
static_assert(sizeof(Deferred) * kMaxStages <= kDeferBytes, "deferred-copy list");

struct GemmSmem {
    uint8_t* ring;
    float* stg;          // [Mpad][128] fp32 epilogue staging
    WorkItem* queue;     // [kGemmQueue]
    Deferred* defer;     // [kMaxStages] producer only
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;     // [2] per MMA issuer
    uint64_t* sf_ready;  // [S] scale factors of the stage are in tensor memory
    uint64_t* sf_drain;  // [4] per copy warp
    uint64_t* q_full;    // [kGemmQueue] item published
    uint64_t* q_empty;   // [kGemmQueue] item read by every consuming role
    uint32_t* tmem_base;
    int* abort_flag;
    int* bcast;
    int* never;  // stays 0: lets the exit-time drains ignore the abort flag
    int* tok;    // [64] tokens of the current group (epilogue)
};

__device__ __forceinline__ void set_error(int32_t* status, int* abort_flag, int code) {
    atomicCAS(status, 0, code);
    *(volatile int*)abort_flag = 1;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Waits until *ctr >= target (acquire, bounded by lim ns or the abort flag), then orders
// this thread's later bulk copies (async proxy) after what the acquire made visible.
__device__ __forceinline__ bool wait_at_least(const int32_t* ctr, int target, volatile int* abort, uint64_t lim) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) break;
        if (i == 0) {
            t0 = globaltimer();
        } else if ((i & 15) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > lim) return false;
        }
        __nanosleep(128);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// One look at *ctr: true (with the same ordering as wait_at_least) when it is >= target.
__device__ __forceinline__ bool poll_at_least(const int32_t* ctr, int target) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v < target) return false;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Reads queue entry i, waiting until it is published; false on a timeout.
__device__ __forceinline__ bool q_read(const GemmSmem& sm, int i, WorkItem& w, volatile int* abort, uint64_t lim) {
    const int qi = i % kGemmQueue;
    if (!mbar_wait_bounded(smem_u32(&sm.q_full[qi]), (uint32_t)(i / kGemmQueue) & 1u, abort, lim))
        return false;
    w = sm.queue[qi];
    return true;
}

// Issues this issuer's MMAs of one item: the steps of [ka, kb) that sit in ring slots of
// parity par (step j = kk - ka of the item with j % 2 == par), accumulated into d_tmem
// (the first of them overwrites it); the ring position advances over every step. Returns
// -1 on a timeout, else the number of steps issued. At small N the issue stream of a
// thread, not the tensor pipe, limits the rate, so every descriptor is precomputed and
// advanced with integer adds (a shared-memory descriptor holds address >> 4 in its low 14
// bits: +16 bytes is +1) and the format branch is taken once per item.
template <int FMT, bool CP>
__device__ __forceinline__ int mma_segment(uint32_t ready0, uint32_t empty0, Ring& rg, int ka, int kb, int par,
                                           uint64_t adesc0, uint64_t bdesc0, uint64_t sfadesc0, uint64_t sfbdesc0,
                                           uint32_t stage16, uint32_t d_tmem, uint32_t sf_t0, uint32_t sf_stride,
                                           uint32_t sfb_cols, uint32_t N, volatile int* abort, uint64_t lim) {
    static_assert(!(CP && FMT == MOE_FMT_NVFP4), "NVFP4 scales are copied by the copy warps");
    uint32_t id[4];
#pragma unroll
    for (int sub = 0; sub < 4; ++sub)
        id[sub] = FMT == MOE_FMT_MXFP8   ? idesc_mxf8(N, sub)
                  : FMT == MOE_FMT_MXFP4 ? idesc_mxf4(N, 2 * (sub % 2))
                  : FMT == MOE_FMT_NVFP4 ? idesc_nvf4(N)
                                         : idesc_bf16(N);
    int issued = 0;
    for (int kk = ka; kk < kb; ++kk, rg.adv1()) {
        const int st = rg.st;
        if ((st & 1) != par) continue;
        if (!mbar_wait_bounded(ready0 + 8u * st, rg.ph, abort, lim)) return -1;
        tc_fence_after();
        const uint64_t so = (uint64_t)st * stage16;
        const uint64_t ad = adesc0 + so, bd = bdesc0 + so;
        const uint32_t sfa = sf_t0 + (uint32_t)st * sf_stride, sfb = sfa + sfb_cols;
        const uint32_t acc0 = issued ? 1u : 0u;
        if (FMT == MOE_FMT_MXFP8) {
            if (CP) {
                tc_cp_sf(sfa, sfadesc0 + so);
                tc_cp_sf(sfb, sfbdesc0 + so);
            }
#pragma unroll
            for (int sub = 0; sub < 4; ++sub)
                mma_mxf8(d_tmem, ad + 2 * sub, bd + 2 * sub, id[sub], sfa, sfb, sub ? 1u : acc0);
        } else if (FMT == MOE_FMT_MXFP4) {
            // two scale atoms per step; MMA sub reads atom sub / 2, byte pair 2 * (sub % 2)
            if (CP) {
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    tc_cp_sf(sfa + 4 * a, sfadesc0 + so + 32 * a);
                    tc_cp_sf(sfb + 4 * a, sfbdesc0 + so + 32 * a);
                }
            }
#pragma unroll
            for (int sub = 0; sub < 4; ++sub)
                mma_mxf4(d_tmem, ad + 2 * sub, bd + 2 * sub, id[sub], sfa + 4 * (sub / 2), sfb + 4 * (sub / 2),
                         sub ? 1u : acc0);
        } else if (FMT == MOE_FMT_NVFP4) {
#pragma unroll
            for (int sub = 0; sub < 4; ++sub)
                mma_nvf4(d_tmem, ad + 2 * sub, bd + 2 * sub, id[sub], sfa + 4 * sub, sfb + 4 * sub, sub ? 1u : acc0);
        } else {
#pragma unroll
            for (int sub = 0; sub < 4; ++sub) mma_bf16(d_tmem, ad + 2 * sub, bd + 2 * sub, id[sub], sub ? 1u : acc0);
        }
        tc_commit(empty0 + 8u * st);
        ++issued;
    }
    return issued;
}

__global__ void __launch_bounds__(kGemmThreads, 1) k_expert_gemm(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int S = p.stages;
    // roles that read every queue entry: 2 issuers, 4 epilogue warps, 4 copy warps
    const uint32_t n_cons = 6u + (p.sf_warps ? 4u : 0u);

    // ---- shared-memory carve-up
    GemmSmem sm;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    sm.ring = base;
    sm.stg = reinterpret_cast<float*>(base + (size_t)S * p.stage_bytes);
    sm.queue = reinterpret_cast<WorkItem*>(sm.stg + p.Mpad * kBlockRows);
    sm.defer = reinterpret_cast<Deferred*>(sm.queue + kGemmQueue);
    sm.full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sm.defer) + kDeferBytes);
    sm.empty = sm.full + S;
    sm.acc_full = sm.empty + S;
    sm.acc_empty = sm.acc_full + kMaxAcc;
    sm.drain = sm.acc_empty + kMaxAcc;
    sm.sf_ready = sm.drain + 2;
    sm.sf_drain = sm.sf_ready + S;
    sm.q_full = sm.sf_drain + 4;
    sm.q_empty = sm.q_full + kGemmQueue;
    sm.tmem_base = reinterpret_cast<uint32_t*>(sm.q_empty + kGemmQueue);
    sm.abort_flag = reinterpret_cast<int*>(sm.tmem_base + 1);
    sm.bcast = sm.abort_flag + 1;
    sm.never = sm.abort_flag + 2;
    sm.tok = sm.abort_flag + 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            mbar_init(smem_u32(&sm.empty[i]), 1);
            mbar_init(smem_u32(&sm.sf_ready[i]), 4);  // one per copy warp
        }
        for (int i = 0; i < kMaxAcc; ++i) {
            mbar_init(smem_u32(&sm.acc_full[i]), 2);  // one per MMA issuer
            mbar_init(smem_u32(&sm.acc_empty[i]), 4);  // one per epilogue warp
        }
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&sm.drain[i]), 1);
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&sm.sf_drain[i]), 1);
        for (int i = 0; i < kGemmQueue; ++i) {
            mbar_init(smem_u32(&sm.q_full[i]), 1);
            mbar_init(smem_u32(&sm.q_empty[i]), n_cons);
        }
        *sm.abort_flag = 0;
        *sm.never = 0;
        fence_mbar_init();
    }
    // The shared expert's weights do not depend on the routing: while the earlier kernels
    // of the step still run (HBM is otherwise idle then), every CTA prefetches its 1/G
    // share of them into L2. They are consumed at the end of the item list; the routed
    // weights streamed meanwhile carry an evict-first hint.
    if (threadIdx.x == 32 && p.has_shared && p.prefetch_shared) {
        const GemmClass& C1 = p.cls[p.mode == 1 ? 1 : 0][1];
        const size_t total = (size_t)C1.MB * C1.KS * record_bytes(C1.fmt);
        const size_t share = (total / gridDim.x + 15) & ~(size_t)15;
        const size_t b0 = (size_t)blockIdx.x * share;
        const size_t b1 = b0 + share < total ? b0 + share : total;
        for (size_t o = b0; o < b1; o += 65536) {
            const size_t n = b1 - o < 65536 ? b1 - o : 65536;
            prefetch_l2(C1.w + o, (uint32_t)n);
        }
    }
    // Tensor memory does not depend on earlier launches either (no kernel before this one in
    // the step holds any, and two GEMM CTAs never share an SM): allocate it before the wait.
    if (warp == 1) {
        tmem_alloc(smem_u32(sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_base;
    // two accumulator banks of nacc buffers (Mpad columns each): the MMA issuers run up to
    // nacc - 1 items ahead of the epilogue
    const int bank = acc_bank_cols(p.atoms_max, p.Mpad);
    const int nacc = min(kMaxAcc, bank / p.Mpad);
    // Everything below reads the previous launches' outputs.
    pdl_wait();
    const int ngroups = p.hdr->num_groups;
    pdl_trigger();

    // the GEMMs of this launch: gate_up (0), down (1) or both, gate_up's items first
    const int g_first = p.mode == 1 ? 1 : 0, g_last = p.mode == 0 ? 0 : 1;
    auto units_of = [&](int gm) { return ngroups * p.cls[gm][0].MB + (p.has_shared ? p.cls[gm][1].MB : 0); };
    // units at the end of the list handed out from the counter (single-GEMM launches only)
    auto pool_of = [&](int gm) {
        const int Ua = units_of(gm);
        return p.mode == 2 ? 0 : (p.pool_units < 0 || p.pool_units > Ua ? Ua : p.pool_units);
    };
    const bool dyn = pool_of(g_first) > 0;
    const int c = blockIdx.x;
    volatile int* abort_flag = sm.abort_flag;
    const uint64_t wlim = p.wait_ns;  // limit of every wait

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            Ring rg{0, 0u, S};
            uint32_t issued_mask = 0;  // stages with a copy in flight at least once
            bool ok = true;
            int qn = 0;  // items published
            // Both GEMMs in one launch: a down item reads its group's hidden activations,
            // written by the gate_up epilogues of any CTA. Its weight copies go out at once;
            // its activation copies wait here, in ring order, until the group's gate_up
            // counter is complete. So the ring fills with down weights while the last
            // gate_up units finish. A deferred slot is issued before anything could wait on
            // it: before its ring slot comes round again, and before its item's queue entry
            // is needed again.
            Deferred* dq = sm.defer;
            int dh = 0, dt = 0;  // deferred slots issued / recorded
            int pos = 0;         // ring slots filled so far (bubbles included)
            int met = -1;        // group counter known to be complete (gu_done index)
            auto dep_target = [&](int d) { return p.cls[0][d == kMaxE ? 1 : 0].MB + p.dep_extra; };
            auto issue_b = [&](const Deferred& e) {
                bulk_g2s(e.stage + p.b_off, e.b, e.bb, e.fb);
                if (e.sb) bulk_g2s(e.stage + p.sfb_off, e.s, e.sb, e.fb);
            };
            // issues deferred slots from the front while their groups are complete; waits
            // for the group of a slot at ring position <= pos_lim or of item <= q_lim
            auto drain = [&](int pos_lim, int q_lim) -> bool {
                while (dh < dt) {
                    const Deferred& e = dq[dh % kMaxStages];
                    if (e.dep != met) {
                        if (e.pos <= pos_lim || e.q <= q_lim) {
                            if (!wait_at_least(p.gu_done + e.dep, dep_target(e.dep), abort_flag, wlim)) return false;
                        } else if (!poll_at_least(p.gu_done + e.dep, dep_target(e.dep))) {
                            return true;
                        }
                        met = e.dep;
                    }
                    issue_b(e);
                    ++dh;
                }
                return true;
            };
            // Publishes one item and issues its copies (plus the bubble after an odd count);
            // dep >= 0: the gu_done counter the item's activations wait for.
            auto issue = [&](const WorkItem& it, int dep) -> bool {
                const int qi = qn % kGemmQueue;
                if (dh < dt && !drain(INT_MIN, qn - kGemmQueue)) return false;
                if (!mbar_wait_bounded(smem_u32(&sm.q_empty[qi]), ((uint32_t)(qn / kGemmQueue) & 1u) ^ 1u, abort_flag,
                                       wlim))
                    return false;
                sm.queue[qi] = it;
                mbar_arrive(smem_u32(&sm.q_full[qi]));
                ++qn;
                const GemmClass& C = p.cls[it.cls >> 1][it.cls & 1];
                const int A = atoms_per_step(C.fmt);
                const uint32_t REC = record_bytes(C.fmt);
                int Rpad;
                const uint8_t *bsrc, *bssrc;
                if ((it.cls >> 1) == 0) {  // gate_up: all rows of x
                    Rpad = p.Mpad;
                    bsrc = C.b;
                    bssrc = C.bs;
                } else {  // down: the group's rows of the hidden activations
                    Rpad = ((it.cls & 1) == 0) ? round_up(it.rows, 16) : p.Mpad;
                    bsrc = C.b + (size_t)it.row_off * C.KS * kStepBytes;
                    bssrc = C.bs + (size_t)it.gidx * C.KS * A * kAtomBytes;
                }
                const uint8_t* wrec0 = C.w + ((size_t)((size_t)it.expert * C.MB + it.b) * C.KS + it.ka) * REC;
                const uint32_t bbytes = (uint32_t)Rpad * kStepBytes;
                const int nst = it.kb - it.ka;
                int jr = it.rot;  // step of the item at position j
                for (int j = 0; j < nst + (nst & 1); ++j, rg.adv1(), ++pos) {
                    const int st = rg.st;
                    if (dh < dt && !drain(pos - S, INT_MIN)) return false;
                    if (!mbar_wait_bounded(smem_u32(&sm.empty[st]), rg.ph ^ 1u, abort_flag, wlim))
                        return false;
                    const uint32_t fb = smem_u32(&sm.full[st]);
                    issued_mask |= 1u << st;
                    if (j == nst) {  // bubble: the slot completes with no data
                        mbar_arrive(fb);
                        continue;
                    }
                    const int kk = it.ka + jr;
                    if (++jr == nst) jr = 0;
                    const uint32_t stage = smem_u32(sm.ring + (size_t)st * p.stage_bytes);
                    mbar_arrive_expect_tx(fb, REC + bbytes + (uint32_t)A * kAtomBytes);
                    bulk_g2s_hint(stage + p.a_off, wrec0 + (size_t)(kk - it.ka) * REC, REC, fb, pol);
                    const Deferred e{bsrc + (size_t)kk * bbytes, bssrc + (size_t)kk * A * kAtomBytes, stage, fb, bbytes,
                                     (uint32_t)A * kAtomBytes, pos, qn - 1, dep};
                    if (dep < 0 || dep == met) {
                        issue_b(e);
                    } else if (dh == dt && poll_at_least(p.gu_done + dep, dep_target(dep))) {
                        met = dep;
                        issue_b(e);
                    } else {
                        dq[dt % kMaxStages] = e;
                        ++dt;
                    }
                }
                return true;
            };
            WorkItem it;
            for (int gm = g_first; ok && gm <= g_last; ++gm) {
            if (gm == 1 && p.mode == 2 && p.has_shared && p.prefetch_shared) {
                // as the down launch does before its wait: this CTA's share of the down
                // GEMM's shared-expert weights into L2 while the gate_up units finish (in a
                // step the router launch has prefetched them already)
                const GemmClass& C1 = p.cls[1][1];
                const size_t total = (size_t)C1.MB * C1.KS * record_bytes(C1.fmt);
                const size_t share = (total / gridDim.x + 15) & ~(size_t)15;
                const size_t b0 = (size_t)blockIdx.x * share;
                const size_t b1 = b0 + share < total ? b0 + share : total;
                for (size_t o = b0; o < b1; o += 65536)
                    prefetch_l2(C1.w + o, (uint32_t)(b1 - o < 65536 ? b1 - o : 65536));
            }
            const int Up = pool_of(gm), U0 = units_of(gm) - Up;  // [0, U0) static, [U0, U) pool
            const long long Tst = Walker::steps_before(p, gm, ngroups, U0);
            // static part: never more CTAs than steps, so every working CTA owns at least one
            // step and the CTAs whose ranges meet a unit are exactly its pieces
            const int G = (int)((long long)gridDim.x < Tst ? (long long)gridDim.x : Tst);
            {
                Walker wk;
                wk.init(p, gm, ngroups, G, c, U0);
                const bool deps = gm == 1 && p.mode == 2;  // down items after gate_up in one launch
                while (ok && wk.next(it, G, c)) ok = issue(it, deps ? ((it.cls & 1) ? kMaxE : it.gidx) : -1);
            }
            if (ok && Up > 0) {
                DynList dl;
                dl.init(p, gm, ngroups, gridDim.x, U0);
                // grab w0 in hand with the records of its first unit's group ga0 and ga0 + 1;
                // w1 taken; w2 requested while w0's copies go out
                auto preload = [&](int w, int& ga, int4& ra, int4& rb) {
                    int ub, ue, pc, P, ti;
                    dl.grab(w, ub, ue, pc, P, ti);
                    ga = dl.group_of(ub);
                    if (ga >= 0) {
                        ra = ld_group(p.groups + ga);
                        rb = ld_group(p.groups + (ga + 1 < ngroups ? ga + 1 : ga));
                    }
                };
                int ga0 = -1;
                int4 r0a = make_int4(0, 0, 0, 0), r0b = r0a;
                int w0 = atomicAdd(p.sched, 1), w1 = dl.W;
                if (w0 < dl.W) {
                    preload(w0, ga0, r0a, r0b);
                    w1 = atomicAdd(p.sched, 1);
                }
                while (ok && w0 < dl.W) {
                    int w2 = dl.W, ga1 = -1;
                    int4 r1a = make_int4(0, 0, 0, 0), r1b = r1a;
                    if (w1 < dl.W) {
                        w2 = atomicAdd(p.sched, 1);  // used one grab later
                        preload(w1, ga1, r1a, r1b);
                    }
                    int ub, ue, pc, P, ti;
                    dl.grab(w0, ub, ue, pc, P, ti);
                    for (int u = ub; u < ue; ++u) {
                        const int g = dl.group_of(u);
                        int4 rec = r0a;
                        if (g >= 0 && g != ga0) rec = (g == ga0 + 1) ? r0b : ld_group(p.groups + g);
                        dl.item(u, pc, P, ti, rec, it);
                        if (!issue(it, -1)) {
                            ok = false;
                            break;
                        }
                    }
                    w0 = w1;
                    w1 = w2;
                    ga0 = ga1;
                    r0a = r1a;
                    r0b = r1b;
                }
            }
            }
            if (ok && dh < dt) ok = drain(INT_MAX, INT_MAX);
            if (!ok) set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
            // after a timeout, slots still deferred get their activation copies anyway (stale
            // data that no MMA reads: the other roles have seen the abort flag), so that every
            // stage's barrier completes and the drain below finds no copy missing
            while (dh < dt) {
                issue_b(dq[dh % kMaxStages]);
                ++dh;
            }
            // the end marker
            if (ok) {
                const int qi = qn % kGemmQueue;
                if (mbar_wait_bounded(smem_u32(&sm.q_empty[qi]), ((uint32_t)(qn / kGemmQueue) & 1u) ^ 1u, abort_flag,
                                      wlim)) {
                    sm.queue[qi].cls = -1;
                    mbar_arrive(smem_u32(&sm.q_full[qi]));
                } else {
                    set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                }
            }
            // make sure no copy is still writing shared memory when the CTA exits: wait for
            // the last phase issued on every stage (stages < st were issued in lap ph,
            // the others in lap ph ^ 1)
            for (int i = 0; i < S; ++i) {
                if (!(issued_mask >> i & 1u)) continue;
                const uint32_t par = (i < rg.st) ? rg.ph : (rg.ph ^ 1u);
                mbar_wait_bounded(smem_u32(&sm.full[i]), par, sm.never, wlim / 2);
            }
        }
    } else if (warp == 1 || warp == 6) {
        // ================================================================ MMA issuers
        // warp 1 consumes the even ring slots (bank 0), warp 6 the odd ones (bank 1)
        if (lane == 0) {
            const int par = warp == 6 ? 1 : 0;
            Ring rg{0, 0u, S};
            int ab = 0;
            uint32_t acc_ph = 0u;  // bit b: phase of accumulator buffer b
            const int am = p.atoms_max;
            // with copy warps the issuers wait for the stage's scales, else for its data
            const uint32_t wait0 = p.sf_warps ? smem_u32(&sm.sf_ready[0]) : smem_u32(&sm.full[0]);
            const uint32_t empty0 = smem_u32(&sm.empty[0]);
            const uint32_t ring = smem_u32(sm.ring);
            const uint64_t adesc0 = smem_desc(ring + p.a_off, 16, 1024, 2);
            const uint64_t bdesc0 = smem_desc(ring + p.b_off, 16, 1024, 2);
            const uint64_t sfadesc0 = smem_desc(ring + p.sfa_off, 0, 128, 0);
            const uint64_t sfbdesc0 = smem_desc(ring + p.sfb_off, 0, 128, 0);
            const uint32_t stage16 = (uint32_t)p.stage_bytes >> 4;
            const uint32_t sf_t0 = tmem + 2 * bank;
            const uint32_t bank_t = tmem + (uint32_t)(par * bank);
            for (int qn = 0;; ++qn) {
                WorkItem it;
                if (!q_read(sm, qn, it, abort_flag, wlim)) {
                    set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive(smem_u32(&sm.q_empty[qn % kGemmQueue]));
                if (it.cls < 0) break;
                const GemmClass& C = p.cls[it.cls >> 1][it.cls & 1];
                const uint32_t N = (it.cls == 2) ? (uint32_t)round_up(it.rows, 16) : (uint32_t)p.Mpad;
                if (!mbar_wait_bounded(smem_u32(&sm.acc_empty[ab]), ((acc_ph >> ab) & 1u) ^ 1u, abort_flag,
                                       wlim)) {
                    set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = bank_t + (uint32_t)(ab * p.Mpad);
#define MOE_SEG(F, CPV)                                                                                        \
    mma_segment<F, CPV>(wait0, empty0, rg, it.ka, it.kb, par, adesc0, bdesc0, sfadesc0, sfbdesc0, stage16, d_tmem, \
                        sf_t0, 8 * am, 4 * am, N, abort_flag, wlim)
                // launches with NVFP4 weights always have the copy warps (host invariant)
                int n;
                if (p.sf_warps) {
                    if (C.fmt == MOE_FMT_MXFP8) n = MOE_SEG(MOE_FMT_MXFP8, false);
                    else if (C.fmt == MOE_FMT_NVFP4) n = MOE_SEG(MOE_FMT_NVFP4, false);
                    else if (C.fmt == MOE_FMT_MXFP4) n = MOE_SEG(MOE_FMT_MXFP4, false);
                    else n = MOE_SEG(MOE_FMT_BF16, false);
                } else {
                    if (C.fmt == MOE_FMT_MXFP8) n = MOE_SEG(MOE_FMT_MXFP8, true);
                    else if (C.fmt == MOE_FMT_MXFP4) n = MOE_SEG(MOE_FMT_MXFP4, true);
                    else if (C.fmt == MOE_FMT_BF16) n = MOE_SEG(MOE_FMT_BF16, true);
                    else {
                        set_error(p.status, sm.abort_flag, MOE_ERR_UNSUPPORTED);
                        break;
                    }
                }
#undef MOE_SEG
                if (n < 0) {
                    set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                    break;
                }
                // after an item of odd length the next slot is a bubble: its owner hands it
                // back to the producer
                if ((it.kb - it.ka) & 1) {
                    if ((rg.st & 1) == par) {
                        if (!mbar_wait_bounded(wait0 + 8u * rg.st, rg.ph, abort_flag, wlim)) {
                            set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                            break;
                        }
                        mbar_arrive(empty0 + 8u * rg.st);
                    }
                    rg.adv1();
                }
                // an item with no step in this issuer's slots (a single step) leaves its bank
                // untouched (the epilogue skips it) and only reports the buffer done
                if (n > 0) tc_commit(smem_u32(&sm.acc_full[ab]));
                else mbar_arrive(smem_u32(&sm.acc_full[ab]));
                acc_ph ^= 1u << ab;
                if (++ab == nacc) ab = 0;
            }
            // wait until every issued MMA has completed before the TMEM is released
            tc_commit(smem_u32(&sm.drain[par]));
            mbar_wait_bounded(smem_u32(&sm.drain[par]), 0u, sm.never, wlim / 2);
        }
    } else if (warp >= 7) {
        // ================================================================ scale-factor copies
        // (launches with NVFP4 weights): warp 7 + j copies scale atoms 2 (j % 2) and
        // 2 (j % 2) + 1 of every stage, of the A operand for j < 2 and of B otherwise. Each
        // warp walks all steps in ring order, so a stage's scale columns are always written
        // by the same warp.
        if (lane == 0 && p.sf_warps) {
            const int j = warp - 7;
            const bool is_b = j >= 2;
            const int a0 = 2 * (j & 1);
            Ring rg{0, 0u, S};
            const int am = p.atoms_max;
            const uint32_t full0 = smem_u32(&sm.full[0]), ready0 = smem_u32(&sm.sf_ready[0]);
            const uint32_t ring = smem_u32(sm.ring);
            const uint64_t desc0 = smem_desc(ring + (is_b ? p.sfb_off : p.sfa_off), 0, 128, 0);
            const uint32_t stage16 = (uint32_t)p.stage_bytes >> 4;
            const uint32_t sf_t0 = tmem + 2 * bank + (is_b ? 4u * am : 0u);
            bool ok = true;
            for (int qn = 0; ok; ++qn) {
                WorkItem it;
                if (!q_read(sm, qn, it, abort_flag, wlim)) {
                    set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive(smem_u32(&sm.q_empty[qn % kGemmQueue]));
                if (it.cls < 0) break;
                const int A = atoms_per_step(p.cls[it.cls >> 1][it.cls & 1].fmt);
                const int a1 = A < a0 + 2 ? A : a0 + 2;
                const int nst = it.kb - it.ka;
                for (int s = 0; s < nst + (nst & 1); ++s, rg.adv1()) {
                    const int st = rg.st;
                    if (!mbar_wait_bounded(full0 + 8u * st, rg.ph, abort_flag, wlim)) {
                        set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    if (s < nst && a1 > a0) {
                        tc_fence_after();
                        const uint64_t sd = desc0 + (uint64_t)st * stage16;
                        const uint32_t sf = sf_t0 + (uint32_t)st * 8 * am;
                        for (int a = a0; a < a1; ++a) tc_cp_sf(sf + 4 * a, sd + 32 * a);
                        tc_commit(ready0 + 8u * st);
                    } else {
                        mbar_arrive(ready0 + 8u * st);
                    }
                }
            }
            tc_commit(smem_u32(&sm.sf_drain[j]));
            mbar_wait_bounded(smem_u32(&sm.sf_drain[j]), 0u, sm.never, wlim / 2);
        }
    } else {
        // ================================================================ epilogue
        const int q = warp % 4;           // TMEM lane quarter of this warp
        const int r = 32 * q + lane;      // accumulator row (weight row of the block)
        const int et = threadIdx.x - 64;  // 0..127
        const int ew = et / 32;
        int ab = 0;
        uint32_t acc_ph = 0u;
        float* stg = sm.stg;
        for (int qn = 0;; ++qn) {
            // one thread waits for the next item and for its accumulator; the barrier's AND
            // tells the others, so the 128 threads always leave the loop together. The
            // barrier also keeps the staging buffer from being refilled while any thread
            // still reads the previous item from it.
            const int qi = qn % kGemmQueue;
            bool ok = true;
            if (et == 0) {
                ok = mbar_wait_bounded(smem_u32(&sm.q_full[qi]), (uint32_t)(qn / kGemmQueue) & 1u, abort_flag,
                                       wlim);
                if (ok && sm.queue[qi].cls >= 0)
                    ok = mbar_wait_bounded(smem_u32(&sm.acc_full[ab]), (acc_ph >> ab) & 1u, abort_flag, wlim);
            }
            if (!named_bar_and(1, 128, ok)) {
                if (et == 0) set_error(p.status, sm.abort_flag, MOE_ERR_TIMEOUT);
                break;
            }
            const WorkItem it = sm.queue[qi];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.q_empty[qi]));
            if (it.cls < 0) break;
            const int gm = it.cls >> 1, cl = it.cls & 1;  // GEMM (0 gate_up, 1 down), class
            const GemmClass& C = p.cls[gm][cl];
            const int expert = it.expert, rows = it.rows, perm_off = it.perm_off, row_off = it.row_off, gidx = it.gidx;
            const int N = (it.cls == 2) ? round_up(rows, 16) : p.Mpad;
            acc_ph ^= 1u << ab;
            tc_fence_after();
            // bank b holds the item's steps j with j % 2 == b; a single-step item wrote bank
            // 0 only (the sum is bank 0 + bank 1, in that order)
            const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * p.Mpad);
            const bool two = it.kb - it.ka >= 2;
            // the NVFP4 global scales (weight x activation): loaded before the accumulator,
            // so that the load's latency overlaps the tensor-memory loads
            const float alpha = C.gs_w ? __ldg(C.gs_w + expert) * C.gs_a : 1.0f;
            // routed gate_up: the group's tokens (its rows' positions in x), loaded early too
            const int tok = (it.cls == 0 && et < rows) ? __ldg(p.perm + perm_off + et) / p.k : 0;
            if (gm == 1 && it.np == 1) {
                // a whole down unit: each thread writes its output feature (weight row r) of
                // every row of the group straight from the accumulator, with no staging and
                // no barrier; the same arithmetic as the staged path (bank 0 + bank 1, then
                // the scales)
                float* yb = p.y + (size_t)perm_off * p.H + kBlockRows * it.b + r;
                for (int c0 = 0; c0 < N; c0 += 16) {
                    uint32_t v0[16], v1[16];
                    tmem_ld16_nowait(t_row + (uint32_t)c0, v0);
                    if (two) tmem_ld16_nowait(t_row + (uint32_t)bank + (uint32_t)c0, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float a = two ? __uint_as_float(v0[i]) + __uint_as_float(v1[i]) : __uint_as_float(v0[i]);
                        if (c0 + i < rows) yb[(size_t)(c0 + i) * p.H] = a * alpha;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[ab]));
                if (++ab == nacc) ab = 0;
                continue;
            }
            for (int c0 = 0; c0 < N; c0 += 16) {
                uint32_t v0[16], v1[16];
                if (two) {
                    tmem_ld16_nowait(t_row + (uint32_t)c0, v0);
                    tmem_ld16_nowait(t_row + (uint32_t)bank + (uint32_t)c0, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        stg[(c0 + i) * kBlockRows + r] = __uint_as_float(v0[i]) + __uint_as_float(v1[i]);
                } else {
                    tmem_ld16_nowait(t_row + (uint32_t)c0, v0);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) stg[(c0 + i) * kBlockRows + r] = __uint_as_float(v0[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[ab]));
            if (++ab == nacc) ab = 0;
            // compact the selected columns: column of group row rg -> stg[rg][r]; the
            // group's tokens are read once (in parallel) into shared memory
            if (it.cls == 0) {
                if (et < rows) sm.tok[et] = tok;
                named_bar(1, 128);
                for (int rg = 0; rg < rows; ++rg) {
                    const int m = sm.tok[rg];
                    stg[rg * kBlockRows + r] = stg[m * kBlockRows + r];
                }
            }
            // a unit cut into pieces: store this piece's partial sum; the CTA finishing the
            // last piece adds them all, in piece order
            if (it.np > 1) {
                const int npieces = it.np;
                float* part = p.partials[gm] + (size_t)it.myslot * kPartialFloats;
                for (int rg = 0; rg < rows; ++rg) __stcg(part + rg * kBlockRows + r, stg[rg * kBlockRows + r]);
                __threadfence();
                named_bar(1, 128);
                if (et == 0) {
                    const int old = atomicAdd(p.counters[gm] + it.unit, 1);
                    *sm.bcast = (old == npieces - 1) ? 1 : 0;
                }
                named_bar(1, 128);
                const int last = *(volatile int*)sm.bcast;
                named_bar(1, 128);
                if (!last) continue;
                __threadfence();
                // loads of 8 rows x 4 pieces are issued before their adds (clamped
                // addresses keep them unconditional)
                for (int rg0 = 0; rg0 < rows; rg0 += 8) {
                    float sum[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) sum[i] = 0.0f;
                    for (int pc0 = 0; pc0 < npieces; pc0 += 4) {
                        float v[4][8];
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const int pc = min(pc0 + qq, npieces - 1);
                            const int slot = pc == 0 ? it.s0 : it.sb + pc * it.sstride;
                            const float* src = p.partials[gm] + (size_t)slot * kPartialFloats + r;
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[qq][i] = __ldcg(src + min(rg0 + i, rows - 1) * kBlockRows);
                        }
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq)
                            if (pc0 + qq < npieces)
#pragma unroll
                                for (int i = 0; i < 8; ++i) sum[i] += v[qq][i];
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (rg0 + i < rows) stg[(rg0 + i) * kBlockRows + r] = sum[i];
                }
                if (et == 0) p.counters[gm][it.unit] = 0;
            }
            named_bar(1, 128);
            // ---- final epilogue
            if (gm == 0) {
                // SwiGLU on (gate, up) = rows (fi, fi + 64); warps take 32 features each
                const int fi = 32 * (ew & 1) + lane;
                const int f = 64 * it.b + fi;  // feature in [0, I)
                const int Rp = (cl == 0) ? round_up(rows, 16) : p.Mpad;
                uint8_t* hq_g = C.hq + (cl == 0 ? (size_t)row_off * row_bytes(C.out_fmt, C.I) : 0);
                const int Aout = atoms_per_step(C.out_fmt);
                const int KSo = steps_of(C.out_fmt, C.I);
                uint8_t* hs_g = C.hs + (cl == 0 ? (size_t)gidx * KSo * Aout * kAtomBytes : 0);
                const float lim = p.swiglu_limit;
                for (int rg = (ew >> 1); rg < rows; rg += 2) {
                    float g = stg[rg * kBlockRows + fi] * alpha;
                    float u = stg[rg * kBlockRows + fi + 64] * alpha;
                    if (lim > 0.0f) {  // clamped SwiGLU: gate cut from above, up to [-lim, lim]
                        g = fminf(g, lim);
                        u = fminf(fmaxf(u, -lim), lim);
                    }
                    const float h = g / (1.0f + expf(-g)) * u;
                    if (C.out_fmt == MOE_FMT_MXFP8) {
                        const float amax = warp_max_f(fabsf(h));
                        const int e = mx_exponent(amax);
                        const uint32_t qb = e4m3(__fmul_rn(h, exp2_int(-e)));
                        // gather 4 consecutive features into one word
                        const uint32_t b1 = __shfl_down_sync(0xffffffffu, qb, 1);
                        const uint32_t b2 = __shfl_down_sync(0xffffffffu, qb, 2);
                        const uint32_t b3 = __shfl_down_sync(0xffffffffu, qb, 3);
                        const int sidx = f / 128, cb = f % 128;
                        if ((lane & 3) == 0) {
                            uint8_t* row = hq_g + (size_t)sidx * Rp * kStepBytes + (size_t)rg * kStepBytes;
                            *reinterpret_cast<uint32_t*>(row + (((cb / 16) ^ (rg & 7)) * 16) + (cb % 16)) =
                                qb | (b1 << 8) | (b2 << 16) | (b3 << 24);
                        }
                        if (lane == 0)
                            hs_g[(size_t)sidx * kAtomBytes + (rg % 32) * 16 + (rg / 32) * 4 + (cb / 32)] = (uint8_t)(e + 127);
                    } else if (C.out_fmt == MOE_FMT_MXFP4) {
                        // one 32-feature block per warp: E8M0 exponent of the rule amax <= 6 * 2^e
                        const float amax = warp_max_f(fabsf(h));
                        const int e = mx4_exponent(amax);
                        const uint32_t nib = e2m1x2(0.0f, __fmul_rn(h, exp2_int(-e))) & 0xFu;
                        const uint32_t nb1 = __shfl_down_sync(0xffffffffu, nib, 1);
                        const uint32_t byte = nib | (nb1 << 4);
                        const uint32_t y1 = __shfl_down_sync(0xffffffffu, byte, 2);
                        const uint32_t y2 = __shfl_down_sync(0xffffffffu, byte, 4);
                        const uint32_t y3 = __shfl_down_sync(0xffffffffu, byte, 6);
                        const int sidx = f / 256, cbyte = (f % 256) / 2;
                        if ((lane & 7) == 0) {
                            uint8_t* row = hq_g + (size_t)sidx * Rp * kStepBytes + (size_t)rg * kStepBytes;
                            *reinterpret_cast<uint32_t*>(row + (((cbyte / 16) ^ (rg & 7)) * 16) + (cbyte % 16)) =
                                (byte & 0xFFu) | ((y1 & 0xFFu) << 8) | ((y2 & 0xFFu) << 16) | ((y3 & 0xFFu) << 24);
                        }
                        if (lane == 0) {
                            const int j = (f % 256) / 32;
                            hs_g[(size_t)sidx * 2 * kAtomBytes + (j / 4) * kAtomBytes + (rg % 32) * 16 + (rg / 32) * 4 +
                                 (j % 4)] = (uint8_t)(e + 127);
                        }
                    } else if (C.out_fmt == MOE_FMT_NVFP4) {
                        float amax = fabsf(h);
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                        const uint8_t s8 = nv_scale(amax, C.gs_out);
                        const float dsc = e4m3_to_f32(s8);
                        const float denom = __fmul_rn(dsc, C.gs_out);
                        const uint32_t nib = (dsc != 0.0f) ? (e2m1x2(0.0f, __fdiv_rn(h, denom)) & 0xFu) : 0u;
                        // byte of features (2j, 2j+1): low nibble even feature
                        const uint32_t nb1 = __shfl_down_sync(0xffffffffu, nib, 1);
                        const uint32_t byte = nib | (nb1 << 4);
                        const uint32_t y1 = __shfl_down_sync(0xffffffffu, byte, 2);
                        const uint32_t y2 = __shfl_down_sync(0xffffffffu, byte, 4);
                        const uint32_t y3 = __shfl_down_sync(0xffffffffu, byte, 6);
                        const int sidx = f / 256, cbyte = (f % 256) / 2;
                        if ((lane & 7) == 0) {
                            uint8_t* row = hq_g + (size_t)sidx * Rp * kStepBytes + (size_t)rg * kStepBytes;
                            *reinterpret_cast<uint32_t*>(row + (((cbyte / 16) ^ (rg & 7)) * 16) + (cbyte % 16)) =
                                (byte & 0xFFu) | ((y1 & 0xFFu) << 8) | ((y2 & 0xFFu) << 16) | ((y3 & 0xFFu) << 24);
                        }
                        if ((lane & 15) == 0) {
                            const int b16 = (f % 256) / 16;
                            hs_g[(size_t)sidx * 4 * kAtomBytes + (b16 / 4) * kAtomBytes + (rg % 32) * 16 + (rg / 32) * 4 +
                                 (b16 % 4)] = s8;
                        }
                    } else {  // BF16 FC2 input
                        const uint32_t hb = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h));
                        const uint32_t hb1 = __shfl_down_sync(0xffffffffu, hb, 1);
                        const int sidx = f / 64, cbyte = (f % 64) * 2;
                        if ((lane & 1) == 0) {
                            uint8_t* row = hq_g + (size_t)sidx * Rp * kStepBytes + (size_t)rg * kStepBytes;
                            *reinterpret_cast<uint32_t*>(row + (((cbyte / 16) ^ (rg & 7)) * 16) + (cbyte % 16)) =
                                hb | (hb1 << 16);
                        }
                    }
                }
            } else {
                const int n = kBlockRows * it.b + et;
                for (int rg = 0; rg < rows; ++rg) {
                    const int pos = perm_off + rg;
                    p.y[(size_t)pos * p.H + n] = stg[rg * kBlockRows + et] * alpha;
                }
            }
            if (p.mode == 2 && gm == 0) {
                // the unit's hidden activations are complete: order the stores before the
                // down items' bulk copies (async proxy) in other CTAs, then count the unit
                asm volatile("fence.proxy.async.global;" ::: "memory");
                named_bar(1, 128);
                if (et == 0) {
                    __threadfence();
                    atomicAdd(p.gu_done + (cl ? kMaxE : gidx), 1);
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // both GEMMs in one launch: the last CTA to finish resets the group counters
    if (p.mode == 2) {
        if (threadIdx.x == 0) {
            __threadfence();
            sm.bcast[0] = atomicAdd(p.gu_done + kMaxE + 1, 1) == (int)gridDim.x - 1 ? 1 : 0;
        }
        __syncthreads();
        if (sm.bcast[0]) {
            for (int i = threadIdx.x; i < ngroups; i += blockDim.x) p.gu_done[i] = 0;
            if (threadIdx.x == 0) {
                p.gu_done[kMaxE] = 0;
                p.gu_done[kMaxE + 1] = 0;
            }
            __threadfence();
        }
    }
    // pool: the last CTA to finish resets the item counter for the next launch
    if (dyn && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
            p.sched[0] = 0;
            p.sched[1] = 0;
            __threadfence();
        }
    }
}

}  // namespace moe
