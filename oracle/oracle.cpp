// CPU oracle for the small-M MoE decode/verify layer step.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, single-threaded definition
// that the CUDA path is checked against. Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load it. It shares no code, header, table or
// helper with the CUDA library; the two never include or link each other.
//
// Everything is computed in IEEE double unless a step is defined in fp32 (the
// activation quantisation, the fp32 sigmoid score and the fp32 selection key).
// It must be compiled with -ffp-contract=off so that no multiply-add is fused.
//
// Sources (page title, section):
//  [README]  "SGLang-NVIDIA-Mega", slot table of "What a covered DeepSeek-V4.1-Flash
//            step runs" (rows hop_b, moe, gate, shared_ll, two_shot) and the Qwen3.5
//            slot tables (rows route, mkm, route_shared).
//  [PR24]    "sgl-nvidia-mega pull request 24" (GLM-5.3 specs), "Modifications /
//            Target spec": one expert group, sigmoid scores, renormalised top-8;
//            moe_split row maps give the same bytes.
//  [GB10]    "SGLang Spark GB10 Optimizations", "Key Optimizations 1": the MoE sum
//            takes a routed_scaling_factor.
//  Block formats follow the OCP Microscaling (MX) definitions of E4M3, E2M1 and
//  E8M0 (MXFP8: E4M3 + E8M0 per 32; MXFP4: packed E2M1 + E8M0 per 32); NVFP4 is E2M1
//  values with an E4M3 scale per 16 and an fp32 global scale.
//
// Readings where the pages are silent (named A1..A13 in the design notes):
//  A1 score = fp32 rounding of the sigmoid evaluated in double.
//  A2 the per-expert bias enters the selection key only; weights use the raw score.
//  A3 MXFP8 scale exponent = smallest e in [-127,127] with amax <= 448*2^e.
//  A4 NVFP4 activation global scales are static per layer (inputs here).
//  A5 SwiGLU is unclamped unless the layer gives a limit L > 0: then g -> min(g, L) and
//     u -> clamp(u, -L, L) before silu(g) u.
//  A6 one bf16 rounding of the residual, RMSNorm reads it.
//  A8 W13 rows: gate rows 0..I-1, then up rows I..2I-1.  A9 shared output unscaled.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdlib>
#include <vector>
#include <algorithm>

namespace {

enum { FMT_BF16 = 0, FMT_MXFP8 = 1, FMT_NVFP4 = 2, FMT_MXFP4 = 3 };

// ---------------------------------------------------------------- number formats
// Round a non-negative double to a binary format with `mbits` explicit mantissa
// bits and minimum normal exponent `emin` (subnormals below it), ties to even.
double round_binary(double a, int mbits, int emin) {
    if (a == 0.0) return 0.0;
    int ex;
    std::frexp(a, &ex);           // a = f * 2^ex, f in [0.5, 1)
    int E = ex - 1;               // a in [2^E, 2^(E+1))
    if (E < emin) E = emin;       // subnormal range keeps the quantum of emin
    double q = std::ldexp(1.0, E - mbits);
    return std::nearbyint(a / q) * q;   // default rounding mode: nearest, ties even
}

double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// One rounding from double to bf16 (ties to even), overflow to infinity.
uint16_t double_to_bf16(double d) {
    if (std::isnan(d)) return 0x7FC0;
    double a = std::fabs(d);
    double r = round_binary(a, 7, -126);
    float f = (float)r;                       // exact: r has <= 8 significant bits
    if (r > 3.3895313892515355e38) f = INFINITY;
    if (d < 0) f = -f;
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

// E4M3 (OCP FP8): sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN.
double e4m3_decode(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = std::ldexp((double)m, -9);
    else v = std::ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

// Round-to-nearest-even, saturating to +-448; NaN maps to 0x7F.
uint8_t e4m3_encode(float x) {
    if (std::isnan(x)) return 0x7F;
    uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    double a = std::fabs((double)x);
    double r = round_binary(a, 3, -6);
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    int ex;
    std::frexp(r, &ex);
    int E = ex - 1;
    uint8_t code;
    if (E < -6) {                                 // subnormal: m * 2^-9
        code = (uint8_t)(int)(r / std::ldexp(1.0, -9));
    } else {
        int m = (int)((r / std::ldexp(1.0, E) - 1.0) * 8.0);
        code = (uint8_t)(((E + 7) << 3) | m);
    }
    return sign | code;
}

// E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; values 0,.5,1,1.5,2,3,4,6.
double e2m1_decode(uint8_t nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double v = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

uint8_t e2m1_encode(float x) {
    uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
    double a = std::fabs((double)x);
    if (std::isnan(x)) a = 6.0;                   // not produced by the generators
    double r = round_binary(a, 1, 0);
    if (r > 6.0) r = 6.0;
    if (r == 0.0) return sign;
    int ex;
    std::frexp(r, &ex);
    int E = ex - 1;
    uint8_t code;
    if (E < 0) code = 1;                          // 0.5, the only subnormal
    else code = (uint8_t)(((E + 1) << 1) | (int)((r / std::ldexp(1.0, E) - 1.0) * 2.0));
    return sign | code;
}

// E8M0: 2^(b-127); 255 is NaN.
double e8m0_decode(uint8_t b) {
    if (b == 255) return NAN;
    return std::ldexp(1.0, (int)b - 127);
}

// ---------------------------------------------------------------- block quantisation
// MXFP8, one block of 32 fp32 values (reading A3): e is the smallest integer in
// [-127, 127] with amax <= 448 * 2^e (e = -127 when amax = 0); element = E4M3(v * 2^-e).
void quant_mxfp8_block(const float* v, uint8_t* q, uint8_t* s) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
    int e = -127;
    if (amax > 0.0f) {
        while (e < 127 && (double)amax > std::ldexp(448.0, e)) ++e;
    }
    *s = (uint8_t)(e + 127);
    float inv = std::ldexp(1.0f, -e);             // exact power of two in fp32
    for (int i = 0; i < 32; ++i) q[i] = e4m3_encode(v[i] * inv);
}

// NVFP4, one block of 16 fp32 values with fp32 global scale gs (reading A4):
// scale = E4M3(amax / (6*gs)); element = E2M1(v / (dec(scale)*gs)); all ops fp32.
void quant_nvfp4_block(const float* v, float gs, uint8_t* q /*8 bytes*/, uint8_t* s) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[i]));
    float six_gs = 6.0f * gs;
    float sf = amax / six_gs;
    uint8_t sc = e4m3_encode(sf);
    *s = sc;
    float dsc = (float)e4m3_decode(sc);           // exact in fp32
    float denom = dsc * gs;
    for (int i = 0; i < 8; ++i) {
        uint8_t lo = 0, hi = 0;
        if (dsc != 0.0f) {
            lo = e2m1_encode(v[2 * i] / denom);
            hi = e2m1_encode(v[2 * i + 1] / denom);
        }
        q[i] = (uint8_t)(lo | (hi << 4));         // low nibble = even element
    }
}

// MXFP4 (OCP MX: E2M1 elements, one E8M0 scale per 32), one block of 32 fp32 values,
// the rule of A3 with E2M1's largest value: e is the smallest integer in [-127, 127] with
// amax <= 6 * 2^e (e = -127 when amax = 0); element = E2M1(v * 2^-e); low nibble = even
// element.
void quant_mxfp4_block(const float* v, uint8_t* q /*16 bytes*/, uint8_t* s) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
    int e = -127;
    if (amax > 0.0f) {
        while (e < 127 && (double)amax > std::ldexp(6.0, e)) ++e;
    }
    *s = (uint8_t)(e + 127);
    float inv = std::ldexp(1.0f, -e);
    for (int i = 0; i < 16; ++i)
        q[i] = (uint8_t)(e2m1_encode(v[2 * i] * inv) | (e2m1_encode(v[2 * i + 1] * inv) << 4));
}

// Bytes of one K-row of codes for a format.
int64_t row_bytes(int fmt, int64_t K) {
    if (fmt == FMT_BF16) return 2 * K;
    if (fmt == FMT_MXFP8) return K;
    return K / 2;
}
int64_t row_scales(int fmt, int64_t K) {
    if (fmt == FMT_MXFP8 || fmt == FMT_MXFP4) return K / 32;
    if (fmt == FMT_NVFP4) return K / 16;
    return 0;
}

// Quantise a row of K fp32 values into `fmt` (BF16 rounds each value to bf16).
void quant_row(int fmt, const float* v, int64_t K, float gs, uint8_t* q, uint8_t* s) {
    if (fmt == FMT_MXFP8) {
        for (int64_t b = 0; b < K / 32; ++b) quant_mxfp8_block(v + 32 * b, q + 32 * b, s + b);
    } else if (fmt == FMT_NVFP4) {
        for (int64_t b = 0; b < K / 16; ++b) quant_nvfp4_block(v + 16 * b, gs, q + 8 * b, s + b);
    } else if (fmt == FMT_MXFP4) {
        for (int64_t b = 0; b < K / 32; ++b) quant_mxfp4_block(v + 32 * b, q + 16 * b, s + b);
    } else {
        uint16_t* o = (uint16_t*)q;
        for (int64_t i = 0; i < K; ++i) o[i] = double_to_bf16((double)v[i]);
    }
}

// Exact dequantisation of one row into doubles; gs multiplies NVFP4 values.
void dequant_row(int fmt, const uint8_t* q, const uint8_t* s, double gs, int64_t K, double* out) {
    if (fmt == FMT_MXFP8) {
        for (int64_t i = 0; i < K; ++i) out[i] = e4m3_decode(q[i]) * e8m0_decode(s[i / 32]);
    } else if (fmt == FMT_NVFP4) {
        for (int64_t i = 0; i < K; ++i) {
            uint8_t byte = q[i / 2];
            uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);
            out[i] = e2m1_decode(nib) * e4m3_decode(s[i / 16]) * gs;
        }
    } else if (fmt == FMT_MXFP4) {
        for (int64_t i = 0; i < K; ++i) {
            uint8_t byte = q[i / 2];
            uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);
            out[i] = e2m1_decode(nib) * e8m0_decode(s[i / 32]);
        }
    } else {
        const uint16_t* b = (const uint16_t*)q;
        for (int64_t i = 0; i < K; ++i) out[i] = bf16_to_double(b[i]);
    }
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

typedef struct {
    int32_t H, E, k, I, I_sh;
    int32_t w_fmt, sh_fmt;
    int32_t has_shared, has_bias, renormalize, emit_next;
    double rsf, eps;
    float gs_a1, gs_a2;         // routed NVFP4 static activation scales (FC1 in, FC2 in)
    float gs_a1_sh, gs_a2_sh;   // shared-expert NVFP4 static activation scales
    double swiglu_limit;        // > 0: clamped SwiGLU (routed and shared experts); <= 0: plain
} or_layer;

// One projection of one expert in canonical layout.
typedef struct {
    const uint8_t* vals;    // [rows][row_bytes(fmt, K)]
    const uint8_t* scales;  // [rows][row_scales(fmt, K)] or NULL for BF16
    float gs;               // NVFP4 global scale (ignored otherwise)
} or_proj;

double or_e4m3_decode(uint8_t b) { return e4m3_decode(b); }
double or_e2m1_decode(uint8_t b) { return e2m1_decode(b); }
double or_e8m0_decode(uint8_t b) { return e8m0_decode(b); }
uint8_t or_e4m3_encode(float x) { return e4m3_encode(x); }
uint8_t or_e2m1_encode(float x) { return e2m1_encode(x); }
uint16_t or_double_to_bf16(double d) { return double_to_bf16(d); }

void or_quant(int fmt, const float* v, int64_t rows, int64_t K, float gs, uint8_t* q, uint8_t* s) {
    for (int64_t r = 0; r < rows; ++r)
        quant_row(fmt, v + r * K, K, gs, q + r * row_bytes(fmt, K), s ? s + r * row_scales(fmt, K) : nullptr);
}

void or_dequant(int fmt, const uint8_t* q, const uint8_t* s, double gs, int64_t rows, int64_t K, double* out) {
    for (int64_t r = 0; r < rows; ++r)
        dequant_row(fmt, q + r * row_bytes(fmt, K), s ? s + r * row_scales(fmt, K) : nullptr, gs, K,
                    out + r * K);
}

// ------------------------------------------------ a1 + a2: router GEMV, sigmoid, top-k
// [README] gate row: one router per row, sigmoid scores, top-k, renormalise;
// [PR24] Target spec: one expert group, sigmoid scores, renormalised top-k;
// [GB10] Key Optimizations 1: the routed sum is scaled by routed_scaling_factor.
// logit = sum_h x*Wg in double, rounded once to fp32 (skipped when logits_in given).
// score = fp32(1/(1+exp(-logit))) evaluated in double (A1).
// key = score (+ bias[e] as one fp32 add, A2); top-k by key descending, ties to the
// lower expert index; w_j = score_j / sum score * rsf in double (or score*rsf if not
// renormalised). margin = key_k - key_(k+1) of the row (k-th vs next), +inf if E == k.
void or_router(const or_layer* L, int M, const uint16_t* x, const uint16_t* wg, const float* bias,
               const float* logits_in, float* logits, float* scores, int32_t* topk_idx,
               double* topk_w, double* margin) {
    const int H = L->H, E = L->E, k = L->k;
    std::vector<double> xr(H), wr(H);
    std::vector<float> key(E), sc(E);
    std::vector<int> order(E);
    for (int m = 0; m < M; ++m) {
        for (int h = 0; h < H; ++h) xr[h] = bf16_to_double(x[(int64_t)m * H + h]);
        for (int e = 0; e < E; ++e) {
            float lg;
            if (logits_in) {
                lg = logits_in[(int64_t)m * E + e];
            } else {
                for (int h = 0; h < H; ++h) wr[h] = bf16_to_double(wg[(int64_t)e * H + h]);
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += xr[h] * wr[h];
                lg = (float)acc;
            }
            sc[e] = (float)(1.0 / (1.0 + std::exp(-(double)lg)));
            if (logits) logits[(int64_t)m * E + e] = lg;
            if (scores) scores[(int64_t)m * E + e] = sc[e];
            key[e] = (L->has_bias && bias) ? sc[e] + bias[e] : sc[e];
        }
        for (int e = 0; e < E; ++e) order[e] = e;
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return key[a] > key[b]; });
        double ssum = 0.0;
        for (int j = 0; j < k; ++j) {
            topk_idx[(int64_t)m * k + j] = order[j];
            ssum += (double)sc[order[j]];
        }
        for (int j = 0; j < k; ++j) {
            double s = (double)sc[order[j]];
            topk_w[(int64_t)m * k + j] = L->renormalize ? s / ssum * L->rsf : s * L->rsf;
        }
        if (margin) margin[m] = (E > k) ? (double)key[order[k - 1]] - (double)key[order[k]] : INFINITY;
    }
}

// ------------------------------------------------ a4: route pairs to 8-row tiles
// [README] moe row: a route kernel, 8-row tiles; an expert chosen by more than 8 rows
// takes several tiles. Pairs (m, j) are sorted by expert ascending, then by (m, j);
// the shared expert is expert E with all M rows (pair ids M*k + m), appended last.
// offsets has E+2 entries, tiles holds (expert, start in perm, rows 1..8) triples.
void or_route(const or_layer* L, int M, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
              int32_t* perm, int32_t* inv_perm, int32_t* tiles, int32_t* num_tiles) {
    const int E = L->E, k = L->k;
    const int nexp = E + 1;
    for (int e = 0; e < nexp; ++e) counts[e] = 0;
    for (int p = 0; p < M * k; ++p) counts[topk_idx[p]]++;
    counts[E] = L->has_shared ? M : 0;
    offsets[0] = 0;
    for (int e = 0; e < nexp; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int pos = 0;
    for (int e = 0; e < E; ++e)
        for (int p = 0; p < M * k; ++p)
            if (topk_idx[p] == e) perm[pos++] = p;
    if (L->has_shared)
        for (int m = 0; m < M; ++m) perm[pos++] = M * k + m;
    for (int i = 0; i < pos; ++i) inv_perm[perm[i]] = i;
    int t = 0;
    for (int e = 0; e < nexp; ++e)
        for (int s = 0; s < counts[e]; s += 8) {
            tiles[3 * t + 0] = e;
            tiles[3 * t + 1] = offsets[e] + s;
            tiles[3 * t + 2] = std::min(8, counts[e] - s);
            ++t;
        }
    *num_tiles = t;
}

// ------------------------------------------------ a3: FC1 activation quantisation
// [README] shared_ll row: one-pass MXFP8 quant of the expert input; Qwen3.5 route row:
// the NVFP4 quantisation of the MoE input. x (bf16, exact in fp32) -> fmt.
void or_quant_x(int fmt, const uint16_t* x, int64_t rows, int64_t H, float gs, uint8_t* q, uint8_t* s) {
    std::vector<float> v(H);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t h = 0; h < H; ++h) v[h] = (float)bf16_to_double(x[r * H + h]);
        quant_row(fmt, v.data(), H, gs, q + r * row_bytes(fmt, H), s ? s + r * row_scales(fmt, H) : nullptr);
    }
}

// ------------------------------------------------ a5 + a6: one expert on one row
// [README] moe row: a pair of block-scaled GEMMs (gate_up then down); shared_ll row:
// SwiGLU between them; Qwen3.5 mkm row: FC1, SwiGLU, NVFP4 requantisation, FC2.
// g_i = sum_h deq(W13[i,h]) deq(xq[h]); u_i the same over row I+i (double sums);
// h_i = silu(g_i) u_i with silu(z) = z/(1+exp(-z)); with a limit L > 0 ("SGLang-NVIDIA-
// Mega" README, shared_ll row: clamped SwiGLU), g_i -> min(g_i, L) and u_i -> clamp(u_i,
// -L, L) first;
// hq = quant(fp32(h)) along I in `fmt` (BF16: one bf16 rounding);
// y_n = sum_i deq(W2[n,i]) deq(hq[i]).
// Outputs: hq (row_bytes(fmt, I)), hs (row_scales(fmt, I)), h_out (double, I) and y (double, H).
void or_expert_row(int fmt, int H, int I, const or_proj* w13, const or_proj* w2, const double* xdq,
                   float gs_a2, double limit, uint8_t* hq, uint8_t* hs, double* h_out, double* y) {
    std::vector<double> wrow(std::max(H, I)), hv(I), hdq(I);
    std::vector<float> hf(I);
    const int64_t rb13 = row_bytes(fmt, H), rs13 = row_scales(fmt, H);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        dequant_row(fmt, w13->vals + (int64_t)i * rb13, w13->scales ? w13->scales + (int64_t)i * rs13 : nullptr,
                    w13->gs, H, wrow.data());
        for (int h = 0; h < H; ++h) g += wrow[h] * xdq[h];
        dequant_row(fmt, w13->vals + (int64_t)(I + i) * rb13,
                    w13->scales ? w13->scales + (int64_t)(I + i) * rs13 : nullptr, w13->gs, H, wrow.data());
        for (int h = 0; h < H; ++h) u += wrow[h] * xdq[h];
        if (limit > 0.0) {
            g = std::min(g, limit);
            u = std::max(-limit, std::min(u, limit));
        }
        double silu = g / (1.0 + std::exp(-g));
        hv[i] = silu * u;
        hf[i] = (float)hv[i];
    }
    if (h_out)
        for (int i = 0; i < I; ++i) h_out[i] = hv[i];
    quant_row(fmt, hf.data(), I, gs_a2, hq, hs);
    dequant_row(fmt, hq, hs, gs_a2, I, hdq.data());
    const int64_t rb2 = row_bytes(fmt, I), rs2 = row_scales(fmt, I);
    for (int n = 0; n < H; ++n) {
        dequant_row(fmt, w2->vals + (int64_t)n * rb2, w2->scales ? w2->scales + (int64_t)n * rs2 : nullptr,
                    w2->gs, I, wrow.data());
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += wrow[i] * hdq[i];
        y[n] = acc;
    }
}

// ------------------------------------------------ a7: finalize + residual + RMSNorm
// [README] hop_b row: top-k finalize and shared-expert add, then RMSNorm; past 8 rows the
// next input's MXFP8 scales per 8-row tile. moe = sum_j w_j y_j (j ascending) + y_shared;
// hres = bf16(residual + moe) is the new residual; out = bf16(hres * (mean(hres^2)+eps)^-1/2
// * gamma) (A6). If outq is given, out is quantised to MXFP8 along H.
void or_finalize_row(const or_layer* L, const double* moe, const uint16_t* residual, const uint16_t* gamma,
                     uint16_t* res_out, uint16_t* out, uint8_t* outq, uint8_t* outs) {
    const int H = L->H;
    std::vector<double> hres(H);
    double ss = 0.0;
    for (int n = 0; n < H; ++n) {
        uint16_t b = double_to_bf16(bf16_to_double(residual[n]) + moe[n]);
        res_out[n] = b;
        hres[n] = bf16_to_double(b);
        ss += hres[n] * hres[n];
    }
    double inv = 1.0 / std::sqrt(ss / H + L->eps);
    std::vector<float> of(H);
    for (int n = 0; n < H; ++n) {
        out[n] = double_to_bf16(hres[n] * inv * bf16_to_double(gamma[n]));
        of[n] = (float)bf16_to_double(out[n]);
    }
    if (outq) quant_row(FMT_MXFP8, of.data(), H, 1.0f, outq, outs);
}

// ------------------------------------------------ whole step for a list of rows
// Runs a1..a7 for each requested row; each row's result depends on that row only.
// w13/w2: per-expert projections (NULL vals for an expert the caller did not supply:
// the call then returns -(expert+1) if that expert is selected). Outputs per row r of
// `rows` (index i in the list): topk_idx/topk_w [i][k], margin[i], y_pairs [i][k][H],
// y_shared [i][H], out/res_out [i][H], outq [i][H] + outs [i][H/32] (optional).
int or_step_rows(const or_layer* L, int M, const int32_t* rows, int nrows, const uint16_t* x,
                 const uint16_t* residual, const uint16_t* gamma, const uint16_t* wg, const float* bias,
                 const float* logits_in, const or_proj* w13, const or_proj* w2, const or_proj* sh13,
                 const or_proj* sh2, int32_t* topk_idx, double* topk_w, double* margin, double* y_pairs,
                 double* y_shared, uint16_t* out, uint16_t* res_out, uint8_t* outq, uint8_t* outs) {
    const int H = L->H, E = L->E, k = L->k;
    std::vector<float> lg(E), sc(E);
    std::vector<double> xdq(H), xdq_sh(H), moe(H), y(H), hbuf(std::max(L->I, L->I_sh));
    std::vector<uint8_t> xq(2 * H), xs(H / 16 + 1), hq(2 * std::max(L->I, L->I_sh) + 16),
        hs(std::max(L->I, L->I_sh) / 16 + 1);
    for (int i = 0; i < nrows; ++i) {
        const int m = rows[i];
        const uint16_t* xr = x + (int64_t)m * H;
        or_router(L, 1, xr, wg, bias, logits_in ? logits_in + (int64_t)m * E : nullptr, lg.data(), sc.data(),
                  topk_idx + (int64_t)i * k, topk_w + (int64_t)i * k, margin ? margin + i : nullptr);
        or_quant_x(L->w_fmt, xr, 1, H, L->gs_a1, xq.data(), xs.data());
        dequant_row(L->w_fmt, xq.data(), xs.data(), L->gs_a1, H, xdq.data());
        for (int n = 0; n < H; ++n) moe[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[(int64_t)i * k + j];
            if (!w13[e].vals || !w2[e].vals) return -(e + 1);
            or_expert_row(L->w_fmt, H, L->I, &w13[e], &w2[e], xdq.data(), L->gs_a2, L->swiglu_limit, hq.data(),
                          hs.data(), hbuf.data(), y.data());
            double w = topk_w[(int64_t)i * k + j];
            for (int n = 0; n < H; ++n) {
                if (y_pairs) y_pairs[((int64_t)i * k + j) * H + n] = y[n];
                moe[n] += w * y[n];
            }
        }
        if (L->has_shared) {
            or_quant_x(L->sh_fmt, xr, 1, H, L->gs_a1_sh, xq.data(), xs.data());
            dequant_row(L->sh_fmt, xq.data(), xs.data(), L->gs_a1_sh, H, xdq_sh.data());
            or_expert_row(L->sh_fmt, H, L->I_sh, sh13, sh2, xdq_sh.data(), L->gs_a2_sh, L->swiglu_limit, hq.data(),
                          hs.data(), hbuf.data(), y.data());
            for (int n = 0; n < H; ++n) {
                if (y_shared) y_shared[(int64_t)i * H + n] = y[n];
                moe[n] += y[n];
            }
        }
        or_finalize_row(L, moe.data(), residual + (int64_t)m * H, gamma, res_out + (int64_t)i * H,
                        out + (int64_t)i * H, outq ? outq + (int64_t)i * H : nullptr,
                        outs ? outs + (int64_t)i * (H / 32) : nullptr);
    }
    return 0;
}

}  // extern "C"
