/*
 * kvq_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously-correct CPU restatement of one decode step over a
 * block-paged, quantized KV cache.  Only the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this file; the CUDA library
 * never links, includes or calls it, and it shares no code with it.
 *
 * Sources (the web pages this method is described on):
 *   [KVC]  "KV Cache优化实战：大模型推理显存占用与加速方案详解",
 *          0539edu.com/news/5800990
 *   [P402] xpshop.cn/articles/article-402.html (INT8 KV + paged cache case study)
 *   [P312] xpshop.cn/articles/article-312.html (PagedAttention + FP8/INT8 KV case study)
 *
 * What is computed, and where it is stated:
 *   - Incremental decode: the new token's K/V are appended to the cache, then the
 *     new Q attends over every cached K/V ([KVC] §1.1).
 *   - KV bytes = 2 x batch x seq x layers x kv_heads x head_dim x bytes ([KVC] §1.2).
 *   - GQA: Q heads are split into groups, each group shares one K/V head
 *     ([KVC] §2.1).  Reading taken: contiguous groups, kv_head = q_head / G.
 *   - Paged storage: fixed-size physical blocks, a block table maps a request's
 *     logical blocks to physical ones ([KVC] §2.2, [P312] §三).
 *   - INT8 symmetric absmax quantization with per-token, per-channel or
 *     per-group scales; FP8 as an alternative ([KVC] §2.3, §3.3).
 *     Readings taken where the pages are silent:
 *       scale s = absmax / 127 in fp32 (IEEE round-to-nearest), code =
 *       clamp(round-half-even(x / s), -127, 127) with an fp32 division; a group
 *       whose absmax is 0 gets s = 0 and all-zero codes.  FP8 uses the e4m3
 *       format with s = absmax / 448 and round-to-nearest-even, saturating to
 *       the largest finite value.  Per-token = one scale per (token, K|V) over
 *       all kv heads; per-group = g contiguous head_dim elements of one
 *       (token, head, K|V) vector; per-channel = a static [2][Hkv][D] scale set
 *       from calibration tokens (absmax / 127 per channel).
 *   - FP8 e5m2 without a scale, the `fp8_e5m2` KV-cache dtype of [P312] §三:
 *     code = e5m2 round-to-nearest-even of x itself, saturating to the largest
 *     finite value (57344); dequantized value = the code's value.
 *   - INT4, listed beside INT8 and FP8 as the more aggressive option ([KVC]
 *     §2.3; measured in [KVC] §3.3 and [P402] §三): read as the same absmax symmetric rule
 *     on 4 bits, per group: s = absmax / 7 (fp32), code =
 *     clamp(round-half-even(x / s), -7, 7), zero group -> s = 0, codes 0.
 *   - Attention: softmax(q.k^T * sm_scale) v over the dequantized cache, in
 *     float64 here ("the same dequantised cache": k^ = code * scale in fp64).
 *
 * Parity pins: see the tests that exercise this file (closed-form quantizer
 * cases, the e4m3 table of the OCP FP8 definition, dense brute-force attention,
 * permutation/prefix/GQA invariants, the size formula).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Cache formats.  Values match the library's public enum so that the tests can
 * pass one number to both sides; the oracle defines its own copy. */
enum {
    OR_FP16 = 0,
    OR_INT8_PER_TOKEN = 1,
    OR_INT8_PER_CHANNEL = 2,
    OR_INT8_PER_GROUP = 3,
    OR_FP8_E4M3_PER_TOKEN = 4,
    OR_INT4_PER_GROUP = 5,
    OR_FP8_E5M2 = 6,
};

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------- */
/* KV-cache size formula ([KVC] §1.2): 2 (K and V) x batch x seq x layers x     */
/* kv_heads x head_dim x precision bytes.                                      */
/* ------------------------------------------------------------------------- */
uint64_t oracle_kv_cache_bytes(uint64_t batch, uint64_t seq_len, uint64_t layers,
                               uint64_t kv_heads, uint64_t head_dim,
                               uint64_t precision_bytes) {
    return 2ull * batch * seq_len * layers * kv_heads * head_dim * precision_bytes;
}

/* ------------------------------------------------------------------------- */
/* FP8 e4m3 (OCP 8-bit floating point, E4M3 variant): 1 sign bit, 4 exponent   */
/* bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals      */
/* 2^-6 * m/8; S.1111.111 is NaN; there is no infinity; largest finite 448.    */
/* ------------------------------------------------------------------------- */
double oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even onto the e4m3 grid, saturating to +-448 (the
 * "satfinite" behaviour: no value ever becomes NaN).  Written as a brute-force
 * search over the 127 non-negative finite codes: the nearest one wins, and an
 * exact tie goes to the code with an even last mantissa bit.  Codes increase
 * with magnitude, so "even code" == "even mantissa". */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    int sign = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    uint8_t best = 0;
    if (a >= 448.0) {
        best = 0x7E;
    } else {
        double best_d = INFINITY;
        for (int c = 0; c <= 0x7E; ++c) {
            double d = fabs(oracle_e4m3_decode((uint8_t)c) - a);
            if (d < best_d || (d == best_d && (c & 1) == 0)) {
                best_d = d;
                best = (uint8_t)c;
            }
        }
    }
    return (uint8_t)(best | (sign << 7));
}

/* ------------------------------------------------------------------------- */
/* Quantizers ([KVC] §2.3: absmax symmetric INT8; per-token / per-channel /   */
/* per-group scales; FP8).  All arithmetic in fp32 as stated in the header.   */
/* ------------------------------------------------------------------------- */

/* OCP FP8 e5m2: sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent
 * 31 is infinity (mantissa 0) or NaN.  Value of a code, from the definition. */
double oracle_e5m2_decode(uint8_t code) {
    int sign = code >> 7, e = (code >> 2) & 0x1F, m = code & 0x3;
    double v;
    if (e == 31) v = m == 0 ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)m / 4.0, -14);
    else v = ldexp(1.0 + (double)m / 4.0, e - 15);
    return sign ? -v : v;
}

/* Nearest finite e5m2 code by brute force over the non-negative finite codes
 * (0x00..0x7B), ties to the even mantissa; |x| beyond the largest finite value
 * saturates to it; the sign is kept (so -0 -> 0x80). */
uint8_t oracle_e5m2_encode(float x) {
    if (isnan(x)) return 0x7F;
    int sign = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    uint8_t best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7B; ++c) {
        double d = fabs(oracle_e5m2_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = (uint8_t)c;
        }
    }
    return (uint8_t)(best | (sign << 7));
}

/* IEEE binary16 -> binary32, exact: the widening every input goes through
 * before the fp32 quantizer.  1 sign bit, 5 exponent bits (bias 15), 10
 * mantissa bits; exponent 0 is zero or subnormal (m * 2^-24), exponent 31 is
 * infinity (m = 0) or NaN (payload kept in the top mantissa bits), otherwise
 * (1024 + m) * 2^(e - 25). */
void oracle_half_to_float(const uint16_t* h, float* f, int64_t n) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t sign = (uint32_t)(h[i] >> 15);
        const int e = (h[i] >> 10) & 0x1F;
        const uint32_t m = h[i] & 0x3FFu;
        float x;
        if (e == 31) {
            const uint32_t bits = (sign << 31) | 0x7F800000u | (m << 13);
            memcpy(&x, &bits, sizeof x);
        } else {
            x = e == 0 ? ldexpf((float)m, -24) : ldexpf((float)(1024u + m), e - 25);
            if (sign) x = -x;
        }
        f[i] = x;
    }
}

/* One dynamic-scale INT8 group of n values. */
void oracle_quant_int8_group(const float* x, int n, int8_t* codes, float* scale) {
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float m = fabsf(x[i]);
        if (m > a) a = m;
    }
    if (a == 0.0f) {
        *scale = 0.0f;
        for (int i = 0; i < n; ++i) codes[i] = 0;
        return;
    }
    float s = a / 127.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) {
        float q = nearbyintf(x[i] / s);
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        codes[i] = (int8_t)q;
    }
}

/* One dynamic-scale INT4 group of n values: s = absmax / 7, codes in [-7, 7]
 * (kept one per byte here). */
void oracle_quant_int4_group(const float* x, int n, int8_t* codes, float* scale) {
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float m = fabsf(x[i]);
        if (m > a) a = m;
    }
    if (a == 0.0f) {
        *scale = 0.0f;
        for (int i = 0; i < n; ++i) codes[i] = 0;
        return;
    }
    float s = a / 7.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) {
        float q = nearbyintf(x[i] / s);
        if (q > 7.0f) q = 7.0f;
        if (q < -7.0f) q = -7.0f;
        codes[i] = (int8_t)q;
    }
}

/* INT8 with a fixed (calibrated) scale per element: values beyond the
 * calibrated range saturate at +-127; a zero scale gives a zero code. */
void oracle_quant_int8_static(const float* x, const float* s, int n, int8_t* codes) {
    for (int i = 0; i < n; ++i) {
        if (s[i] == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float q = nearbyintf(x[i] / s[i]);
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        codes[i] = (int8_t)q;
    }
}

/* One dynamic-scale FP8 e4m3 group of n values: s = absmax / 448. */
void oracle_quant_e4m3_group(const float* x, int n, uint8_t* codes, float* scale) {
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float m = fabsf(x[i]);
        if (m > a) a = m;
    }
    if (a == 0.0f) {
        *scale = 0.0f;
        for (int i = 0; i < n; ++i) codes[i] = 0;
        return;
    }
    float s = a / 448.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(x[i] / s);
}

/* Per-channel calibration: s[c] = absmax over the T calibration tokens / 127.
 * x is [T][C]; s is [C]. */
void oracle_calibrate_channels(const float* x, int64_t T, int C, float* s) {
    for (int c = 0; c < C; ++c) {
        float a = 0.0f;
        for (int64_t t = 0; t < T; ++t) {
            float m = fabsf(x[t * C + c]);
            if (m > a) a = m;
        }
        s[c] = a / 127.0f;
    }
}

/* ------------------------------------------------------------------------- */
/* The oracle's cache store.  A plain slot-indexed array, deliberately unlike */
/* any tiled device layout:                                                  */
/*   codes : [num_slots][2 (K,V)][Hkv][D], one byte per element (int8, int4   */
/*           or e4m3), or one float per element for FP16 (the fp16 value,      */
/*           widened)                                                         */
/*   scales: per-group   [num_slots][2][Hkv][D/g]  (INT8 and INT4)             */
/*           per-token   [num_slots][2]                                        */
/*           per-channel / FP16: unused                                        */
/* slot = physical_block * block_size + offset_in_block ([KVC] §2.2).          */
/* ------------------------------------------------------------------------- */

static int scales_per_slot(int fmt, int Hkv, int D, int g) {
    switch (fmt) {
    case OR_INT8_PER_GROUP:
    case OR_INT4_PER_GROUP: return 2 * Hkv * (D / g);
    case OR_INT8_PER_TOKEN:
    case OR_FP8_E4M3_PER_TOKEN: return 2;
    default: return 0;
    }
}

/* Append T new tokens ([KVC] §1.1: each decode step appends the new token's
 * K/V to the end of the cache).  k, v: [T][Hkv][D] (fp16 widened to fp32);
 * slots: [T], a negative slot means "skip this token"; chan_scales: [2][Hkv][D]
 * for the per-channel format.  The non-negative slots must be distinct: each
 * token then writes only its own slot, and the tokens are taken in parallel.
 * (OracleCache.append keeps only the last token of a repeated slot, which is
 * what processing every token in order would leave there.) */
void oracle_append(int fmt, int64_t T, int Hkv, int D, int g,
                   const float* k, const float* v, const int64_t* slots,
                   const float* chan_scales, void* codes, float* scales) {
    const int per = Hkv * D;
    const int nsc = scales_per_slot(fmt, Hkv, D, g);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        for (int kv = 0; kv < 2; ++kv) {
            const float* x = (kv == 0 ? k : v) + t * per;
            int64_t base = (slot * 2 + kv) * (int64_t)per;
            switch (fmt) {
            case OR_FP16: {
                float* c = (float*)codes + base;
                for (int i = 0; i < per; ++i) c[i] = x[i];
                break;
            }
            case OR_INT8_PER_GROUP: {
                int8_t* c = (int8_t*)codes + base;
                int ng = D / g;
                for (int h = 0; h < Hkv; ++h)
                    for (int gi = 0; gi < ng; ++gi)
                        oracle_quant_int8_group(x + h * D + gi * g, g, c + h * D + gi * g,
                                                scales + slot * nsc + (kv * Hkv + h) * ng + gi);
                break;
            }
            case OR_INT4_PER_GROUP: {
                int8_t* c = (int8_t*)codes + base;
                int ng = D / g;
                for (int h = 0; h < Hkv; ++h)
                    for (int gi = 0; gi < ng; ++gi)
                        oracle_quant_int4_group(x + h * D + gi * g, g, c + h * D + gi * g,
                                                scales + slot * nsc + (kv * Hkv + h) * ng + gi);
                break;
            }
            case OR_INT8_PER_TOKEN: {
                int8_t* c = (int8_t*)codes + base;
                oracle_quant_int8_group(x, per, c, scales + slot * nsc + kv);
                break;
            }
            case OR_FP8_E4M3_PER_TOKEN: {
                uint8_t* c = (uint8_t*)codes + base;
                oracle_quant_e4m3_group(x, per, c, scales + slot * nsc + kv);
                break;
            }
            case OR_FP8_E5M2: {
                uint8_t* c = (uint8_t*)codes + base;
                for (int i = 0; i < per; ++i) c[i] = oracle_e5m2_encode(x[i]);
                break;
            }
            case OR_INT8_PER_CHANNEL: {
                int8_t* c = (int8_t*)codes + base;
                oracle_quant_int8_static(x, chan_scales + kv * per, per, c);
                break;
            }
            default: break;
            }
        }
    }
}

/* Dequantized value of element (slot, kv, h, d) in float64: code * scale. */
static double dequant(int fmt, int Hkv, int D, int g, const void* codes,
                      const float* scales, const float* chan_scales,
                      int64_t slot, int kv, int h, int d) {
    int64_t idx = ((slot * 2 + kv) * Hkv + h) * (int64_t)D + d;
    int nsc = scales_per_slot(fmt, Hkv, D, g);
    switch (fmt) {
    case OR_FP16: return (double)((const float*)codes)[idx];
    case OR_INT8_PER_GROUP:
    case OR_INT4_PER_GROUP: {
        int ng = D / g;
        double s = (double)scales[slot * nsc + (kv * Hkv + h) * ng + d / g];
        return (double)((const int8_t*)codes)[idx] * s;
    }
    case OR_INT8_PER_TOKEN:
        return (double)((const int8_t*)codes)[idx] * (double)scales[slot * nsc + kv];
    case OR_FP8_E4M3_PER_TOKEN:
        return oracle_e4m3_decode(((const uint8_t*)codes)[idx]) * (double)scales[slot * nsc + kv];
    case OR_FP8_E5M2:
        return oracle_e5m2_decode(((const uint8_t*)codes)[idx]);
    case OR_INT8_PER_CHANNEL:
        return (double)((const int8_t*)codes)[idx] *
               (double)chan_scales[(kv * Hkv + h) * D + d];
    default: return 0.0;
    }
}

/* Paged decode attention ([KVC] §1.1 decode step, §2.1 GQA, §2.2 block table,
 * §2.3 dequantize-then-compute).  For each sequence s and Q head hq:
 *   kv head  = hq / (Hq / Hkv)
 *   token t < L_s lives at slot table[s][t / bs] * bs + t % bs
 *   z_t      = sm_scale * sum_d q[d] * k^_t[d]
 *   out      = sum_t exp(z_t - max z) v^_t / sum_t exp(z_t - max z)
 * all in float64.  L_s == 0 gives a zero output.
 * q: [S][Hq][D] (fp16 widened), table: [S][max_blocks], lens: [S],
 * out: [S][Hq][D] float64.  Pairs (s, hq) run in parallel when built with
 * OpenMP; each pair's arithmetic is sequential and independent. */
void oracle_decode(int fmt, int S, int Hq, int Hkv, int D, int g, int bs,
                   const float* q, const int32_t* table, int max_blocks,
                   const int32_t* lens, double sm_scale,
                   const void* codes, const float* scales, const float* chan_scales,
                   double* out) {
    const int G = Hq / Hkv;
    const int64_t pairs = (int64_t)S * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t p = 0; p < pairs; ++p) {
        int s = (int)(p / Hq), hq = (int)(p % Hq);
        int h = hq / G;
        int L = lens[s];
        double* o = out + p * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (L <= 0) continue;
        const float* qv = q + p * D;
        double* z = (double*)malloc(sizeof(double) * (size_t)L);
        double zmax = -INFINITY;
        for (int t = 0; t < L; ++t) {
            int64_t slot = (int64_t)table[(int64_t)s * max_blocks + t / bs] * bs + t % bs;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)qv[d] * dequant(fmt, Hkv, D, g, codes, scales, chan_scales, slot, 0, h, d);
            z[t] = sm_scale * acc;
            if (z[t] > zmax) zmax = z[t];
        }
        double denom = 0.0;
        for (int t = 0; t < L; ++t) {
            int64_t slot = (int64_t)table[(int64_t)s * max_blocks + t / bs] * bs + t % bs;
            double w = exp(z[t] - zmax);
            denom += w;
            for (int d = 0; d < D; ++d)
                o[d] += w * dequant(fmt, Hkv, D, g, codes, scales, chan_scales, slot, 1, h, d);
        }
        for (int d = 0; d < D; ++d) o[d] /= denom;
        free(z);
    }
}
