/*
 * kvq_oracle.c -- plain, slow, CPU oracle for the 8-bit block-scaled paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file:
 * only the tests, __graft_entry__.smoke() and bench.py's cpu_baseline / reference arm do.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it follows (sources are the four pull-request pages on the 8-bit KV cache):
 *   - "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section
 *     "What": one fp16 scale per 32 elements along head_dim; s = max/448 for fp8_e4m3 and
 *     s = max/127 for q8_0 (int8); 1.0625 bytes per element; K/V dequantized to bf16 before the
 *     dot because the scale varies along the reduction dim.
 *   - same page, review comment "A bug on sm_89": int8 codes round half away from zero and then
 *     clamp to +-127; fp8 codes are clamped to +-448 and rounded to nearest-even in a single
 *     rounding (the one-sided double rounding through fp16 is the bug; kept here only as the
 *     negative control kvo_e4m3_double_round).
 *   - "Add fp8 KV-cache quantization (--kv-dtype)", section "How it works": the unscaled variant, where
 *     the store casts bf16 K/V straight to the pool's fp8 type (e4m3 or e5m2, scale 1.0, 1 byte per
 *     element) and the attention reads the fp8 values back exactly.
 *   - "feat(kvcache): 8-bit DSV4 window/compressed KV", sections "What this adds" (one MLA latent
 *     row per token serves as both K and V, one scale array) and "Testing" (split-K decode,
 *     masked -1 columns, saturation).
 *
 * Readings where the pages leave a step open (each is listed with its reason in the design notes):
 *   scale = fp16_RNE(fp32(amax / Q)); a block whose fp16 scale is +0 stores all-zero codes and a zero
 *   scale; an fp32 scale above 65504 saturates to 65504; codes are computed by IEEE fp32 division by
 *   the fp16-rounded scale; fp8 keeps the sign of zero; a block_table entry of -1 masks a whole
 *   page; q head h reads kv head h / (Hq / Hkv); the softmax scale is an explicit argument; a
 *   sequence with no valid token outputs zeros.
 *
 * Number formats are written out from their definitions:
 *   binary16 (IEEE 754): 1 sign, 5 exponent bits (bias 15), 10 fraction bits, subnormal quantum 2^-24.
 *   bfloat16:            1 sign, 8 exponent bits (bias 127), 7 fraction bits, subnormal quantum 2^-133.
 *   E4M3 "fn" (OCP 8-bit floating point): 1 sign, 4 exponent bits (bias 7), 3 fraction bits,
 *                        subnormals M * 2^-9, no infinities, 0x7F / 0xFF are NaN, largest finite 448.
 *   E5M2 (OCP 8-bit floating point): 1 sign, 5 exponent bits (bias 15), 2 fraction bits, subnormals
 *                        M * 2^-16, exponent 31 is infinity / NaN, largest finite 57344.
 *
 * Arithmetic: every rounding is done explicitly on exact double values.  fp32 steps that the method
 * fixes (amax / Q, x / s) are done in C float, which is IEEE binary32 with round-to-nearest on the
 * supported hosts (FLT_EVAL_METHOD == 0); build without -ffast-math and with -ffp-contract=off.
 * The decode is exact-math attention evaluated in double.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float arithmetic evaluated in binary32"
#endif

/* Kinds: the block-scaled 8-bit caches, and the unscaled fp8 casts ("Add fp8 KV-cache quantization
   (--kv-dtype)", section "How it works": the store casts bf16 K/V to the pool's fp8 type, scale 1.0). */
enum { KVO_FP8_E4M3 = 1, KVO_Q8_0 = 2, KVO_FP8_E4M3_UNSCALED = 3, KVO_FP8_E5M2_UNSCALED = 4 };

static int kind_is_unscaled(int kind)
{
    return kind == KVO_FP8_E4M3_UNSCALED || kind == KVO_FP8_E5M2_UNSCALED;
}

/* ------------------------------------------------------------------------------------------ */
/* Rounding a non-negative double that is exactly representable to the nearest integer, ties to */
/* the even integer.                                                                            */
/* ------------------------------------------------------------------------------------------ */
static double round_half_even(double v)
{
    double fl = floor(v);
    double frac = v - fl; /* exact: v and fl are close doubles */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* floor(log2(a)) for a > 0, exact (frexp returns a = f * 2^e with f in [0.5, 1)). */
static int floor_log2(double a)
{
    int e;
    frexp(a, &e);
    return e - 1;
}

/* ------------------------------------------------------------------------------------------ */
/* binary16                                                                                     */
/* ------------------------------------------------------------------------------------------ */
double kvo_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int E = (h >> 10) & 0x1F;
    int M = h & 0x3FF;
    double v;
    if (E == 0x1F)
        v = (M == 0) ? INFINITY : NAN;
    else if (E == 0)
        v = ldexp((double)M, -24);                  /* subnormal: M * 2^-24 */
    else
        v = ldexp(1.0 + (double)M / 1024.0, E - 15); /* normal */
    return sign ? -v : v;
}

/* Round a finite double to binary16, nearest-even; magnitudes that round past 65504 give inf. */
uint16_t kvo_f16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00u;
    if (a == 0.0) return sign;
    int E = floor_log2(a);
    if (E < -14) E = -14;               /* below 2^-14 the quantum stays 2^-24 (subnormals) */
    double quantum = ldexp(1.0, E - 10); /* 10 fraction bits */
    double n = round_half_even(a / quantum);
    if (n >= 2048.0) { /* rounded up into the next binade */
        E += 1;
        n = 1024.0;
    }
    if (E > 15) return (uint16_t)(sign | 0x7C00u); /* overflow: infinity */
    if (n < 1024.0) {                               /* subnormal (only possible at E == -14) */
        return (uint16_t)(sign | (uint16_t)n);
    }
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024.0));
}

/* ------------------------------------------------------------------------------------------ */
/* bfloat16                                                                                     */
/* ------------------------------------------------------------------------------------------ */
double kvo_bf16_value(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int E = (b >> 7) & 0xFF;
    int M = b & 0x7F;
    double v;
    if (E == 0xFF)
        v = (M == 0) ? INFINITY : NAN;
    else if (E == 0)
        v = ldexp((double)M, -133);
    else
        v = ldexp(1.0 + (double)M / 128.0, E - 127);
    return sign ? -v : v;
}

uint16_t kvo_bf16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7FC0u;
    if (a == 0.0) return sign;
    int E = floor_log2(a);
    if (E < -126) E = -126;
    double quantum = ldexp(1.0, E - 7); /* 7 fraction bits */
    double n = round_half_even(a / quantum);
    if (n >= 256.0) {
        E += 1;
        n = 128.0;
    }
    if (E > 127) return (uint16_t)(sign | 0x7F80u);
    if (n < 128.0) return (uint16_t)(sign | (uint16_t)n);
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)(n - 128.0));
}

/* ------------------------------------------------------------------------------------------ */
/* E4M3 (fn)                                                                                    */
/* ------------------------------------------------------------------------------------------ */
double kvo_e4m3_value(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int E = (c >> 3) & 0xF;
    int M = c & 0x7;
    double v;
    if (E == 0xF && M == 0x7)
        v = NAN;
    else if (E == 0)
        v = ldexp((double)M, -9);
    else
        v = ldexp(1.0 + (double)M / 8.0, E - 7);
    return sign ? -v : v;
}

/* Nearest-even E4M3 code of a finite value with |y| <= 448 (callers clamp first). */
uint8_t kvo_e4m3_rne(double y)
{
    uint8_t sign = signbit(y) ? 0x80u : 0u;
    double a = fabs(y);
    if (a == 0.0) return sign;
    int E = floor_log2(a);
    if (E < -6) E = -6;                /* subnormal binade keeps quantum 2^-9 */
    double quantum = ldexp(1.0, E - 3); /* 3 fraction bits */
    double n = round_half_even(a / quantum);
    if (n >= 16.0) {
        E += 1;
        n = 8.0;
    }
    if (n < 8.0) return (uint8_t)(sign | (uint8_t)n); /* subnormal codes 0..7 (E == -6 only) */
    return (uint8_t)(sign | (uint8_t)((E + 7) << 3) | (uint8_t)(n - 8.0));
}

/* Clamp to [-448, 448] first, then one nearest-even rounding (the corrected fp8 path). */
uint8_t kvo_e4m3_sat_rne(float y)
{
    double d = (double)y;
    if (d > 448.0) d = 448.0;
    if (d < -448.0) d = -448.0;
    return kvo_e4m3_rne(d);
}

/*
 * Negative control, NOT the method: the lowering the review comment describes -- fp32 to fp16 by
 * truncation (toward zero), then to E4M3 with ties to even.  A value just above an E4M3 midpoint
 * truncates onto the midpoint and then ties downward.
 */
uint8_t kvo_e4m3_double_round(float y)
{
    double d = (double)y;
    if (d > 448.0) d = 448.0;
    if (d < -448.0) d = -448.0;
    double a = fabs(d);
    double t = 0.0;
    if (a > 0.0) {
        int E = floor_log2(a);
        if (E < -14) E = -14;
        double quantum = ldexp(1.0, E - 10);
        t = floor(a / quantum) * quantum; /* binary16 truncation of a */
    }
    return kvo_e4m3_rne(signbit(d) ? -t : t);
}

/* ------------------------------------------------------------------------------------------ */
/* E5M2 (OCP 8-bit floating point): 1 sign, 5 exponent bits (bias 15), 2 fraction bits;          */
/* subnormals M * 2^-16; exponent 31 holds infinity (M = 0) and NaN; largest finite 57344.        */
/* ------------------------------------------------------------------------------------------ */
double kvo_e5m2_value(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int E = (c >> 2) & 0x1F;
    int M = c & 0x3;
    double v;
    if (E == 0x1F)
        v = (M == 0) ? INFINITY : NAN;
    else if (E == 0)
        v = ldexp((double)M, -16);
    else
        v = ldexp(1.0 + (double)M / 4.0, E - 15);
    return sign ? -v : v;
}

/* Nearest-even E5M2 code of a finite value with |y| <= 57344 (callers clamp first). */
uint8_t kvo_e5m2_rne(double y)
{
    uint8_t sign = signbit(y) ? 0x80u : 0u;
    double a = fabs(y);
    if (a == 0.0) return sign;
    int E = floor_log2(a);
    if (E < -14) E = -14;                /* subnormal binade keeps quantum 2^-16 */
    double quantum = ldexp(1.0, E - 2);  /* 2 fraction bits */
    double n = round_half_even(a / quantum);
    if (n >= 8.0) {
        E += 1;
        n = 4.0;
    }
    if (n < 4.0) return (uint8_t)(sign | (uint8_t)n); /* subnormal codes 0..3 (E == -14 only) */
    return (uint8_t)(sign | (uint8_t)((E + 15) << 2) | (uint8_t)(n - 4.0));
}

/* Clamp to the largest finite value first (a cache holds no infinity), then one nearest-even rounding. */
uint8_t kvo_e5m2_sat_rne(float y)
{
    double d = (double)y;
    if (d > 57344.0) d = 57344.0;
    if (d < -57344.0) d = -57344.0;
    return kvo_e5m2_rne(d);
}

/* ------------------------------------------------------------------------------------------ */
/* q8_0 code: round half away from zero (exact), then clamp to [-127, 127].                     */
/* ------------------------------------------------------------------------------------------ */
int8_t kvo_q8_rhaz(float y)
{
    double d = (double)y;
    double r = (d >= 0.0) ? floor(d + 0.5) : -floor(-d + 0.5); /* exact in double for fp32 d */
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

double kvo_code_value(int kind, uint8_t c)
{
    if (kind == KVO_FP8_E4M3 || kind == KVO_FP8_E4M3_UNSCALED) return kvo_e4m3_value(c);
    if (kind == KVO_FP8_E5M2_UNSCALED) return kvo_e5m2_value(c);
    return (double)(int8_t)c;
}

/* Dequantize to bf16: RNE_bf16(value(code) * fp16 scale).  The product is exact in double. */
double kvo_dequant(int kind, uint8_t c, uint16_t s16)
{
    double prod = kvo_code_value(kind, c) * kvo_f16_value(s16);
    return kvo_bf16_value(kvo_bf16_rne(prod));
}

/* ------------------------------------------------------------------------------------------ */
/* One 32-element block: amax -> fp16 scale -> codes.                                           */
/* ------------------------------------------------------------------------------------------ */
static const float kvo_qmax_fp8 = 448.0f;
static const float kvo_qmax_q8 = 127.0f;

static float bf16_bits_to_float(uint16_t b)
{
    return (float)kvo_bf16_value(b); /* exact: every bf16 value is a float */
}

uint16_t kvo_block_scale(int kind, const uint16_t* x_bits, int n)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(bf16_bits_to_float(x_bits[i]));
        if (a > amax) amax = a;
    }
    float s32 = amax / (kind == KVO_FP8_E4M3 ? kvo_qmax_fp8 : kvo_qmax_q8); /* IEEE binary32 */
    if (s32 > 65504.0f) s32 = 65504.0f; /* fp16 scale saturates at its largest finite value */
    return kvo_f16_rne((double)s32);
}

/* Code of one element x (bf16 bits) against a nonzero fp16 block scale s16: y = x / s in IEEE binary32,
 * then the fp8 or q8_0 rounding. */
uint8_t kvo_code_of(int kind, uint16_t x_bits, uint16_t s16)
{
    float sf = (float)kvo_f16_value(s16);
    float y = bf16_bits_to_float(x_bits) / sf; /* IEEE binary32 division */
    if (kind == KVO_FP8_E4M3) return kvo_e4m3_sat_rne(y);
    return (uint8_t)kvo_q8_rhaz(y);
}

void kvo_quantize_block(int kind, const uint16_t* x_bits, int n, uint8_t* codes, uint16_t* scale_out)
{
    uint16_t s16 = kvo_block_scale(kind, x_bits, n);
    *scale_out = s16;
    if (s16 == 0) { /* zero (or fully underflowed) block: zero scale, zero codes */
        memset(codes, 0, (size_t)n);
        return;
    }
    for (int i = 0; i < n; ++i) codes[i] = kvo_code_of(kind, x_bits[i], s16);
}

/* Every pairing of ns scales with nx elements: codes[i * nx + j] = code of x[j] against s[i]. */
void kvo_code_table(int kind, const uint16_t* x_bits, int64_t nx, const uint16_t* s_bits, int64_t ns,
                    uint8_t* codes, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < ns; ++i)
        for (int64_t j = 0; j < nx; ++j) codes[i * nx + j] = kvo_code_of(kind, x_bits[j], s_bits[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* Pool layout.  Codes: [page][kv][head][slot-in-page][D] bytes, scales: [page][kv][head][slot]  */
/* [D/32] fp16; kv in {K, V} for GQA pools (n_kv = 2) and a single latent row for MLA (n_kv = 1). */
/* ------------------------------------------------------------------------------------------ */
static int64_t row_index(int64_t page, int kv, int h, int off, int n_kv, int Hkv, int P)
{
    return ((page * n_kv + kv) * (int64_t)Hkv + h) * P + off;
}

/* Bytes per cached token for one layer: codes plus one fp16 per 32 elements = 17/16 per element. */
double kvo_bytes_per_token(int n_kv, int Hkv, int D)
{
    double elems = (double)n_kv * Hkv * D;
    return elems + 2.0 * elems / 32.0;
}

/* Bytes per element of a kind: 17/16 with the block scales, 1 for an unscaled fp8 cast. */
double kvo_bytes_per_element(int kind)
{
    return kind_is_unscaled(kind) ? 1.0 : 17.0 / 16.0;
}

/*
 * Store: quantize rows k[t][h][:] (and v for GQA) and scatter them to slot slot_mapping[t];
 * slot -1 skips the row and leaves the pool untouched.  Returns 0, or -1 on bad arguments.
 */
int kvo_store(uint8_t* codes, uint16_t* scales, const uint16_t* k_bits, const uint16_t* v_bits,
              const int64_t* slot_mapping, int64_t T, int Hkv, int D, int P, int mla, int kind,
              int64_t num_pages)
{
    if (D % 32 != 0 || kind < KVO_FP8_E4M3 || kind > KVO_FP8_E5M2_UNSCALED) return -1;
    if (!kind_is_unscaled(kind) && !scales) return -1;
    int n_kv = mla ? 1 : 2;
    int nb = D / 32;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t page = slot / P;
        int off = (int)(slot % P);
        if (page >= num_pages) return -1;
        for (int kv = 0; kv < n_kv; ++kv) {
            const uint16_t* src = (kv == 0) ? k_bits : v_bits;
            for (int h = 0; h < Hkv; ++h) {
                const uint16_t* row = src + (t * Hkv + h) * (int64_t)D;
                int64_t r = row_index(page, kv, h, off, n_kv, Hkv, P);
                if (kind_is_unscaled(kind)) { /* the plain cast: no scale, no block */
                    for (int d = 0; d < D; ++d) {
                        float x = bf16_bits_to_float(row[d]);
                        codes[r * D + d] = (kind == KVO_FP8_E4M3_UNSCALED) ? kvo_e4m3_sat_rne(x) : kvo_e5m2_sat_rne(x);
                    }
                    continue;
                }
                for (int j = 0; j < nb; ++j)
                    kvo_quantize_block(kind, row + 32 * j, 32, codes + r * D + 32 * j, scales + r * nb + j);
            }
        }
    }
    return 0;
}

/* Scatter unquantized bf16 rows into a pool of the same layout (2 bytes per element); used only */
/* to report the error of the 8-bit cache against unquantized attention.                        */
int kvo_scatter_bf16(uint16_t* pool16, const uint16_t* k_bits, const uint16_t* v_bits,
                     const int64_t* slot_mapping, int64_t T, int Hkv, int D, int P, int mla, int64_t num_pages)
{
    int n_kv = mla ? 1 : 2;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t page = slot / P;
        int off = (int)(slot % P);
        if (page >= num_pages) return -1;
        for (int kv = 0; kv < n_kv; ++kv) {
            const uint16_t* src = (kv == 0) ? k_bits : v_bits;
            for (int h = 0; h < Hkv; ++h) {
                int64_t r = row_index(page, kv, h, off, n_kv, Hkv, P);
                memcpy(pool16 + r * D, src + (t * Hkv + h) * (int64_t)D, (size_t)D * 2);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Decode attention, exact math in double.                                                      */
/*   for batch b and query head h (kv head g = h / (Hq / Hkv)):                                 */
/*     valid tokens t < seq_lens[b] whose page block_table[b][t / P] is not -1                  */
/*     z_t = sm_scale * sum_d q[b][h][d] * Kd_t[d]                                              */
/*     out[b][h][:] = sum_t softmax(z)_t * Vd_t[0:Dv]      (zeros when no token is valid)       */
/*   Kd, Vd are the dequantized bf16 rows; for MLA, Vd is the first Dv entries of the same row. */
/*   quantized = 0 reads a bf16 pool (from kvo_scatter_bf16) instead.                            */
/* ------------------------------------------------------------------------------------------ */
static double row_elem(int quantized, int kind, const uint8_t* codes, const uint16_t* scales,
                       const uint16_t* pool16, int64_t r, int D, int d)
{
    if (!quantized) return kvo_bf16_value(pool16[r * D + d]);
    if (kind_is_unscaled(kind)) return kvo_code_value(kind, codes[r * D + d]); /* exact in bf16 */
    int nb = D / 32;
    return kvo_dequant(kind, codes[r * D + d], scales[r * nb + d / 32]);
}

static int decode_impl(double* out, const uint16_t* q_bits, int quantized, const uint8_t* codes,
                       const uint16_t* scales, const uint16_t* pool16, const int32_t* block_table,
                       int max_pages, const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int Dv,
                       int P, int mla, int kind, double sm_scale, int nthreads)
{
    if (Hq % Hkv != 0 || Dv > D) return -1;
    int n_kv = mla ? 1 : 2;
    int G = Hq / Hkv;
    int64_t units = (int64_t)B * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; ++u) {
        int b = (int)(u / Hq), h = (int)(u % Hq);
        int g = h / G;
        int L = seq_lens[b];
        const uint16_t* qrow = q_bits + ((int64_t)b * Hq + h) * D;
        double* o = out + ((int64_t)b * Hq + h) * Dv;
        double* z = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double zmax = -INFINITY;
        for (int t = 0; t < L; ++t) {
            int32_t page = block_table[(int64_t)b * max_pages + t / P];
            if (page < 0) {
                z[t] = -INFINITY;
                continue;
            }
            int64_t r = row_index(page, 0, g, t % P, n_kv, Hkv, P);
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += kvo_bf16_value(qrow[d]) * row_elem(quantized, kind, codes, scales, pool16, r, D, d);
            z[t] = sm_scale * dot;
            if (z[t] > zmax) zmax = z[t];
        }
        for (int d = 0; d < Dv; ++d) o[d] = 0.0;
        if (zmax == -INFINITY) { /* no valid token */
            free(z);
            continue;
        }
        double denom = 0.0;
        for (int t = 0; t < L; ++t) {
            if (z[t] == -INFINITY) continue;
            double p = exp(z[t] - zmax);
            denom += p;
            int32_t page = block_table[(int64_t)b * max_pages + t / P];
            int64_t r = row_index(page, mla ? 0 : 1, g, t % P, n_kv, Hkv, P);
            for (int d = 0; d < Dv; ++d) o[d] += p * row_elem(quantized, kind, codes, scales, pool16, r, D, d);
        }
        for (int d = 0; d < Dv; ++d) o[d] /= denom;
        free(z);
    }
    return 0;
}

int kvo_decode(double* out, const uint16_t* q_bits, const uint8_t* codes, const uint16_t* scales,
               const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B, int Hq,
               int Hkv, int D, int Dv, int P, int mla, int kind, double sm_scale, int nthreads)
{
    return decode_impl(out, q_bits, 1, codes, scales, NULL, block_table, max_pages, seq_lens, B, Hq,
                       Hkv, D, Dv, P, mla, kind, sm_scale, nthreads);
}

int kvo_decode_bf16(double* out, const uint16_t* q_bits, const uint16_t* pool16, const int32_t* block_table,
                    int max_pages, const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int Dv, int P,
                    int mla, double sm_scale, int nthreads)
{
    return decode_impl(out, q_bits, 0, NULL, NULL, pool16, block_table, max_pages, seq_lens, B, Hq, Hkv,
                       D, Dv, P, mla, 0, sm_scale, nthreads);
}

/* ------------------------------------------------------------------------------------------ */
/* Sparse (top-K) decode ("Experimental FP8 KV Cache", the SPARSE_MLA_DECODE profile line: each  */
/* query reads K selected tokens of the latent pool; "feat(kvcache): 8-bit DSV4 window/compressed */
/* KV", section "Testing": masked -1 columns).  For sequence b the index list holds topk token   */
/* positions; a column is valid when its position p satisfies 0 <= p < seq_lens[b] and the page  */
/* block_table[b][p / P] is not -1.  Every valid column is one term (a position listed twice     */
/* counts twice):                                                                               */
/*     z_i = sm_scale * sum_d q[b][h][d] * Kd(p_i)[d],   out[b][h] = sum_i softmax(z)_i Vd(p_i)   */
/* with the dequantized rows of kv head h / (Hq / Hkv); zeros when no column is valid.           */
/* ------------------------------------------------------------------------------------------ */
int kvo_decode_sparse(double* out, const uint16_t* q_bits, const uint8_t* codes, const uint16_t* scales,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens, const int32_t* indices,
                      int topk, int B, int Hq, int Hkv, int D, int Dv, int P, int mla, int kind, double sm_scale,
                      int nthreads)
{
    if (Hq % Hkv != 0 || Dv > D || topk < 0) return -1;
    int n_kv = mla ? 1 : 2;
    int G = Hq / Hkv;
    int64_t units = (int64_t)B * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; ++u) {
        int b = (int)(u / Hq), h = (int)(u % Hq);
        int g = h / G;
        const int32_t* idx = indices + (int64_t)b * topk;
        const uint16_t* qrow = q_bits + ((int64_t)b * Hq + h) * D;
        double* o = out + ((int64_t)b * Hq + h) * Dv;
        double* z = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
        int64_t* krow = (int64_t*)malloc(sizeof(int64_t) * (size_t)(topk > 0 ? topk : 1));
        double zmax = -INFINITY;
        for (int i = 0; i < topk; ++i) {
            int32_t p = idx[i];
            z[i] = -INFINITY;
            krow[i] = -1;
            if (p < 0 || p >= seq_lens[b]) continue;
            int32_t page = block_table[(int64_t)b * max_pages + p / P];
            if (page < 0) continue;
            krow[i] = row_index(page, 0, g, p % P, n_kv, Hkv, P);
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += kvo_bf16_value(qrow[d]) * row_elem(1, kind, codes, scales, NULL, krow[i], D, d);
            z[i] = sm_scale * dot;
            if (z[i] > zmax) zmax = z[i];
        }
        for (int d = 0; d < Dv; ++d) o[d] = 0.0;
        if (zmax != -INFINITY) {
            double denom = 0.0;
            for (int i = 0; i < topk; ++i) {
                if (krow[i] < 0) continue;
                double w = exp(z[i] - zmax);
                denom += w;
                int32_t p = idx[i];
                int32_t page = block_table[(int64_t)b * max_pages + p / P];
                int64_t r = row_index(page, mla ? 0 : 1, g, p % P, n_kv, Hkv, P);
                for (int d = 0; d < Dv; ++d) o[d] += w * row_elem(1, kind, codes, scales, NULL, r, D, d);
            }
            for (int d = 0; d < Dv; ++d) o[d] /= denom;
        }
        free(z);
        free(krow);
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Extend (prefill) attention over the quantized pool ("feat(kvcache): 8-bit KV cache (q8_0 /    */
/* fp8_e4m3) behind --kv-cache-dtype", section "What": the dequant sits inside every attention   */
/* kernel, prefill included; "feat(kvcache): 8-bit DSV4 window/compressed KV", section           */
/* "Testing": quantized attention on the prefill kernel).  Sequence b holds seq_lens[b] tokens,  */
/* the last n_b = q_start[b + 1] - q_start[b] of them new and already stored.  New token i sits  */
/* at position pos = seq_lens[b] - n_b + i; its query row q[q_start[b] + i][h] attends causally  */
/* to every position t <= pos whose page is not masked:                                         */
/*     z_t = sm_scale * sum_d q[row][h][d] * Kd(t)[d],   out[row][h] = sum_t softmax(z)_t Vd(t)  */
/* with the dequantized rows of kv head h / (Hq / Hkv); zeros when no position is valid.         */
/* ------------------------------------------------------------------------------------------ */
int kvo_extend(double* out, const uint16_t* q_bits, const uint8_t* codes, const uint16_t* scales,
               const int32_t* block_table, int max_pages, const int32_t* seq_lens, const int32_t* q_start,
               int B, int Hq, int Hkv, int D, int Dv, int P, int mla, int kind, double sm_scale, int nthreads)
{
    if (Hq % Hkv != 0 || Dv > D || B < 0) return -1;
    if (B > 0 && q_start[0] != 0) return -1;
    for (int b = 0; b < B; ++b) {
        int n = q_start[b + 1] - q_start[b];
        if (n < 0 || n > seq_lens[b]) return -1;
    }
    int n_kv = mla ? 1 : 2;
    int G = Hq / Hkv;
    int64_t total = B > 0 ? q_start[B] : 0;
    int64_t units = total * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; ++u) {
        int64_t row = u / Hq;
        int h = (int)(u % Hq);
        int g = h / G;
        int b = 0;
        while (q_start[b + 1] <= row) ++b;       /* the sequence this query row belongs to */
        int n = q_start[b + 1] - q_start[b];
        int pos = seq_lens[b] - n + (int)(row - q_start[b]);
        const uint16_t* qrow = q_bits + (row * Hq + h) * D;
        double* o = out + (row * Hq + h) * Dv;
        double* z = (double*)malloc(sizeof(double) * (size_t)(pos + 1));
        double zmax = -INFINITY;
        for (int t = 0; t <= pos; ++t) {
            int32_t page = block_table[(int64_t)b * max_pages + t / P];
            z[t] = -INFINITY;
            if (page < 0) continue;
            int64_t r = row_index(page, 0, g, t % P, n_kv, Hkv, P);
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += kvo_bf16_value(qrow[d]) * row_elem(1, kind, codes, scales, NULL, r, D, d);
            z[t] = sm_scale * dot;
            if (z[t] > zmax) zmax = z[t];
        }
        for (int d = 0; d < Dv; ++d) o[d] = 0.0;
        if (zmax != -INFINITY) {
            double denom = 0.0;
            for (int t = 0; t <= pos; ++t) {
                if (z[t] == -INFINITY) continue;
                double w = exp(z[t] - zmax);
                denom += w;
                int32_t page = block_table[(int64_t)b * max_pages + t / P];
                int64_t r = row_index(page, mla ? 0 : 1, g, t % P, n_kv, Hkv, P);
                for (int d = 0; d < Dv; ++d) o[d] += w * row_elem(1, kind, codes, scales, NULL, r, D, d);
            }
            for (int d = 0; d < Dv; ++d) o[d] /= denom;
        }
        free(z);
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* The store fused with its producer ("feat(kvcache): 8-bit DSV4 window/compressed KV", section  */
/* "Why the precision cost is small": the model rounds the latent part of each MLA row (all but  */
/* the last rope_dim elements) onto the E4M3 grid with one scale per 64 elements immediately     */
/* before every store; the rope tail stays bf16).  The pages do not print that rounding's scale  */
/* format; the reading here is an fp32 scale s = amax / 448 (IEEE division), the code            */
/* E4M3_sat_RNE(x / s) (IEEE division) and the value code * s in fp32, written back as bf16      */
/* (RNE); an all-zero block stays zero.  The fused store is that rounding followed by kvo_store. */
/* ------------------------------------------------------------------------------------------ */
void kvo_act_quant64(const uint16_t* x_bits, int64_t n, uint16_t* out_bits)
{
    for (int64_t b0 = 0; b0 < n; b0 += 64) {
        int64_t len = (n - b0 < 64) ? n - b0 : 64;
        float amax = 0.0f;
        for (int64_t i = 0; i < len; ++i) {
            float a = fabsf(bf16_bits_to_float(x_bits[b0 + i]));
            if (a > amax) amax = a;
        }
        if (amax == 0.0f) {
            for (int64_t i = 0; i < len; ++i) out_bits[b0 + i] = x_bits[b0 + i]; /* zeros keep their sign */
            continue;
        }
        float s = amax / kvo_qmax_fp8; /* IEEE binary32 */
        for (int64_t i = 0; i < len; ++i) {
            float y = bf16_bits_to_float(x_bits[b0 + i]) / s;
            float v = (float)kvo_e4m3_value(kvo_e4m3_sat_rne(y)) * s; /* exact code value, fp32 product */
            out_bits[b0 + i] = kvo_bf16_rne((double)v);
        }
    }
}

/* The fused MLA store: each row's first D - rope_dim elements through kvo_act_quant64, the rope tail */
/* as is, then the block-scaled store.  Returns kvo_store's status, or -1 on bad arguments.           */
int kvo_store_act_quant(uint8_t* codes, uint16_t* scales, const uint16_t* k_bits, const int64_t* slot_mapping,
                        int64_t T, int D, int rope_dim, int P, int kind, int64_t num_pages)
{
    if (rope_dim < 0 || rope_dim > D || (D - rope_dim) % 64 != 0) return -1;
    uint16_t* rows = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T > 0 ? T * D : 1));
    if (!rows) return -1;
    for (int64_t t = 0; t < T; ++t) {
        kvo_act_quant64(k_bits + t * D, D - rope_dim, rows + t * D);
        memcpy(rows + t * D + (D - rope_dim), k_bits + t * D + (D - rope_dim), sizeof(uint16_t) * (size_t)rope_dim);
    }
    int rc = kvo_store(codes, scales, rows, NULL, slot_mapping, T, 1, D, P, 1, kind, num_pages);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Batch helpers for the pins (elementwise maps over arrays).                                   */
/* ------------------------------------------------------------------------------------------ */
void kvo_f16_rne_f32_batch(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_f16_rne((double)x[i]);
}
void kvo_bf16_rne_f64_batch(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_bf16_rne(x[i]);
}
void kvo_e4m3_sat_rne_batch(const float* y, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_e4m3_sat_rne(y[i]);
}
void kvo_e4m3_double_round_batch(const float* y, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_e4m3_double_round(y[i]);
}
void kvo_q8_rhaz_batch(const float* y, int8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_q8_rhaz(y[i]);
}
void kvo_e5m2_sat_rne_batch(const float* y, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_e5m2_sat_rne(y[i]);
}

void kvo_dequant_batch(int kind, const uint8_t* c, const uint16_t* s16, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_dequant(kind, c[i], s16[i]);
}
int kvo_has_openmp(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 0;
#endif
}
