/*
 * kvd_oracle.c -- plain, slow, fp64 CPU oracle for decode-phase KV-cache
 * attention, KV append, paged gather, paged attention and the log-sum-exp
 * combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file.  Only the test suite, the smoke check of the graft
 * entry point and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, constant or helper with the CUDA library; it has its own
 * element decoding, its own index arithmetic and its own status bits.
 *
 * Every function is the direct definition, written out loop by loop: no
 * blocking, no online softmax, no split of the sequence.  Floating point is
 * carried in double; bf16 and fp32 inputs are widened exactly.
 *
 * Sources (page title, section):
 *  [NPU-KV]   "Intel NPU running LLMs" (OpenVINO community article 882),
 *             Part 1 "解决方案：预分配 + Attention Mask" (static buffer of
 *             capacity MAX_PROMPT_LEN + MIN_RESPONSE_LEN, 0/1 mask, mask=0
 *             positions set to -inf before the softmax); Part 2 "NPUW 的核心
 *             设计" (update_kvcache_for writes only the new row at the next
 *             empty slot); Part 3 "Attention 在 NPU 上的完整实现"
 *             (decomposed SDPA: Q x K^T, x scale, + mask, softmax, x V);
 *             Part 5 "当前限制" (over capacity is an error).
 *  [FlashMLA] "FlashMLA на Huawei Ascend: ядро разреженного внимания
 *             изнутри", section "Математическая постановка" (P = Q K^T,
 *             S = softmax(P * sm_scale), out = S V; lse per row).
 *  [FlashMLA-KV] same page, "Ограничение по деквантованию" (decoding reads
 *             the KV cache in FP8, dequantises it to bf16 and feeds the
 *             matrix unit) and "Оптимизация раскладки KV-кэша при decoding"
 *             (each token's quantised values and its scale are stored side
 *             by side).  The scale granularity and encoding are not given;
 *             the reading taken here is one fp32 scale per token row of a kv
 *             head (absmax / 448), stored right after the row's E4M3 codes.
 *             The same page names FP4 beside FP8: E2M1 codes (OCP 4-bit
 *             floating point), two per byte (element 2j in the low nibble of
 *             byte j), one fp32 scale per row (absmax / 6) after them.
 *  [PyPTO]    "PyPTO 实现 AscendC GatherPaKvCache（Norm/ND 分支）", sections
 *             3.1 (tensor contract), 3.2 (gather semantics: logical_block =
 *             t // block_size, slot = t % block_size, physical_block =
 *             block_tables[q, table_offset(q) + logical_block], output row
 *             seq_lens[q] + t), 3.3 (shape and value constraints), 7 (only
 *             the cumsum form of seq_lens).
 *
 * Parity pins for every function live in tests/test_oracle_*.py (closed
 * forms, invariants, a library cross-check and brute force on tiny inputs).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element types of the storage */
#define ORC_BF16 0
#define ORC_F32 1
#define ORC_FP8ROW 2 /* K/V only: rows of D E4M3 codes + fp32 scale + 12 zero bytes */
#define ORC_FP4ROW 3 /* K/V only: rows of D/2 bytes of E2M1 codes + fp32 scale + 12 zero bytes */

/* error bits reported by the data-movement oracles (own numbering) */
#define ORC_ERR_POS 1        /* append position outside [0, capacity) */
#define ORC_ERR_BLOCK 2      /* block id outside [0, num_blocks) */
#define ORC_ERR_COLS 4       /* table_offset + needed blocks > table columns */
#define ORC_ERR_SEQLENS 8    /* cumsum not starting at 0, decreasing, or past total */
#define ORC_ERR_OFFSET 16    /* seq_offset negative or not a multiple of block_size */

/* Exact widening of one stored element to double.  bf16 is the upper half
 * of an IEEE binary32, so shifting its 16 bits up gives the same number. */
static double orc_elem(const void* base, size_t i, int dtype) {
    if (dtype == ORC_BF16) {
        uint16_t h = ((const uint16_t*)base)[i];
        uint32_t w = ((uint32_t)h) << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[i];
}

/* ------------------------------------------------------------ E4M3 codes
 * OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 holds the subnormals f * 2^-9;
 * no infinities; S.1111.111 is NaN, so the largest finite value is
 * 1.75 * 2^8 = 448. */
static double orc_e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 15, f = c & 7;
    double x;
    if (e == 15 && f == 7)
        x = NAN;
    else if (e == 0)
        x = ldexp((double)f, -9);
    else
        x = ldexp((double)(8 + f), e - 10); /* (1 + f/8) * 2^(e-7) */
    return (c & 0x80) ? -x : x;
}

/* Nearest E4M3 value of x, ties to the even code, magnitudes from 448 up
 * (and infinities) saturated to 448; NaN stays NaN. */
static uint8_t orc_e4m3_code(float x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x)) return sign | 0x7F;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
    int e = ex - 1;
    if (e < -6) e = -6; /* below 2^-6 the spacing stays that of the subnormals */
    const double step = ldexp(1.0, e - 3);
    const double val = nearbyint(a / step) * step; /* exact quotient; ties to even */
    if (val == 0.0) return sign;
    int ev;
    frexp(val, &ev);
    const int E = ev - 1 + 7;
    if (E <= 0) return sign | (uint8_t)(val * 512.0); /* f * 2^-9 */
    const int f = (int)(val / ldexp(1.0, ev - 1) * 8.0) - 8;
    return sign | (uint8_t)(E << 3) | (uint8_t)f;
}

/* ------------------------------------------------------------ E2M1 codes
 * OCP 4-bit floating point, E2M1: 1 sign bit, 2 exponent bits with bias 1,
 * 1 mantissa bit; exponent 0 is subnormal (m * 0.5).  The magnitudes are 0,
 * 0.5, 1, 1.5, 2, 3, 4, 6; there is no infinity or NaN. */
static double orc_e2m1_value(uint8_t c) {
    const double sign = (c & 0x8) ? -1.0 : 1.0;
    const int e = (c >> 1) & 0x3, m = c & 0x1;
    if (e == 0) return sign * 0.5 * m;
    return sign * ldexp(1.0 + 0.5 * m, e - 1);
}

/* Nearest E2M1 value of x, ties to the even code (mantissa bit 0),
 * magnitudes from 6 up saturating to 6; NaN gives +6 (this reading follows
 * the saturating conversion's rule for NaN inputs). */
static uint8_t orc_e2m1_code(float x) {
    if (isnan(x)) return 0x7;
    const uint8_t sign = signbit(x) ? 0x8 : 0;
    const double a = fabs((double)x);
    if (a >= 6.0) return sign | 0x7;
    /* spacing: 0.5 below 2 (subnormals and [1, 2)), then 2^(e - 1) in [2^e, 2^(e+1)) */
    double step = 0.5;
    if (a >= 2.0) {
        int ex;
        frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
        step = ldexp(1.0, ex - 2);
    }
    const double val = nearbyint(a / step) * step; /* exact quotient; ties to even */
    /* the grid's magnitudes in code order */
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    for (int i = 0; i < 8; ++i)
        if (val == grid[i]) return sign | (uint8_t)i;
    return sign | 0x7; /* val == 6 after rounding up from (5, 6) */
}

/* fp32 scale of a quantised row (bytes D..D+3, little-endian). */
static float orc_row_scale(const uint8_t* row, int D) {
    const uint32_t u = (uint32_t)row[D] | ((uint32_t)row[D + 1] << 8) |
                       ((uint32_t)row[D + 2] << 16) | ((uint32_t)row[D + 3] << 24);
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Element d of K/V row `row` (rows of D elements, or quantised rows). */
static double orc_kv(const void* base, size_t row, int d, int kvtype, int D) {
    if (kvtype == ORC_FP8ROW) {
        const uint8_t* r = (const uint8_t*)base + row * (size_t)(D + 16);
        return (double)orc_row_scale(r, D) * orc_e4m3_value(r[d]);
    }
    if (kvtype == ORC_FP4ROW) {
        const uint8_t* r = (const uint8_t*)base + row * (size_t)(D / 2 + 16);
        const uint8_t code = (uint8_t)((r[d / 2] >> (4 * (d & 1))) & 0xF);
        return (double)orc_row_scale(r, D / 2) * orc_e2m1_value(code);
    }
    return orc_elem(base, row * (size_t)D + d, kvtype);
}

/*
 * Row quantisation ([FlashMLA-KV], reading above): for each row of D values,
 * amax = max |v_d|, scale = amax / 448 and code_d = E4M3(v_d / scale), both
 * divisions in fp32 with round-to-nearest; a row of zeros gets scale 0 and
 * zero codes.  dst rows: codes, the scale's 4 bytes (little-endian), 12 zero
 * bytes.  Inputs are finite.
 */
static void orc_quantize_row(const void* src, size_t row, int dtype, int D, uint8_t* dst) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        const float a = fabsf((float)orc_elem(src, row * (size_t)D + d, dtype));
        if (a > amax) amax = a;
    }
    const float scale = amax / 448.0f;
    for (int d = 0; d < D; ++d) {
        const float v = (float)orc_elem(src, row * (size_t)D + d, dtype);
        dst[d] = scale > 0.0f ? orc_e4m3_code(v / scale) : 0;
    }
    uint32_t u;
    memcpy(&u, &scale, sizeof u);
    for (int i = 0; i < 4; ++i) dst[D + i] = (uint8_t)(u >> (8 * i));
    memset(dst + D + 4, 0, 12);
}

/*
 * FP4 row quantisation ([FlashMLA-KV], FP4 reading above): for each row of D
 * values, amax = max |v_d|, scale = amax / 6 and code_d = E2M1(v_d / scale),
 * both divisions in fp32 with round-to-nearest; a row of zeros gets scale 0
 * and zero codes.  dst rows: D/2 bytes of codes (element 2j in the low
 * nibble of byte j), the scale's 4 bytes (little-endian), 12 zero bytes.
 */
static void orc_quantize_row_fp4(const void* src, size_t row, int dtype, int D, uint8_t* dst) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        const float a = fabsf((float)orc_elem(src, row * (size_t)D + d, dtype));
        if (a > amax) amax = a;
    }
    const float scale = amax / 6.0f;
    memset(dst, 0, (size_t)D / 2);
    for (int d = 0; d < D; ++d) {
        const float v = (float)orc_elem(src, row * (size_t)D + d, dtype);
        const uint8_t c = scale > 0.0f ? orc_e2m1_code(v / scale) : 0;
        dst[d / 2] |= (uint8_t)(c << (4 * (d & 1)));
    }
    uint32_t u;
    memcpy(&u, &scale, sizeof u);
    for (int i = 0; i < 4; ++i) dst[D / 2 + i] = (uint8_t)(u >> (8 * i));
    memset(dst + D / 2 + 4, 0, 12);
}

int kvd_oracle_quantize_rows_fp4(const void* src, int dtype, long rows, int D, uint8_t* dst) {
    if (rows < 0 || D <= 0 || D % 2) return -1;
    for (long r = 0; r < rows; ++r)
        orc_quantize_row_fp4(src, (size_t)r, dtype, D, dst + (size_t)r * (D / 2 + 16));
    return 0;
}

int kvd_oracle_e2m1_codes(const float* x, long n, uint8_t* out) {
    for (long i = 0; i < n; ++i) out[i] = orc_e2m1_code(x[i]);
    return 0;
}

int kvd_oracle_e2m1_values(const uint8_t* c, long n, double* out) {
    for (long i = 0; i < n; ++i) out[i] = orc_e2m1_value(c[i]);
    return 0;
}

int kvd_oracle_quantize_rows(const void* src, int dtype, long rows, int D, uint8_t* dst) {
    if (rows < 0 || D <= 0) return -1;
    for (long r = 0; r < rows; ++r)
        orc_quantize_row(src, (size_t)r, dtype, D, dst + (size_t)r * (D + 16));
    return 0;
}

int kvd_oracle_e4m3_codes(const float* x, long n, uint8_t* out) {
    for (long i = 0; i < n; ++i) out[i] = orc_e4m3_code(x[i]);
    return 0;
}

int kvd_oracle_e4m3_values(const uint8_t* c, long n, double* out) {
    for (long i = 0; i < n; ++i) out[i] = orc_e4m3_value(c[i]);
    return 0;
}

int kvd_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Masked decode attention over a static buffer.
 *   q    [B, Hq, D]          k, v [B, Hkv, C, D]        mask [B, C] (0 = padding)
 *   out  [B, Hq, D] double   lse  [B, Hq] double (natural log), may be NULL
 * Query head h reads kv head h / (Hq / Hkv) (contiguous GQA groups).
 * Masked slots are excluded from the softmax by selection, which is the
 * same as adding -inf to their scores for finite contents and stays exact
 * when the padding holds inf or NaN.  A row with no valid slot gives out = 0
 * and lse = -inf.
 */
static int orc_attend_masked(const void* q, int dtype, const void* k, const void* v,
                             int kvtype, const uint8_t* mask, int B, int Hq, int Hkv,
                             int C, int D, double scale, double* out, double* lse,
                             int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || C < 0 || D <= 0 || Hq % Hkv) return -1;
    const int g = Hq / Hkv;
    const long units = (long)B * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        const int b = (int)(u / Hq), h = (int)(u % Hq), kvh = h / g;
        double* s = (double*)malloc(sizeof(double) * (C > 0 ? C : 1));
        double* num = (double*)malloc(sizeof(double) * D);
        if (!s || !num) {
            free(s);
            free(num);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        const size_t qbase = ((size_t)b * Hq + h) * D;
        const size_t kvrow = ((size_t)b * Hkv + kvh) * (size_t)C;
        /* pass 1: scores of the valid slots and their maximum */
        double m = -INFINITY;
        long nvalid = 0;
        for (int t = 0; t < C; ++t) {
            if (!mask[(size_t)b * C + t]) continue;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += orc_elem(q, qbase + d, dtype) * orc_kv(k, kvrow + t, d, kvtype, D);
            s[t] = scale * dot;
            if (s[t] > m) m = s[t];
            ++nvalid;
        }
        double* o = out + qbase;
        if (nvalid == 0) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (lse) lse[(size_t)b * Hq + h] = -INFINITY;
            free(s);
            free(num);
            continue;
        }
        /* pass 2: softmax weights and the weighted sum of V rows */
        double den = 0.0;
        for (int d = 0; d < D; ++d) num[d] = 0.0;
        for (int t = 0; t < C; ++t) {
            if (!mask[(size_t)b * C + t]) continue;
            const double w = exp(s[t] - m);
            den += w;
            for (int d = 0; d < D; ++d) num[d] += w * orc_kv(v, kvrow + t, d, kvtype, D);
        }
        for (int d = 0; d < D; ++d) o[d] = num[d] / den;
        if (lse) lse[(size_t)b * Hq + h] = m + log(den);
        free(s);
        free(num);
    }
    return failed ? -2 : 0;
}

int kvd_oracle_attend_masked(const void* q, const void* k, const void* v,
                             const uint8_t* mask, int dtype, int B, int Hq,
                             int Hkv, int C, int D, double scale, double* out,
                             double* lse, int nthreads) {
    return orc_attend_masked(q, dtype, k, v, dtype, mask, B, Hq, Hkv, C, D, scale, out, lse,
                             nthreads);
}

/*
 * Masked decode attention over quantised K/V rows ([FlashMLA-KV]): the same
 * definition as kvd_oracle_attend_masked with every K and V element taken as
 * scale_row * E4M3(code), exactly, in double.
 *   q [B, Hq, D] (qtype); k, v [B, Hkv, C, D + 16] bytes.
 */
int kvd_oracle_attend_masked_fp8(const void* q, int qtype, const uint8_t* k, const uint8_t* v,
                                 const uint8_t* mask, int B, int Hq, int Hkv, int C, int D,
                                 double scale, double* out, double* lse, int nthreads) {
    return orc_attend_masked(q, qtype, k, v, ORC_FP8ROW, mask, B, Hq, Hkv, C, D, scale, out, lse,
                             nthreads);
}

/*
 * The same masked attention over FP4 rows (E2M1 codes + fp32 row scale):
 * every K/V element is scale_row * E2M1(code), exactly, in double.
 */
int kvd_oracle_attend_masked_fp4(const void* q, int qtype, const uint8_t* k, const uint8_t* v,
                                 const uint8_t* mask, int B, int Hq, int Hkv, int C, int D,
                                 double scale, double* out, double* lse, int nthreads) {
    return orc_attend_masked(q, qtype, k, v, ORC_FP4ROW, mask, B, Hq, Hkv, C, D, scale, out, lse,
                             nthreads);
}

/*
 * Index-list decode attention ([FlashMLA] "Математическая постановка": the
 * indexer's top-k indices pick the KV rows; P = Q . gathered^T,
 * S = softmax(P * sm_scale), out = S . gathered).
 *   q [B, Hq, D]; k, v [B, Hkv, C, D]; indices [B, topk] (int32)
 *   out [B, Hq, D] double; lse [B, Hq] double or NULL
 * Every list entry j with 0 <= indices[b, j] < C is one term of the softmax
 * (a repeated index counts once per entry); -1 marks an unused entry; any
 * other value is skipped and sets ORC_ERR_POS.  No valid entry: out = 0,
 * lse = -inf.  Returns the error bits (or < 0 on bad sizes / no memory).
 */
int kvd_oracle_attend_indexed(const void* q, const void* k, const void* v,
                              const int32_t* indices, int dtype, int B, int Hq, int Hkv,
                              int C, int topk, int D, double scale, double* out, double* lse,
                              int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || C < 0 || topk < 0 || D <= 0 || Hq % Hkv) return -1;
    const int g = Hq / Hkv;
    const long units = (long)B * Hq;
    int err = 0;
    for (long i = 0; i < (long)B * topk; ++i)
        if (indices[i] < -1 || indices[i] >= C) err |= ORC_ERR_POS;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        const int b = (int)(u / Hq), h = (int)(u % Hq), kvh = h / g;
        double* s = (double*)malloc(sizeof(double) * (topk > 0 ? topk : 1));
        double* num = (double*)malloc(sizeof(double) * D);
        if (!s || !num) {
            free(s);
            free(num);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        const size_t qbase = ((size_t)b * Hq + h) * D;
        const size_t kvbase = ((size_t)b * Hkv + kvh) * (size_t)C * D;
        const int32_t* idx = indices + (size_t)b * topk;
        /* pass 1: scores of the listed rows and their maximum */
        double m = -INFINITY;
        long nvalid = 0;
        for (int j = 0; j < topk; ++j) {
            const int t = idx[j];
            if (t < 0 || t >= C) continue;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += orc_elem(q, qbase + d, dtype) * orc_elem(k, kvbase + (size_t)t * D + d, dtype);
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
            ++nvalid;
        }
        double* o = out + qbase;
        if (nvalid == 0) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (lse) lse[(size_t)b * Hq + h] = -INFINITY;
            free(s);
            free(num);
            continue;
        }
        /* pass 2: softmax weights and the weighted sum of the listed V rows */
        double den = 0.0;
        for (int d = 0; d < D; ++d) num[d] = 0.0;
        for (int j = 0; j < topk; ++j) {
            const int t = idx[j];
            if (t < 0 || t >= C) continue;
            const double w = exp(s[j] - m);
            den += w;
            for (int d = 0; d < D; ++d) num[d] += w * orc_elem(v, kvbase + (size_t)t * D + d, dtype);
        }
        for (int d = 0; d < D; ++d) o[d] = num[d] / den;
        if (lse) lse[(size_t)b * Hq + h] = m + log(den);
        free(s);
        free(num);
    }
    return failed ? -2 : err;
}

/*
 * KV append: row pos[b] of every kv head of k_cache / v_cache [B, Hkv, C, D]
 * becomes k_new / v_new [B, Hkv, D]; if mask [B, C] is given its slot
 * pos[b] becomes 1.  A position outside [0, C) writes nothing for that batch
 * entry and sets ORC_ERR_POS.  Pure byte copy.
 */
int kvd_oracle_append(void* k_cache, void* v_cache, const void* k_new,
                      const void* v_new, const int32_t* pos, uint8_t* mask,
                      int B, int Hkv, int C, int D, int elem_bytes) {
    int err = 0;
    const size_t row = (size_t)D * elem_bytes;
    for (int b = 0; b < B; ++b) {
        const int p = pos[b];
        if (p < 0 || p >= C) {
            err |= ORC_ERR_POS;
            continue;
        }
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)b * Hkv + h) * C + p) * row;
            const size_t src = ((size_t)b * Hkv + h) * row;
            memcpy((char*)k_cache + dst, (const char*)k_new + src, row);
            memcpy((char*)v_cache + dst, (const char*)v_new + src, row);
        }
        if (mask) mask[(size_t)b * C + p] = 1;
    }
    return err;
}

/*
 * KV append into quantised caches ([NPU-KV] Part 2, update_kvcache_for, with
 * the row format of [FlashMLA-KV]): row pos[b] of every kv head of k_cache /
 * v_cache [B, Hkv, C, D + 16] bytes becomes the quantised k_new / v_new
 * [B, Hkv, D] (dtype); mask slot pos[b] becomes 1.  A position outside
 * [0, C) writes nothing for that entry and sets ORC_ERR_POS.
 */
int kvd_oracle_append_fp8(uint8_t* k_cache, uint8_t* v_cache, const void* k_new,
                          const void* v_new, int dtype, const int32_t* pos, uint8_t* mask,
                          int B, int Hkv, int C, int D) {
    int err = 0;
    const size_t rb = (size_t)D + 16;
    for (int b = 0; b < B; ++b) {
        const int p = pos[b];
        if (p < 0 || p >= C) {
            err |= ORC_ERR_POS;
            continue;
        }
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)b * Hkv + h) * C + p) * rb;
            orc_quantize_row(k_new, (size_t)b * Hkv + h, dtype, D, k_cache + dst);
            orc_quantize_row(v_new, (size_t)b * Hkv + h, dtype, D, v_cache + dst);
        }
        if (mask) mask[(size_t)b * C + p] = 1;
    }
    return err;
}

/*
 * KV append into FP4 caches: row pos[b] of every kv head of k_cache /
 * v_cache [B, Hkv, C, D/2 + 16] bytes becomes the FP4-quantised k_new / v_new
 * [B, Hkv, D] (dtype); mask slot pos[b] becomes 1.  A position outside
 * [0, C) writes nothing for that entry and sets ORC_ERR_POS.
 */
int kvd_oracle_append_fp4(uint8_t* k_cache, uint8_t* v_cache, const void* k_new,
                          const void* v_new, int dtype, const int32_t* pos, uint8_t* mask,
                          int B, int Hkv, int C, int D) {
    int err = 0;
    const size_t rb = (size_t)D / 2 + 16;
    for (int b = 0; b < B; ++b) {
        const int p = pos[b];
        if (p < 0 || p >= C) {
            err |= ORC_ERR_POS;
            continue;
        }
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)b * Hkv + h) * C + p) * rb;
            orc_quantize_row_fp4(k_new, (size_t)b * Hkv + h, dtype, D, k_cache + dst);
            orc_quantize_row_fp4(v_new, (size_t)b * Hkv + h, dtype, D, v_cache + dst);
        }
        if (mask) mask[(size_t)b * C + p] = 1;
    }
    return err;
}

/*
 * Prefill -> generate hand-over (copy_kvcache) for one layer
 * ([NPU-KV] Part 2 "NPUW 的核心设计", step 3: the prefill model's present
 * K/V, capacity 1024, are copied as the slice [0:N] into the generate
 * model's past K/V, capacity 1152; 32 layers x K and V):
 *   k_src, v_src [B, Hkv, C_src, D];  k_dst, v_dst [B, Hkv, C_dst, D]
 *   n [B]: rows to copy for batch entry b (the prompt length)
 *   mask [B, C_dst] uint8 or NULL: becomes 1 on [0, n[b]) and 0 after.
 * n[b] outside [0, min(C_src, C_dst)] copies nothing for b, leaves its mask
 * alone and sets ORC_ERR_POS.  Pure byte copy.
 */
int kvd_oracle_copy_prefix(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                           uint8_t* mask, const int32_t* n, int B, int Hkv, int C_src,
                           int C_dst, int D, int elem_bytes) {
    int err = 0;
    const size_t row = (size_t)D * elem_bytes;
    const int cmax = C_src < C_dst ? C_src : C_dst;
    for (int b = 0; b < B; ++b) {
        const int nb = n[b];
        if (nb < 0 || nb > cmax) {
            err |= ORC_ERR_POS;
            continue;
        }
        for (int h = 0; h < Hkv; ++h)
            for (int t = 0; t < nb; ++t) {
                const size_t src = (((size_t)b * Hkv + h) * C_src + t) * row;
                const size_t dst = (((size_t)b * Hkv + h) * C_dst + t) * row;
                memcpy((char*)k_dst + dst, (const char*)k_src + src, row);
                memcpy((char*)v_dst + dst, (const char*)v_src + src, row);
            }
        if (mask)
            for (int t = 0; t < C_dst; ++t) mask[(size_t)b * C_dst + t] = t < nb ? 1 : 0;
    }
    return err;
}

/*
 * Paged gather (gather_pa_kv_cache, Norm/ND branch):
 *   key_cache [NB, BS, Hk, Dk], value_cache [NB, BS, Hv, Dv]
 *   block_tables [Q, cols], seq_lens [Q + 1] cumsum with seq_lens[0] = 0,
 *   seq_offset [Q] or NULL (zeros)
 *   key_out [total, Hk, Dk], value_out [total, Hv, Dv]
 * For every sequence q and token t < seq_lens[q+1] - seq_lens[q]:
 *   physical = block_tables[q, seq_offset[q] / BS + t / BS]
 *   key_out[seq_lens[q] + t] = key_cache[physical, t % BS]   (same for value)
 * Checks follow the page's constraints; a violating sequence (or token) is
 * not written and its error bit is returned.
 */
int kvd_oracle_gather_paged(const void* key_cache, const void* value_cache,
                            const int32_t* block_tables,
                            const int32_t* seq_lens, const int32_t* seq_offset,
                            void* key_out, void* value_out, int Q, int NB,
                            int BS, int cols, int Hk, int Dk, int Hv, int Dv,
                            int total_tokens, int elem_bytes) {
    int err = 0;
    const size_t krow = (size_t)Hk * Dk * elem_bytes;
    const size_t vrow = (size_t)Hv * Dv * elem_bytes;
    if (seq_lens[0] != 0) err |= ORC_ERR_SEQLENS;
    for (int q = 0; q < Q; ++q) {
        const long start = seq_lens[q], end = seq_lens[q + 1];
        if (end < start || start < 0 || end > total_tokens) {
            err |= ORC_ERR_SEQLENS;
            continue;
        }
        const long len = end - start;
        const long off = seq_offset ? seq_offset[q] : 0;
        if (off < 0 || off % BS) {
            err |= ORC_ERR_OFFSET;
            continue;
        }
        const long first_col = off / BS;
        const long nblocks = (len + BS - 1) / BS;
        if (first_col + nblocks > cols) {
            err |= ORC_ERR_COLS;
            continue;
        }
        for (long t = 0; t < len; ++t) {
            const long logical = t / BS, slot = t % BS;
            const long phys = block_tables[(size_t)q * cols + first_col + logical];
            if (phys < 0 || phys >= NB) {
                err |= ORC_ERR_BLOCK;
                continue;
            }
            memcpy((char*)key_out + (size_t)(start + t) * krow,
                   (const char*)key_cache + ((size_t)phys * BS + slot) * krow, krow);
            memcpy((char*)value_out + (size_t)(start + t) * vrow,
                   (const char*)value_cache + ((size_t)phys * BS + slot) * vrow, vrow);
        }
    }
    return err;
}

/*
 * Paged KV append: the step's new token of sequence q goes where the paged
 * gather (above) finds token pos[q] of q -- the same index mapping, written
 * instead of read:
 *   physical = block_tables[q, seq_offset[q] / BS + pos[q] / BS]
 *   key_cache[physical, pos[q] % BS] = k_new[q]   (all Hkv x D; same for value)
 *   key_cache, value_cache [NB, BS, Hkv, D]; k_new, v_new [Q, Hkv, D];
 *   pos [Q]; seq_offset [Q] or NULL (zeros).
 * A sequence whose pos is negative (ORC_ERR_POS), whose seq_offset is
 * negative or not a multiple of BS (ORC_ERR_OFFSET), whose column is past the
 * table (ORC_ERR_COLS) or whose block id is outside [0, NB) (ORC_ERR_BLOCK)
 * writes nothing; the bits are returned.  Pure byte copy.
 */
int kvd_oracle_append_paged(void* key_cache, void* value_cache, const int32_t* block_tables,
                            const int32_t* seq_offset, const void* k_new, const void* v_new,
                            const int32_t* pos, int Q, int NB, int BS, int cols, int Hkv, int D,
                            int elem_bytes) {
    int err = 0;
    const size_t row = (size_t)Hkv * D * elem_bytes;
    for (int q = 0; q < Q; ++q) {
        const long t = pos[q];
        if (t < 0) {
            err |= ORC_ERR_POS;
            continue;
        }
        const long off = seq_offset ? seq_offset[q] : 0;
        if (off < 0 || off % BS) {
            err |= ORC_ERR_OFFSET;
            continue;
        }
        const long col = off / BS + t / BS;
        if (col >= cols) {
            err |= ORC_ERR_COLS;
            continue;
        }
        const long phys = block_tables[(size_t)q * cols + col];
        if (phys < 0 || phys >= NB) {
            err |= ORC_ERR_BLOCK;
            continue;
        }
        const size_t dst = ((size_t)phys * BS + (size_t)(t % BS)) * row;
        memcpy((char*)key_cache + dst, (const char*)k_new + (size_t)q * row, row);
        memcpy((char*)value_cache + dst, (const char*)v_new + (size_t)q * row, row);
    }
    return err;
}

/*
 * Paged decode attention: for sequence q, the keys and values are the rows
 * the gather above produces for q (all of them valid), and the query
 * q_in[q, h, :] attends over them with kv head h / (Hq / Hkv).
 *   q_in [Q, Hq, D], caches [NB, BS, Hkv, D], out [Q, Hq, D], lse [Q, Hq]
 * Written as the composition "gather, then masked attention with an
 * all-ones mask", with no other arithmetic of its own.
 */
int kvd_oracle_attend_paged(const void* q_in, const void* key_cache,
                            const void* value_cache,
                            const int32_t* block_tables,
                            const int32_t* seq_lens, const int32_t* seq_offset,
                            int dtype, int Q, int Hq, int Hkv, int NB, int BS,
                            int cols, int D, double scale, double* out,
                            double* lse, int nthreads) {
    const int eb = dtype == ORC_BF16 ? 2 : 4;
    if (seq_lens[0] != 0) return ORC_ERR_SEQLENS;
    const int total = seq_lens[Q];
    for (int q = 0; q < Q; ++q)
        if (seq_lens[q + 1] < seq_lens[q]) return ORC_ERR_SEQLENS;
    const size_t row = (size_t)Hkv * D * eb;
    char* kg = (char*)malloc(row * (size_t)(total > 0 ? total : 1));
    char* vg = (char*)malloc(row * (size_t)(total > 0 ? total : 1));
    if (!kg || !vg) {
        free(kg);
        free(vg);
        return -2;
    }
    int err = kvd_oracle_gather_paged(key_cache, value_cache, block_tables,
                                      seq_lens, seq_offset, kg, vg, Q, NB, BS,
                                      cols, Hkv, D, Hkv, D, total, eb);
    if (err) {
        free(kg);
        free(vg);
        return err;
    }
    int rc = 0;
    for (int q = 0; q < Q && rc == 0; ++q) {
        const int len = seq_lens[q + 1] - seq_lens[q];
        /* the gathered rows of q, viewed as a [1, len, Hkv, D] block, are
         * re-laid as [1, Hkv, len, D] for the static-buffer oracle */
        const size_t e = (size_t)eb;
        char* kq = (char*)malloc((size_t)Hkv * (len > 0 ? len : 1) * D * e);
        char* vq = (char*)malloc((size_t)Hkv * (len > 0 ? len : 1) * D * e);
        uint8_t* ones = (uint8_t*)malloc(len > 0 ? len : 1);
        if (!kq || !vq || !ones) {
            free(kq);
            free(vq);
            free(ones);
            rc = -2;
            break;
        }
        for (int t = 0; t < len; ++t) {
            ones[t] = 1;
            for (int h = 0; h < Hkv; ++h) {
                const size_t src = ((size_t)(seq_lens[q] + t) * Hkv + h) * D * e;
                const size_t dst = ((size_t)h * len + t) * D * e;
                memcpy(kq + dst, kg + src, D * e);
                memcpy(vq + dst, vg + src, D * e);
            }
        }
        rc = kvd_oracle_attend_masked((const char*)q_in + (size_t)q * Hq * D * e,
                                      kq, vq, ones, dtype, 1, Hq, Hkv, len, D,
                                      scale, out + (size_t)q * Hq * D,
                                      lse ? lse + (size_t)q * Hq : NULL,
                                      nthreads);
        free(kq);
        free(vq);
        free(ones);
    }
    free(kg);
    free(vg);
    return rc;
}

/*
 * Log-sum-exp combine of partial results over disjoint key ranges:
 *   part_o [R, S, D] (each normalised within its range), part_lse [R, S]
 *   LSE = log sum_s exp(lse_s),  out = sum_s exp(lse_s - LSE) * o_s.
 * Ranges with lse = -inf carry weight 0; a row whose ranges are all empty
 * gives out = 0 and LSE = -inf.
 */
int kvd_oracle_combine(const double* part_o, const double* part_lse, int R,
                       int S, int D, double* out, double* lse) {
    for (int r = 0; r < R; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (part_lse[(size_t)r * S + s] > m) m = part_lse[(size_t)r * S + s];
        double* o = out + (size_t)r * D;
        if (m == -INFINITY) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (lse) lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int s = 0; s < S; ++s) sum += exp(part_lse[(size_t)r * S + s] - m);
        const double L = m + log(sum);
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int s = 0; s < S; ++s) {
            const double ls = part_lse[(size_t)r * S + s];
            if (ls == -INFINITY) continue;
            const double w = exp(ls - L);
            for (int d = 0; d < D; ++d)
                o[d] += w * part_o[((size_t)r * S + s) * D + d];
        }
        if (lse) lse[r] = L;
    }
    return 0;
}
