/*
 * qmlp_oracle.c -- plain, slow CPU oracle for the weight-quantized SwiGLU MLP.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links,
 * loads or calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header, table or constant with the
 * CUDA sources: every table here is built from the format definitions below.
 *
 * Arithmetic: every weight is decoded exactly (by table) to double, every dot
 * product is a sequential double-precision sum over k = 0..K-1, and results
 * are rounded (IEEE round-to-nearest-even, directly from double) only where the
 * computed method rounds:
 *   - the SwiGLU intermediate act is rounded to bf16 before the down
 *     projection, and the MLP output is rounded to bf16;
 *   - the AWQ routed-expert path rounds gate/up, act and each route's output
 *     to fp16 and the router-weighted sum to fp16 ("What it does", 1Cat-vLLM
 *     PR "[Kernel][SM70] Add native-g32 AWQ QPN M1 operator").
 * Output rows are independent; they are spread over OpenMP threads without
 * changing any per-output summation order.
 *
 * Readings taken where the pages are silent:
 *   - E2M1 is the OCP MX FP4 element (sign, 2 exponent bits with bias 1,
 *     1 mantissa bit); the pages only name it.
 *   - The NVFP4 global factor is the fp32 value 1.0f/global, applied to the
 *     fp64 dot product of x with E2M1*E4M3 (one IEEE fp32 division).
 *   - SiLU(t) = t / (1 + exp(-t)).
 *   - AWQ metadata records are packed little-endian: fp16 scale in bytes 0-1,
 *     then the fp16 bias (4-byte record) or the u8 zero (3-byte record).
 *   - An expert id outside [0, E) marks an invalid route.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Element decode tables                                                    */
/* ------------------------------------------------------------------------ */

static double E2M1_TABLE[16];
static double E4M3_TABLE[256];
static int TABLES_READY = 0;

/* E2M1 (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented": "two E2M1 values
 * per byte"): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 encodes the subnormals 0 and 0.5. */
static double e2m1_from_fields(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 / float8_e4m3fn (same page, "weight_scale -- E4M3"; vllm.cpp issue,
 * "Mechanism on the tp>1 path": "e4m3fn [n,k] bytes"): bit 7 sign, bits 6..3
 * exponent (bias 7), bits 2..0 mantissa, no infinities, S.1111.111 is NaN. */
static double e4m3_from_fields(int byte) {
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

static void init_tables(void) {
    if (TABLES_READY) return;
    for (int c = 0; c < 16; ++c) E2M1_TABLE[c] = e2m1_from_fields(c);
    for (int b = 0; b < 256; ++b) E4M3_TABLE[b] = e4m3_from_fields(b);
    TABLES_READY = 1;
}

double qo_e2m1(int code) { init_tables(); return E2M1_TABLE[code & 15]; }
double qo_e4m3(int byte) { init_tables(); return E4M3_TABLE[byte & 255]; }

/* ------------------------------------------------------------------------ */
/* IEEE binary16 / bfloat16 rounding from double (round to nearest even)     */
/* ------------------------------------------------------------------------ */

/* Round |v| to a binary format with `ebits` exponent bits and `mbits` stored
 * mantissa bits; returns the encoding. One rounding, directly from double. */
static uint16_t round_to_format(double v, int ebits, int mbits) {
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias;
    const uint16_t sign = signbit(v) ? (uint16_t)(1u << (ebits + mbits)) : 0;
    const uint16_t exp_all = (uint16_t)(((1u << ebits) - 1) << mbits);
    if (isnan(v)) return (uint16_t)(sign | exp_all | (1u << (mbits - 1)));
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | exp_all);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);                 /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    if (E < emin) E = emin;        /* subnormal range shares emin's quantum */
    double quantum = ldexp(1.0, E - mbits);
    double n = a / quantum;        /* exact: division by a power of two */
    double fl = floor(n), r = n - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    if (fl == 0.0) return sign;
    double lead = ldexp(1.0, mbits);
    if (fl >= 2.0 * lead) { fl /= 2.0; E += 1; }       /* carry into exponent */
    if (fl < lead) return (uint16_t)(sign | (uint16_t)fl); /* subnormal */
    int biased = E + bias;
    if (biased >= (1 << ebits) - 1) return (uint16_t)(sign | exp_all); /* overflow */
    return (uint16_t)(sign | (uint16_t)(biased << mbits) | (uint16_t)(fl - lead));
}

static double value_of_format(uint16_t bits, int ebits, int mbits) {
    const int bias = (1 << (ebits - 1)) - 1;
    int s = (bits >> (ebits + mbits)) & 1;
    int e = (bits >> mbits) & ((1 << ebits) - 1);
    int m = bits & ((1 << mbits) - 1);
    double mag;
    if (e == (1 << ebits) - 1) mag = m ? NAN : INFINITY;
    else if (e == 0) mag = ldexp((double)m, 1 - bias - mbits);
    else mag = ldexp(1.0 + ldexp((double)m, -mbits), e - bias);
    return s ? -mag : mag;
}

uint16_t qo_bf16_rne(double v) { return round_to_format(v, 8, 7); }
uint16_t qo_fp16_rne(double v) { return round_to_format(v, 5, 10); }
double qo_bf16_value(uint16_t b) { return value_of_format(b, 8, 7); }
double qo_fp16_value(uint16_t b) { return value_of_format(b, 5, 10); }

void qo_bf16_rne_array(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = qo_bf16_rne(v[i]);
}
void qo_fp16_rne_array(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = qo_fp16_rne(v[i]);
}

static double silu(double t) { return t / (1.0 + exp(-t)); }

/* ------------------------------------------------------------------------ */
/* Dense projections (NVFP4 group-16 and FP8 per-channel)                    */
/* ------------------------------------------------------------------------ */

enum { QO_NVFP4 = 1, QO_FP8 = 2 };

typedef struct {
    const uint8_t* w;      /* NVFP4: [N, K/2] packed; FP8: [N, K] e4m3fn */
    const void* scale;     /* NVFP4: e4m3 [N, K/16]; FP8: float [N]      */
    float global_scale;    /* NVFP4 only                                  */
} qo_proj;

/* Decode row n of a projection to double, WITHOUT the per-tensor global
 * factor (NVFP4) or the per-channel scale (FP8).
 *  NVFP4 (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented"): the weight at
 *  (n, k) is E2M1(nibble) * E4M3(scale[n, k/16]); byte k/2 of row n holds k
 *  in its low nibble when k is even ("the low nibble is the earlier logical
 *  weight").
 *  FP8 (vllm.cpp issue, "Mechanism on the tp>1 path"): F8E4M3ToF32(w[n, k]). */
static void decode_row(int fmt, const qo_proj* p, int K, int n, double* out) {
    if (fmt == QO_NVFP4) {
        const uint8_t* wr = p->w + (size_t)n * (K / 2);
        const uint8_t* sr = (const uint8_t*)p->scale + (size_t)n * (K / 16);
        for (int k = 0; k < K; ++k) {
            uint8_t byte = wr[k / 2];
            int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
            out[k] = E2M1_TABLE[code] * E4M3_TABLE[sr[k / 16]];
        }
    } else {
        const uint8_t* wr = p->w + (size_t)n * K;
        for (int k = 0; k < K; ++k) out[k] = E4M3_TABLE[wr[k]];
    }
}

void qo_decode_proj(int fmt, const qo_proj* p, int N, int K, double* out) {
    init_tables();
    for (int n = 0; n < N; ++n) decode_row(fmt, p, K, n, out + (size_t)n * K);
}

/* Output-channel factor sigma of a projection:
 *  NVFP4: fp32(1/global) (Qwen3.8-27B-NVFP4: "The runtime dequantization
 *  factor is 1 / weight_global_scale"); FP8: scale[n] (vllm.cpp issue,
 *  "out[n,k] = F8E4M3ToF32(w[n,k]) * scale[n]"). */
static double channel_factor(int fmt, const qo_proj* p, int n) {
    if (fmt == QO_NVFP4) {
        float inv = 1.0f / p->global_scale;
        return (double)inv;
    }
    return (double)((const float*)p->scale)[n];
}

static double dot(const double* a, const double* b, int K) {
    double s = 0.0;
    for (int k = 0; k < K; ++k) s += a[k] * b[k];
    return s;
}

/* y[r, n] = sum_k x[rows[r], k] * decode(W)[n, k]  (no channel factor), the
 * projection in isolation; x given as bf16 bits [M, K]. */
void qo_project(int fmt, const qo_proj* p, int N, int K, const uint16_t* x, int nrows,
                const int32_t* rows, double* y) {
    init_tables();
    double* xr = (double*)malloc(sizeof(double) * (size_t)nrows * K);
    for (int r = 0; r < nrows; ++r)
        for (int k = 0; k < K; ++k) xr[(size_t)r * K + k] = qo_bf16_value(x[(size_t)rows[r] * K + k]);
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * K);
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            decode_row(fmt, p, K, n, wrow);
            for (int r = 0; r < nrows; ++r) y[(size_t)r * N + n] = dot(xr + (size_t)r * K, wrow, K);
        }
        free(wrow);
    }
    free(xr);
}

/* The SwiGLU MLP block on token rows `rows` of x (bf16 bits [M, K]).
 * vllm.cpp issue, "Proposed fix":
 *   act[i] = SiLU(sum_k x[k] * Wg[i,k] * sg[i]) * (sum_k x[k] * Wu[i,k] * su[i])
 *   out[o] = sum_q act[q] * Wd[o,q] * sd[o]
 * with the per-channel factors sigma applied to each dot product. act is
 * rounded to bf16 before the down projection and out is rounded to bf16.
 * Optional outputs: g_pre/u_pre = sigma*dot before SiLU ([nrows, I], double),
 * act_bits ([nrows, I], bf16), out_pre ([nrows, K], double, before rounding). */
void qo_dense_forward(int fmt, int K, int I, const uint16_t* x, int nrows, const int32_t* rows,
                      const qo_proj* gate, const qo_proj* up, const qo_proj* down,
                      uint16_t* out_bits, uint16_t* act_bits_opt, double* g_pre_opt,
                      double* u_pre_opt, double* out_pre_opt) {
    init_tables();
    double* xr = (double*)malloc(sizeof(double) * (size_t)nrows * K);
    double* act = (double*)malloc(sizeof(double) * (size_t)nrows * I);
    for (int r = 0; r < nrows; ++r)
        for (int k = 0; k < K; ++k) xr[(size_t)r * K + k] = qo_bf16_value(x[(size_t)rows[r] * K + k]);

#pragma omp parallel
    {
        double* wg = (double*)malloc(sizeof(double) * K);
        double* wu = (double*)malloc(sizeof(double) * K);
#pragma omp for schedule(static)
        for (int i = 0; i < I; ++i) {
            decode_row(fmt, gate, K, i, wg);
            decode_row(fmt, up, K, i, wu);
            double sg = channel_factor(fmt, gate, i), su = channel_factor(fmt, up, i);
            for (int r = 0; r < nrows; ++r) {
                double g = sg * dot(xr + (size_t)r * K, wg, K);
                double u = su * dot(xr + (size_t)r * K, wu, K);
                uint16_t a = qo_bf16_rne(silu(g) * u);
                act[(size_t)r * I + i] = qo_bf16_value(a);
                if (act_bits_opt) act_bits_opt[(size_t)r * I + i] = a;
                if (g_pre_opt) g_pre_opt[(size_t)r * I + i] = g;
                if (u_pre_opt) u_pre_opt[(size_t)r * I + i] = u;
            }
        }
        free(wg);
        free(wu);
    }

#pragma omp parallel
    {
        double* wd = (double*)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
        for (int o = 0; o < K; ++o) {
            decode_row(fmt, down, I, o, wd);
            double sd = channel_factor(fmt, down, o);
            for (int r = 0; r < nrows; ++r) {
                double v = sd * dot(act + (size_t)r * I, wd, I);
                out_bits[(size_t)r * K + o] = qo_bf16_rne(v);
                if (out_pre_opt) out_pre_opt[(size_t)r * K + o] = v;
            }
        }
        free(wd);
    }
    free(act);
    free(xr);
}

/* ------------------------------------------------------------------------ */
/* AWQ int4 group-32 routed experts, M = 1                                   */
/* ------------------------------------------------------------------------ */

/* One AWQ weight (1Cat-vLLM PR, "What it does"): the u4 code q becomes a half,
 * and the weight is half_fma(q, scale, bias), i.e. q*scale + bias rounded once
 * to fp16; bias is the stored fp16 bias (4-byte record) or half(-zero*scale)
 * (3-byte record). q*s + b is exact in double (every term is a multiple of
 * 2^-24 below 2^5), so one fp16 rounding of the double reproduces the single
 * rounding of half_fma. */
static double awq_weight(int q, const uint8_t* rec, int meta_bytes) {
    uint16_t s_bits = (uint16_t)(rec[0] | (rec[1] << 8));
    double s = qo_fp16_value(s_bits);
    double b;
    if (meta_bytes == 4) {
        b = qo_fp16_value((uint16_t)(rec[2] | (rec[3] << 8)));
    } else {
        b = qo_fp16_value(qo_fp16_rne(-(double)rec[2] * s));
    }
    return qo_fp16_value(qo_fp16_rne((double)q * s + b));
}

/* Decoded row n of expert e of a [E, N, Kr] AWQ tensor (packed [E, N, Kr/2],
 * metadata [E, N, Kr/32] records). */
static void awq_decode_row(const uint8_t* w, const uint8_t* meta, int meta_bytes, int N, int Kr,
                           int e, int n, double* out) {
    const uint8_t* wr = w + ((size_t)e * N + n) * (Kr / 2);
    const uint8_t* mr = meta + ((size_t)e * N + n) * (Kr / 32) * meta_bytes;
    for (int k = 0; k < Kr; ++k) {
        uint8_t byte = wr[k / 2];
        int q = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
        out[k] = awq_weight(q, mr + (size_t)(k / 32) * meta_bytes, meta_bytes);
    }
}

void qo_awq_decode(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int N, int Kr,
                   int e, double* out /* [N, Kr] */) {
    (void)E;
    for (int n = 0; n < N; ++n) awq_decode_row(w, meta, meta_bytes, N, Kr, e, n, out + (size_t)n * Kr);
}

/* The routed-expert M=1 step (1Cat-vLLM PR, "What it does"):
 *  W13: for each route r in router order with a valid id, h[n] = sum_k x[k] *
 *       w13[id][n, k] over n < 2I; g = fp16(h[:I]), u = fp16(h[I:]);
 *       act[r] = fp16(SiLU(g) * u);
 *  W2:  y[r, n] = fp16(sum_q act[r, q] * w2[id][n, q]);
 *  out[n] = fp16(sum over valid r, in router order, of rw[r] * y[r, n]).
 * Invalid routes contribute zero; duplicate valid ids are separate routes with
 * their own router weights. x is fp16 (x_is_bf16 = 0) or bf16 bits [K].
 * Optional per-stage outputs (fp16 bits): gu [topk, 2I], act [topk, I],
 * y [topk, K]; rows of invalid routes are left untouched. */
void qo_moe_m1_forward(int E, int K, int I, int meta_bytes, const uint8_t* w13,
                       const uint8_t* w13_meta, const uint8_t* w2, const uint8_t* w2_meta,
                       const uint16_t* x, int x_is_bf16, const int32_t* ids, const float* rw,
                       int topk, uint16_t* out_bits, uint16_t* gu_opt, uint16_t* act_opt,
                       uint16_t* y_opt) {
    init_tables();
    const int N13 = 2 * I;
    double* xd = (double*)malloc(sizeof(double) * K);
    for (int k = 0; k < K; ++k) xd[k] = x_is_bf16 ? qo_bf16_value(x[k]) : qo_fp16_value(x[k]);
    double* y = (double*)calloc((size_t)topk * K, sizeof(double));
    int* valid = (int*)calloc((size_t)topk, sizeof(int));

    for (int r = 0; r < topk; ++r) {
        int id = ids[r];
        if (id < 0 || id >= E) continue;
        valid[r] = 1;
        double* gu = (double*)malloc(sizeof(double) * N13);
        double* act = (double*)malloc(sizeof(double) * I);
#pragma omp parallel
        {
            double* wrow = (double*)malloc(sizeof(double) * K);
#pragma omp for schedule(static)
            for (int n = 0; n < N13; ++n) {
                awq_decode_row(w13, w13_meta, meta_bytes, N13, K, id, n, wrow);
                uint16_t h = qo_fp16_rne(dot(xd, wrow, K));
                gu[n] = qo_fp16_value(h);
                if (gu_opt) gu_opt[(size_t)r * N13 + n] = h;
            }
            free(wrow);
        }
        for (int q = 0; q < I; ++q) {
            uint16_t a = qo_fp16_rne(silu(gu[q]) * gu[I + q]);
            act[q] = qo_fp16_value(a);
            if (act_opt) act_opt[(size_t)r * I + q] = a;
        }
#pragma omp parallel
        {
            double* wrow = (double*)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
            for (int n = 0; n < K; ++n) {
                awq_decode_row(w2, w2_meta, meta_bytes, K, I, id, n, wrow);
                uint16_t h = qo_fp16_rne(dot(act, wrow, I));
                y[(size_t)r * K + n] = qo_fp16_value(h);
                if (y_opt) y_opt[(size_t)r * K + n] = h;
            }
            free(wrow);
        }
        free(gu);
        free(act);
    }
    for (int n = 0; n < K; ++n) {
        double s = 0.0;
        for (int r = 0; r < topk; ++r)
            if (valid[r]) s += (double)rw[r] * y[(size_t)r * K + n];
        out_bits[n] = qo_fp16_rne(s);
    }
    free(valid);
    free(y);
    free(xd);
}

int qo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
