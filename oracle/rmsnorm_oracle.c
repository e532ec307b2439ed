/*
 * CPU oracle for the fused residual-add + RMSNorm (TEST INFRASTRUCTURE).
 *
 * This file is the plain, slow reference that the CUDA path is checked
 * against.  Only the tests, the package's smoke check and the bench's CPU
 * baseline use it; the library's compute path never calls it.  It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * What it computes (blog "CuTeDSL at Perplexity", section "QK norm"): the
 * regular RMS norm.  The formula printed in that section has lost its
 * reciprocal square root; the kernel listing that follows it is read
 * instead: square and sum the elements, divide by the vector length, add EPS,
 * take the reciprocal square root, multiply the input by it and then by the
 * weight plus the scalar WEIGHT_BIAS, and cast to the element type.
 * WEIGHT_BIAS is the "with or without weight bias" knob of section
 * "Inference at Perplexity"; here it is `weight_offset`.  On top of the norm,
 * per the fused hot path:
 *
 *   per token t, for j in [0, H):
 *     h_j    = RN_in(x_j + r_j)            (exact sum, rounded once; or x_j)
 *     ms     = (sum_j h_j^2) / H            (fp64)
 *     inv    = 1 / sqrt(ms + eps)           (fp64)
 *     yhat_j = (w_j + weight_offset) * (h_j * inv) + b_j     (fp64)
 *     out    : RN_out(yhat_j) for f32 / bf16 / f64 outputs, or
 *              a = max_j |yhat_j|, s = a / 448, scale_t = RN_f32(s),
 *              q_j = E4M3_RNE_SATFINITE(yhat_j / s)   (q_j = +0 if a == 0)
 *
 * The FP8 path (section "Blackwell support": FP8 block scaling with an
 * absolute-maximum reduction) uses one block per token; 448 is the largest
 * finite OCP FP8 E4M3 value.  The norm is taken on the ROUNDED residual h,
 * the value written to residual_out.
 *
 * Everything is accumulated in double and rounded once at the end.  The
 * bfloat16 and E4M3 encoders below are written from the IEEE-754 binary
 * format rules and the OCP 8-bit floating point specification (E4M3: bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, max 448).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_FP8E4M3 = 2, ORC_F64 = 3, ORC_F16 = 4 };

/* ------------------------------------------------------------------ */
/* number formats                                                      */

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double f32_bits_to_f64(const void *p, int64_t i) {
    float f;
    memcpy(&f, (const char *)p + 4 * i, 4);
    return (double)f;
}

/* Round |v| to a multiple of 2^q_exp, ties to even.  Scaling by a power of
 * two is exact, so rint (round-half-even in the default mode) is the only
 * rounding step. */
static double round_to_quantum(double a, int q_exp) {
    return ldexp(rint(ldexp(a, -q_exp)), q_exp);
}

/* bfloat16: 8 significant bits, exponent range of binary32
 * (normal >= 2^-126, subnormal quantum 2^-133, max (2 - 2^-7) * 2^127). */
uint16_t oracle_bf16_from_f64(double v) {
    if (isnan(v)) return 0x7FC0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    double r;
    if (isinf(a)) {
        r = INFINITY;
    } else if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
        int q = e - 8;                /* 8 significant bits */
        if (q < -133) q = -133;       /* subnormal quantum */
        r = round_to_quantum(a, q);
        const double maxf = ldexp(255.0, 127 - 7);
        if (r > maxf) r = INFINITY;   /* rounded past the largest finite */
    }
    float f = (float)r;               /* exact: r is a bfloat16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t b = (uint16_t)(u >> 16);
    return (uint16_t)(b | (neg ? 0x8000 : 0));
}

float oracle_f32_from_f64(double v) { return (float)v; /* IEEE cast: RNE */ }

/* IEEE-754 binary16: 11 significant bits, normal >= 2^-14, subnormal quantum
 * 2^-24, largest finite 65504 = (2 - 2^-10) * 2^15; rounding past it gives
 * infinity. */
double oracle_f16_to_f64(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

uint16_t oracle_f16_from_f64(double v) {
    if (isnan(v)) return 0x7E00;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v), r;
    if (isinf(a)) {
        r = INFINITY;
    } else if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);              /* a in [2^(e-1), 2^e) */
        int q = e - 11;            /* 11 significant bits */
        if (q < -24) q = -24;      /* subnormal quantum */
        r = round_to_quantum(a, q);
        if (r > 65504.0) r = INFINITY;
    }
    uint16_t h;
    if (isinf(r)) {
        h = 0x7C00;
    } else if (r < ldexp(1.0, -14)) {
        h = (uint16_t)ldexp(r, 24);          /* subnormal: m * 2^-24 */
    } else {
        int e;
        double f = frexp(r, &e);             /* r = f * 2^e, f in [0.5, 1) */
        h = (uint16_t)(((e - 1 + 15) << 10) | ((int)ldexp(f, 11) - 1024));
    }
    return (uint16_t)(h | (neg ? 0x8000 : 0));
}

double oracle_e4m3_to_f64(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* OCP E4M3 with round-to-nearest-even and saturation to +-448 for finite
 * magnitudes above the largest finite value (and for infinities). */
uint8_t oracle_e4m3_from_f64(double v) {
    if (isnan(v)) return 0x7F;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else if (isinf(a)) {
        r = 448.0;
    } else {
        int e;
        frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
        int q = e - 4;                /* 4 significant bits */
        if (q < -9) q = -9;           /* subnormal quantum 2^-9 */
        r = round_to_quantum(a, q);
        if (r > 448.0) r = 448.0;
    }
    uint8_t code;
    if (r < ldexp(1.0, -6)) {
        code = (uint8_t)ldexp(r, 9);  /* subnormal: m * 2^-9 */
    } else {
        int e;
        double f = frexp(r, &e);      /* r = f * 2^e, f in [0.5, 1) */
        int ef = e - 1 + 7;           /* biased exponent of r in [2^(e-1), 2^e) */
        int m = (int)ldexp(f, 4) - 8; /* 3 mantissa bits */
        code = (uint8_t)((ef << 3) | m);
    }
    return (uint8_t)(code | (neg ? 0x80 : 0));
}

/* ------------------------------------------------------------------ */
/* the norm                                                            */

typedef struct {
    const void *x, *residual, *weight, *bias;
    void *out, *residual_out;
    float *out_scale;
    int64_t n_tokens, hidden;
    double eps, weight_offset;
    int in_dtype, out_dtype;
    int res_dtype; /* storage of residual and residual_out */
    int64_t row_begin, row_end;
    int status;
} job_t;

static double load_in(const void *p, int dtype, int64_t i) {
    if (dtype == ORC_F32) return f32_bits_to_f64(p, i);
    uint16_t b;
    memcpy(&b, (const char *)p + 2 * i, 2);
    return dtype == ORC_F16 ? oracle_f16_to_f64(b) : oracle_bf16_to_f64(b);
}

/* RN to the input type; returns the rounded value and stores its bits. */
static double round_store_in(void *p, int dtype, int64_t i, double v) {
    if (dtype == ORC_F32) {
        float f = oracle_f32_from_f64(v);
        if (p) memcpy((char *)p + 4 * i, &f, 4);
        return (double)f;
    }
    if (dtype == ORC_F16) {
        uint16_t h = oracle_f16_from_f64(v);
        if (p) memcpy((char *)p + 2 * i, &h, 2);
        return oracle_f16_to_f64(h);
    }
    uint16_t b = oracle_bf16_from_f64(v);
    if (p) memcpy((char *)p + 2 * i, &b, 2);
    return oracle_bf16_to_f64(b);
}

static void norm_row(const job_t *J, int64_t t, double *h, double *yhat) {
    const int64_t H = J->hidden;
    const int64_t base = t * H;
    /* residual add, rounded once to the input type */
    for (int64_t j = 0; j < H; ++j) {
        double xv = load_in(J->x, J->in_dtype, base + j);
        if (J->residual) {
            double rv = load_in(J->residual, J->res_dtype, base + j);
            h[j] = round_store_in(J->residual_out, J->res_dtype, base + j, xv + rv);
        } else {
            h[j] = xv;
        }
    }
    /* mean square over the true hidden size, eps inside the root */
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) ss += h[j] * h[j];
    const double ms = ss / (double)H;
    const double inv = 1.0 / sqrt(ms + J->eps);
    /* scale */
    for (int64_t j = 0; j < H; ++j) {
        double w = J->weight ? load_in(J->weight, J->in_dtype, j) : 1.0;
        double b = J->bias ? load_in(J->bias, J->in_dtype, j) : 0.0;
        yhat[j] = (w + J->weight_offset) * (h[j] * inv) + b;
    }
    /* output */
    switch (J->out_dtype) {
    case ORC_F64:
        memcpy((double *)J->out + base, yhat, (size_t)H * sizeof(double));
        break;
    case ORC_F32:
        for (int64_t j = 0; j < H; ++j) {
            float f = oracle_f32_from_f64(yhat[j]);
            memcpy((char *)J->out + 4 * (base + j), &f, 4);
        }
        break;
    case ORC_BF16:
        for (int64_t j = 0; j < H; ++j) {
            uint16_t b = oracle_bf16_from_f64(yhat[j]);
            memcpy((char *)J->out + 2 * (base + j), &b, 2);
        }
        break;
    case ORC_F16:
        for (int64_t j = 0; j < H; ++j) {
            uint16_t h = oracle_f16_from_f64(yhat[j]);
            memcpy((char *)J->out + 2 * (base + j), &h, 2);
        }
        break;
    case ORC_FP8E4M3: {
        double a = 0.0;
        for (int64_t j = 0; j < H; ++j)
            if (fabs(yhat[j]) > a) a = fabs(yhat[j]);
        const double s = a / 448.0;
        J->out_scale[t] = oracle_f32_from_f64(s);
        uint8_t *q = (uint8_t *)J->out + base;
        for (int64_t j = 0; j < H; ++j)
            q[j] = (a == 0.0) ? 0 : oracle_e4m3_from_f64(yhat[j] / s);
        break;
    }
    }
}

static void *run_job(void *arg) {
    job_t *J = (job_t *)arg;
    double *h = (double *)malloc((size_t)J->hidden * sizeof(double));
    double *yhat = (double *)malloc((size_t)J->hidden * sizeof(double));
    if (!h || !yhat) {
        J->status = -2;
    } else {
        for (int64_t t = J->row_begin; t < J->row_end; ++t) norm_row(J, t, h, yhat);
        J->status = 0;
    }
    free(h);
    free(yhat);
    return NULL;
}

int oracle_num_cpus(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n < 1 ? 1 : (int)n;
}

/*
 * All pointers are host pointers to contiguous row-major [n_tokens, hidden]
 * arrays (weight and bias: [hidden]).  residual / weight / bias may be NULL
 * (no residual add / w = 1 / b = 0).  residual_out is required when residual
 * is given.  out_scale ([n_tokens] float) is required for ORC_FP8E4M3.
 * n_threads <= 0 uses every online CPU.  Returns 0, or -1 on a bad
 * argument, -2 when a buffer could not be allocated.
 */
int oracle_rmsnorm_res(const void *x, const void *residual, const void *weight, const void *bias,
                       void *out, void *residual_out, float *out_scale, int64_t n_tokens,
                       int64_t hidden, double eps, double weight_offset, int in_dtype,
                       int res_dtype, int out_dtype, int n_threads);

int oracle_rmsnorm(const void *x, const void *residual, const void *weight, const void *bias,
                   void *out, void *residual_out, float *out_scale, int64_t n_tokens,
                   int64_t hidden, double eps, double weight_offset, int in_dtype,
                   int out_dtype, int n_threads) {
    return oracle_rmsnorm_res(x, residual, weight, bias, out, residual_out, out_scale, n_tokens,
                              hidden, eps, weight_offset, in_dtype, in_dtype, out_dtype,
                              n_threads);
}

/*
 * As oracle_rmsnorm, with the residual stream in its own storage type
 * res_dtype (residual and residual_out): h = RN_res(x + r), the norm taken
 * on that h.  An fp32 residual stream with bf16 / fp16 activations keeps h
 * in fp32 (the exact sum rounded once to fp32).
 */
int oracle_rmsnorm_res(const void *x, const void *residual, const void *weight, const void *bias,
                       void *out, void *residual_out, float *out_scale, int64_t n_tokens,
                       int64_t hidden, double eps, double weight_offset, int in_dtype,
                       int res_dtype, int out_dtype, int n_threads) {
    if (n_tokens < 0 || hidden <= 0) return -1;
    if (in_dtype != ORC_F32 && in_dtype != ORC_BF16 && in_dtype != ORC_F16) return -1;
    if (res_dtype != ORC_F32 && res_dtype != ORC_BF16 && res_dtype != ORC_F16) return -1;
    if (out_dtype < ORC_F32 || out_dtype > ORC_F16) return -1;
    if (!x || !out || (residual && !residual_out)) return -1;
    if (out_dtype == ORC_FP8E4M3 && !out_scale) return -1;
    if (n_tokens == 0) return 0;
    if (n_threads <= 0) n_threads = oracle_num_cpus();
    if (n_threads > n_tokens) n_threads = (int)n_tokens;
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    for (int i = 0; i < n_threads; ++i) {
        job_t *J = &jobs[i];
        J->x = x; J->residual = residual; J->weight = weight; J->bias = bias;
        J->out = out; J->residual_out = residual_out; J->out_scale = out_scale;
        J->n_tokens = n_tokens; J->hidden = hidden;
        J->eps = eps; J->weight_offset = weight_offset;
        J->in_dtype = in_dtype; J->out_dtype = out_dtype; J->res_dtype = res_dtype;
        J->row_begin = n_tokens * i / n_threads;
        J->row_end = n_tokens * (i + 1) / n_threads;
        J->status = -3;
    }
    int status = 0;
    int started = 0;
    for (int i = 1; i < n_threads; ++i) {
        if (pthread_create(&tids[i], NULL, run_job, &jobs[i]) != 0) break;
        started = i;
    }
    run_job(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(tids[i], NULL);
    /* rows of threads that could not be started run here */
    for (int i = started + 1; i < n_threads; ++i) run_job(&jobs[i]);
    for (int i = 0; i < n_threads; ++i)
        if (jobs[i].status != 0) status = jobs[i].status;
    free(jobs);
    free(tids);
    return status;
}

/* ------------------------------------------------------------------ */
/* QK norm                                                             */
/*
 * Per-head RMS norm of the query and key heads (blog "CuTeDSL at
 * Perplexity", section "QK norm"): every head vector of length head_dim is
 * normalised on its own, with the query weight for query heads and the key
 * weight for key heads, the scalar WEIGHT_BIAS (weight_offset) added to the
 * weight, and the result cast back to the element type IN PLACE.
 *
 * q holds n_tokens rows of n_q_heads * head_dim elements, row t starting at
 * element t * q_token_stride (likewise k); elements between the heads of a
 * row and the next row start are not touched.  Weights are [head_dim] or
 * NULL (1).  Per head, in fp64, rounded once:
 *   inv = 1 / sqrt(sum_j x_j^2 / head_dim + eps);  x_j <- RN((w_j + off) * (x_j * inv))
 */
static void qk_head(void *base, int dtype, int64_t off0, int64_t head_dim, const void *w,
                    double eps, double woff) {
    double ss = 0.0;
    for (int64_t j = 0; j < head_dim; ++j) {
        double v = load_in(base, dtype, off0 + j);
        ss += v * v;
    }
    const double inv = 1.0 / sqrt(ss / (double)head_dim + eps);
    for (int64_t j = 0; j < head_dim; ++j) {
        double v = load_in(base, dtype, off0 + j);
        double wj = w ? load_in(w, dtype, j) : 1.0;
        round_store_in(base, dtype, off0 + j, (wj + woff) * (v * inv));
    }
}

int oracle_qk_norm(void *q, void *k, const void *q_weight, const void *k_weight,
                   int64_t n_tokens, int64_t n_q_heads, int64_t n_k_heads, int64_t head_dim,
                   int64_t q_token_stride, int64_t k_token_stride, double eps,
                   double weight_offset, int dtype) {
    if (n_tokens < 0 || n_q_heads < 0 || n_k_heads < 0 || head_dim <= 0) return -1;
    if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F16) return -1;
    if (q_token_stride < n_q_heads * head_dim || k_token_stride < n_k_heads * head_dim) return -1;
    if ((n_q_heads && !q) || (n_k_heads && !k)) return -1;
    for (int64_t t = 0; t < n_tokens; ++t) {
        for (int64_t h = 0; h < n_q_heads; ++h)
            qk_head(q, dtype, t * q_token_stride + h * head_dim, head_dim, q_weight, eps,
                    weight_offset);
        for (int64_t h = 0; h < n_k_heads; ++h)
            qk_head(k, dtype, t * k_token_stride + h * head_dim, head_dim, k_weight, eps,
                    weight_offset);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* block-scaled quantisation of the normalised rows                    */
/*
 * Section "Blackwell support" of the blog: MXFP8, MXFP4 and NVFP4 outputs,
 * with the absolute maximum taken over 32 (MX) or 16 (NVFP4) elements.
 * Applied to the fp64 output yhat of the norm, row by row:
 *
 *  MXFP8 / MXFP4 (OCP Microscaling formats): blocks of 32 elements share a
 *   power-of-two scale X = 2^s, s = floor(log2(max|y|)) - emax, where emax is
 *   the exponent of the element format's largest normal (8 for E4M3, 2 for
 *   E2M1), clamped to [-127, 127] and stored as E8M0 (code s + 127); each
 *   element is y / X rounded to the element format (RNE, saturating).  An
 *   all-zero block stores scale code 0 and zero elements.
 *  NVFP4: a per-token fp32 scale g = max|row| / (448 * 6) (stored), blocks of
 *   16 elements with an E4M3 scale s_b = E4M3(max|block| / (6 g)) (RNE,
 *   saturating) and E2M1 elements RN_sat(y / (s_b g)); zero scales give zero
 *   elements.
 *
 * FP4 codes are packed two per byte, element 2j in the low nibble.  The
 * E2M1 format (OCP): sign, 2 exponent bits with bias 1, 1 mantissa bit;
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  E8M0: 2^(code - 127), 255 = NaN.
 */
enum { ORC_MXFP8 = 10, ORC_MXFP4 = 11, ORC_NVFP4 = 12 };

double oracle_e2m1_to_f64(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

uint8_t oracle_e2m1_from_f64(double v) {
    if (isnan(v)) return 0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v), r;
    if (a == 0.0) {
        r = 0.0;
    } else if (isinf(a)) {
        r = 6.0;
    } else {
        int e;
        frexp(a, &e);              /* a in [2^(e-1), 2^e) */
        int q = e - 2;             /* 2 significant bits */
        if (q < -1) q = -1;        /* subnormal quantum 0.5 */
        r = round_to_quantum(a, q);
        if (r > 6.0) r = 6.0;
    }
    uint8_t code;
    if (r < 1.0) {
        code = (uint8_t)(r * 2.0); /* 0 or 0.5 */
    } else {
        int e;
        double f = frexp(r, &e);   /* r = f * 2^e, exponent field e - 1 + 1 */
        code = (uint8_t)((e << 1) | ((int)ldexp(f, 2) - 2));
    }
    return (uint8_t)(code | (neg ? 0x8 : 0));
}

double oracle_e8m0_to_f64(uint8_t c) { return c == 255 ? NAN : ldexp(1.0, (int)c - 127); }

static void quantize_mx_row(const double *y, int64_t H, int elem_fp4, uint8_t *q, uint8_t *sc) {
    const int emax = elem_fp4 ? 2 : 8;
    for (int64_t b = 0; b < H / 32; ++b) {
        const double *yb = y + 32 * b;
        double amax = 0.0;
        for (int j = 0; j < 32; ++j)
            if (fabs(yb[j]) > amax) amax = fabs(yb[j]);
        int s = -127;
        if (amax > 0.0) {
            int e;
            frexp(amax, &e);       /* floor(log2(amax)) = e - 1 */
            s = e - 1 - emax;
            if (s < -127) s = -127;
            if (s > 127) s = 127;
        }
        sc[b] = (uint8_t)(s + 127);
        for (int j = 0; j < 32; ++j) {
            const double v = amax > 0.0 ? ldexp(yb[j], -s) : 0.0;
            const int64_t i = 32 * b + j;
            if (elem_fp4) {
                const uint8_t c = oracle_e2m1_from_f64(v);
                if (i & 1) q[i / 2] = (uint8_t)((q[i / 2] & 0x0F) | (c << 4));
                else q[i / 2] = c;
            } else {
                q[i] = oracle_e4m3_from_f64(v);
            }
        }
    }
}

static void quantize_nvfp4_row(const double *y, int64_t H, uint8_t *q, uint8_t *sc, float *g_out) {
    double a = 0.0;
    for (int64_t j = 0; j < H; ++j)
        if (fabs(y[j]) > a) a = fabs(y[j]);
    const float g = oracle_f32_from_f64(a / (448.0 * 6.0));
    *g_out = g;
    for (int64_t b = 0; b < H / 16; ++b) {
        const double *yb = y + 16 * b;
        double amax = 0.0;
        for (int j = 0; j < 16; ++j)
            if (fabs(yb[j]) > amax) amax = fabs(yb[j]);
        uint8_t sb = 0;
        if (g > 0.0f) sb = oracle_e4m3_from_f64(amax / (6.0 * (double)g));
        sc[b] = sb;
        const double s = oracle_e4m3_to_f64(sb) * (double)g;
        for (int j = 0; j < 16; ++j) {
            const int64_t i = 16 * b + j;
            const uint8_t c = s > 0.0 ? oracle_e2m1_from_f64(yb[j] / s) : 0;
            if (i & 1) q[i / 2] = (uint8_t)((q[i / 2] & 0x0F) | (c << 4));
            else q[i / 2] = c;
        }
    }
}

/*
 * y: [n_tokens, hidden] fp64 rows (the norm's output).  q: [n_tokens,
 * hidden] bytes (MXFP8) or [n_tokens, hidden / 2] (FP4 packed); block_scale:
 * [n_tokens, hidden / 32] (MX) or [n_tokens, hidden / 16] (NVFP4);
 * token_scale: [n_tokens] fp32 (NVFP4 only).  Returns 0, or -1 on a bad
 * argument (hidden must be a multiple of the block size).
 */
int oracle_block_quantize(const double *y, int64_t n_tokens, int64_t hidden, int fmt, uint8_t *q,
                          uint8_t *block_scale, float *token_scale) {
    if (n_tokens < 0 || hidden <= 0 || !y || !q || !block_scale) return -1;
    if (fmt == ORC_NVFP4) {
        if (hidden % 16 || !token_scale) return -1;
        for (int64_t t = 0; t < n_tokens; ++t)
            quantize_nvfp4_row(y + t * hidden, hidden, q + t * (hidden / 2),
                               block_scale + t * (hidden / 16), token_scale + t);
        return 0;
    }
    if ((fmt != ORC_MXFP8 && fmt != ORC_MXFP4) || hidden % 32) return -1;
    const int fp4 = fmt == ORC_MXFP4;
    for (int64_t t = 0; t < n_tokens; ++t)
        quantize_mx_row(y + t * hidden, hidden, fp4, q + t * (fp4 ? hidden / 2 : hidden),
                        block_scale + t * (hidden / 32));
    return 0;
}
