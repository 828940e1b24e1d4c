/*
 * hgemm_oracle.c -- the CPU oracle for the half-precision GEMM C = A.B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it is used by tests/, by the smoke check and by the bench's
 * cpu_baseline leg.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, nothing more):
 *
 *   Cref[b][i][j] = sum_{k=0}^{K-1} dec(A_b[i][k]) * dec(B_b[k][j])
 *   Den [b][i][j] = sum_{k=0}^{K-1} |dec(A_b[i][k])| * |dec(B_b[k][j])|
 *
 * in IEEE binary64, k ascending.  The definition of the matrix product with
 * A (M x K) and B (K x N) both row-major is stated in
 *   "hgemm_mma_m16n8k16_mma2x4_warp4x4_kernel" (yuyanqi.com), section 1.1,
 * and the contraction with wide accumulation in
 *   "tensor-cores-cutlass-and-cute" (arganzheng.life), section 四.1
 * (fp32 accumulation there; the oracle accumulates in fp64 so that it is a
 * bound-checked reference for any fp32 summation order).
 *
 * Den is the error normaliser: any summation order of the same products in
 * fp32 differs from Cref by at most about K * 2^-24 * Den.
 *
 * Element (i,k) of A_b lives at A[b*strideA + i*lda + k]; (k,j) of B_b at
 * B[b*strideB + k*ldb + j].  Inputs are raw 16-bit patterns; `dtype_in` says
 * how to read them: 0 = IEEE binary16 (fp16), 1 = bfloat16, 2 = E4M3 and
 * 3 = E5M2 (8-bit patterns in the low byte: the 8-bit inputs of the
 * tensor-core path, "tensor-cores-cutlass-and-cute" section 二.1, its table
 * of input types: FP8 e4m3 with twice the K per instruction).
 *
 * Parity pins (tests/test_oracle_pins.py): the single-warp worked example of
 * the "post_1787550000" mma.sync layout experiment (section 6.1: A[i][k] = i,
 * B[k][j] = j gives D[i][j] = 16*i*j), exact rational brute force on tiny
 * shapes, identity / one-hot / zero special cases, and the decoders against
 * library decoders over all 65536 patterns.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- decoders ---------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 holds zero and the subnormals (value = frac * 2^-24),
 * exponent 31 holds infinities (frac 0) and NaNs. */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE 754 binary32 -- 1 sign bit,
 * 8 exponent bits (bias 127), 7 fraction bits.  Exponent 0 holds zero and
 * subnormals (frac * 2^-133), exponent 255 holds infinities and NaNs. */
double oracle_decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* 8-bit floating point, E4M3 (the "fn" variant): 1 sign bit, 4 exponent
 * bits (bias 7), 3 fraction bits.  Exponent 0 holds zero and the subnormals
 * (frac * 2^-9); there are no infinities, and only S.1111.111 is NaN, so the
 * largest value is 1.75 * 2^8 = 448.  Patterns above 0xff are not E4M3. */
double oracle_decode_e4m3(uint16_t h) {
    if (h > 0xff) return NAN;
    int sign = (h >> 7) & 1;
    int e = (h >> 3) & 0xf;
    int f = h & 0x7;
    double v;
    if (e == 0xf && f == 0x7)
        return NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp(1.0 + f / 8.0, e - 7);
    return sign ? -v : v;
}

/* 8-bit floating point, E5M2: 1 sign bit, 5 exponent bits (bias 15), 2
 * fraction bits, laid out like binary16's upper byte: exponent 0 holds zero
 * and the subnormals (frac * 2^-16), exponent 31 infinities (frac 0) and
 * NaNs; the largest finite value is 1.75 * 2^15 = 57344. */
double oracle_decode_e5m2(uint16_t h) {
    if (h > 0xff) return NAN;
    int sign = (h >> 7) & 1;
    int e = (h >> 2) & 0x1f;
    int f = h & 0x3;
    double v;
    if (e == 0x1f)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -16);
    else
        v = ldexp(1.0 + f / 4.0, e - 15);
    return sign ? -v : v;
}

/* dtype_in: 0 fp16, 1 bf16, 2 E4M3, 3 E5M2 (8-bit patterns stored in the
 * low byte of each 16-bit element). */
static double decode(uint16_t h, int dtype_in) {
    switch (dtype_in) {
        case 0: return oracle_decode_f16(h);
        case 1: return oracle_decode_bf16(h);
        case 2: return oracle_decode_e4m3(h);
        default: return oracle_decode_e5m2(h);
    }
}

/* ---- full product ------------------------------------------------------ */

typedef struct {
    const uint16_t *A, *B;
    const double *table; /* decode(h) for all 65536 patterns */
    int64_t M, N, K, lda, ldb, sA, sB, batch;
    double *Cref, *Den; /* [batch][M][N], dense */
    int64_t row_begin, row_end; /* rows over the flattened (b, i) range */
} job_t;

static void *gemm_rows(void *arg) {
    job_t *J = (job_t *)arg;
    for (int64_t r = J->row_begin; r < J->row_end; ++r) {
        int64_t b = r / J->M, i = r % J->M;
        double *c = J->Cref + r * J->N;
        double *d = J->Den + r * J->N;
        for (int64_t j = 0; j < J->N; ++j) { c[j] = 0.0; d[j] = 0.0; }
        const uint16_t *arow = J->A + b * J->sA + i * J->lda;
        const uint16_t *Bb = J->B + b * J->sB;
        for (int64_t k = 0; k < J->K; ++k) {
            double a = J->table[arow[k]];
            double aa = fabs(a);
            const uint16_t *brow = Bb + k * J->ldb;
            for (int64_t j = 0; j < J->N; ++j) {
                double bv = J->table[brow[j]];
                c[j] += a * bv;
                d[j] += aa * fabs(bv);
            }
        }
    }
    return NULL;
}

static double *make_table(int dtype_in) {
    double *t = (double *)malloc(65536 * sizeof(double));
    if (!t) return NULL;
    for (int h = 0; h < 65536; ++h) t[h] = decode((uint16_t)h, dtype_in);
    return t;
}

/* Full product.  Returns 0 on success, -1 on bad arguments or no memory.
 * `threads` worker threads split the (b, i) rows; each row's sums run in
 * k order inside one thread, so the result does not depend on `threads`. */
int oracle_gemm(const uint16_t *A, const uint16_t *B, int dtype_in,
                int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                int64_t batch, int64_t strideA, int64_t strideB,
                double *Cref, double *Den, int threads) {
    if (M < 0 || N < 0 || K < 0 || batch < 1 || (dtype_in < 0 || dtype_in > 3))
        return -1;
    if (threads < 1) threads = 1;
    double *table = make_table(dtype_in);
    if (!table) return -1;
    int64_t rows = batch * M;
    if (threads > rows && rows > 0) threads = (int)rows;
    job_t *jobs = (job_t *)calloc((size_t)threads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tid) { free(table); free(jobs); free(tid); return -1; }
    for (int t = 0; t < threads; ++t) {
        job_t *J = &jobs[t];
        J->A = A; J->B = B; J->table = table;
        J->M = M; J->N = N; J->K = K; J->lda = lda; J->ldb = ldb;
        J->sA = strideA; J->sB = strideB; J->batch = batch;
        J->Cref = Cref; J->Den = Den;
        J->row_begin = rows * t / threads;
        J->row_end = rows * (t + 1) / threads;
    }
    int rc = 0;
    int started = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[t], NULL, gemm_rows, &jobs[t]) != 0) { rc = -1; break; }
        started = t;
    }
    if (threads > 0) gemm_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    if (rc != 0) { /* a thread could not start: finish its rows here */
        for (int t = started + 1; t < threads; ++t) gemm_rows(&jobs[t]);
        rc = 0;
    }
    free(jobs); free(tid); free(table);
    return rc;
}

/* ---- sampled entries --------------------------------------------------- */

/* The same definition for a list of n entries (b[e], i[e], j[e]): used to
 * check products too large to compute whole on the CPU. */
int oracle_gemm_entries(const uint16_t *A, const uint16_t *B, int dtype_in,
                        int64_t K, int64_t lda, int64_t ldb,
                        int64_t strideA, int64_t strideB, int64_t n,
                        const int64_t *eb, const int64_t *ei, const int64_t *ej,
                        double *Cref, double *Den) {
    if (K < 0 || n < 0 || (dtype_in < 0 || dtype_in > 3)) return -1;
    for (int64_t e = 0; e < n; ++e) {
        const uint16_t *arow = A + eb[e] * strideA + ei[e] * lda;
        const uint16_t *bcol = B + eb[e] * strideB + ej[e];
        double c = 0.0, d = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = decode(arow[k], dtype_in);
            double bv = decode(bcol[k * ldb], dtype_in);
            c += a * bv;
            d += fabs(a) * fabs(bv);
        }
        Cref[e] = c;
        Den[e] = d;
    }
    return 0;
}

/* Decodes n raw 16-bit patterns (used to read the GPU's fp16/bf16 output
 * with the oracle's own decoder). */
void oracle_decode_array(const uint16_t *h, int dtype, int64_t n, double *out) {
    for (int64_t e = 0; e < n; ++e) out[e] = decode(h[e], dtype);
}

/* ---- attention forward ------------------------------------------------- */

/*
 * The attention block the GEMM pages build toward ("post_1787550000",
 * sections 1-2: the FlashAttention kernel's two products S = Q K^T and
 * O = P V moved to tensor cores, with the softmax between them; the causal
 * mask is named there too).  Its plain definition, per (bh, i):
 *
 *   s_j   = scale * sum_{c<D} q_i[c] * k_j[c]          for allowed j
 *   p_j   = exp(s_j - max_j s_j)                       (softmax, shifted)
 *   l     = sum_j p_j
 *   O[c]  = sum_j p_j * v_j[c] / l
 *   Den[c]= sum_j p_j * |v_j[c]| / l                   (error normaliser)
 *   lse   = max_j s_j + log(l)
 *   sden  = max_j scale * sum_c |q_i[c]| * |k_j[c]|    (bound on |s_j|'s sum)
 *
 * all in IEEE binary64, j and c ascending.  Allowed keys: j < SKV and, when
 * `causal`, j <= i + (SKV - SQ) (the last query row sees every key).  A row
 * with no allowed key has O = Den = 0, lse = -inf, sden = 0.
 *
 * Layout: Q [BH][SQ][D], K and V [BH][SKV][D], row-major and dense; 16-bit
 * patterns read with `dtype_in` as above.  Rows (rb[r], ri[r]) for r < nrows
 * are computed into O[r][D], Den[r][D], lse[r], sden[r].
 */
typedef struct {
    const uint16_t *Q, *K, *V;
    const double *table;
    int64_t SQ, SKV, D;
    double scale;
    int causal;
    const int64_t *rb, *ri;
    double *O, *Den, *lse, *sden;
    double *s; /* SKV scores of the current row */
    int64_t row_begin, row_end;
} attn_job_t;

static void *attention_rows(void *arg) {
    attn_job_t *J = (attn_job_t *)arg;
    const int64_t D = J->D;
    for (int64_t r = J->row_begin; r < J->row_end; ++r) {
        const int64_t b = J->rb[r], i = J->ri[r];
        const uint16_t *q = J->Q + (b * J->SQ + i) * D;
        const uint16_t *Kb = J->K + b * J->SKV * D;
        const uint16_t *Vb = J->V + b * J->SKV * D;
        double *o = J->O + r * D;
        double *den = J->Den + r * D;
        for (int64_t c = 0; c < D; ++c) { o[c] = 0.0; den[c] = 0.0; }
        int64_t nkeys = J->SKV;
        if (J->causal) {
            int64_t last = i + (J->SKV - J->SQ); /* last allowed key */
            nkeys = last + 1 < 0 ? 0 : (last + 1 < J->SKV ? last + 1 : J->SKV);
        }
        if (nkeys == 0) { J->lse[r] = -INFINITY; J->sden[r] = 0.0; continue; }
        double m = -INFINITY, sd = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            const uint16_t *k = Kb + j * D;
            double acc = 0.0, mag = 0.0;
            for (int64_t c = 0; c < D; ++c) {
                double qv = J->table[q[c]], kv = J->table[k[c]];
                acc += qv * kv;
                mag += fabs(qv) * fabs(kv);
            }
            J->s[j] = J->scale * acc;
            if (J->s[j] > m) m = J->s[j];
            if (fabs(J->scale) * mag > sd) sd = fabs(J->scale) * mag;
        }
        double l = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            double p = exp(J->s[j] - m);
            l += p;
            const uint16_t *v = Vb + j * D;
            for (int64_t c = 0; c < D; ++c) {
                double vv = J->table[v[c]];
                o[c] += p * vv;
                den[c] += p * fabs(vv);
            }
        }
        for (int64_t c = 0; c < D; ++c) { o[c] /= l; den[c] /= l; }
        J->lse[r] = m + log(l);
        J->sden[r] = sd;
    }
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments or no memory.  Rows are split
 * over `threads` worker threads; each row is computed inside one thread, so
 * the result does not depend on `threads`. */
int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype_in,
                     int64_t SQ, int64_t SKV, int64_t D, double scale, int causal,
                     int64_t nrows, const int64_t *rb, const int64_t *ri,
                     double *O, double *Den, double *lse, double *sden, int threads) {
    if (SQ < 0 || SKV < 0 || D < 0 || nrows < 0 || dtype_in < 0 || dtype_in > 3) return -1;
    if (threads < 1) threads = 1;
    if (threads > nrows && nrows > 0) threads = (int)nrows;
    double *table = make_table(dtype_in);
    attn_job_t *jobs = (attn_job_t *)calloc((size_t)threads, sizeof(attn_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    double *scratch = (double *)malloc((size_t)threads * (size_t)(SKV > 0 ? SKV : 1) * sizeof(double));
    if (!table || !jobs || !tid || !scratch) {
        free(table); free(jobs); free(tid); free(scratch);
        return -1;
    }
    for (int t = 0; t < threads; ++t) {
        attn_job_t *J = &jobs[t];
        J->Q = Q; J->K = K; J->V = V; J->table = table;
        J->SQ = SQ; J->SKV = SKV; J->D = D; J->scale = scale; J->causal = causal;
        J->rb = rb; J->ri = ri;
        J->O = O; J->Den = Den; J->lse = lse; J->sden = sden;
        J->s = scratch + (size_t)t * (size_t)(SKV > 0 ? SKV : 1);
        J->row_begin = nrows * t / threads;
        J->row_end = nrows * (t + 1) / threads;
    }
    int started = 0, rc = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[t], NULL, attention_rows, &jobs[t]) != 0) { rc = -1; break; }
        started = t;
    }
    attention_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    if (rc != 0) {
        for (int t = started + 1; t < threads; ++t) attention_rows(&jobs[t]);
    }
    free(table); free(jobs); free(tid); free(scratch);
    return 0;
}
