/*
 * dgemm_oracle.c -- the CPU oracle for dense row-major GEMM,
 *
 *     C = alpha * A * B + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library and includes none of its files.
 *
 * What it computes (the plain definition, written out):
 *
 *   ref[i][j] = alpha * sum_{k<K} a[i][k] * b[k][j]  +  beta * c[i][j]
 *   abs[i][j] =         sum_{k<K} |a[i][k]| * |b[k][j]|
 *
 * accumulated in IEEE double over the exact operand values that the GPU path
 * multiplies:
 *   - FP32 operands: the float values themselves;
 *   - TF32 operands: each float first reduced to TF32 (1 sign, 8 exponent,
 *     10 mantissa bits), round-to-nearest-ties-away or truncation;
 *   - FP16 operands: the IEEE binary16 values;
 *   - BF16 operands: the bfloat16 values (the top half of a float);
 *   - TN layout: b[k][j] is read from the store at B[j*ldb + k]; NN: B[k*ldb + j].
 * When beta == 0 the C term is dropped (C is never read), and when
 * alpha == 0 or K == 0 the sum is skipped (A and B are never read).
 *
 * Sources (page title, section):
 *   - "SGEMM CUDA代码学习", section "问题定义与记号": C[M,N] = A[M,K] x B[K,N],
 *     all row-major, A[m][k] at m*K + k; one output element is one
 *     K-long dot product.
 *   - "CUDA GEMM：从基础写法到工程优化", opening definition and
 *     "1. 最基础版本": C = alpha*A*B + beta*C, A is MxK, B is KxN.
 *   - "如何优化一个 CUDA Matmul Kernel ... Worklog", "Kernel 1: Naive 实现":
 *     C = alpha*(A@B) + beta*C, one thread per entry.
 *   - "SGEMM CUDA代码学习", "第 5 步": TF32 is a 19-bit float, 1+8+10.
 *   - "HGEMM SMEM Swizzle 代码学习" and "Warp Specialization HGEMM", section
 *     "6. B 的 RowMajor(K,N) 与 TN 布局": the TN convention, B stored N x K.
 *
 * Readings taken where the pages are silent: accumulation in double; the
 * beta == 0 / alpha == 0 conventions above (the pages always read C); the
 * TF32 rounding mode is a parameter (ties-away by default).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OPERAND_F32 0
#define ORACLE_OPERAND_TF32_NEAREST_AWAY 1
#define ORACLE_OPERAND_TF32_TRUNCATE 2
#define ORACLE_OPERAND_F16 3
#define ORACLE_OPERAND_BF16 4

/* ------------------------------------------------------------------ */
/* Operand value definitions                                           */
/* ------------------------------------------------------------------ */

/* IEEE 754 binary16 -> double, from the format: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits; exponent 0 encodes subnormals f * 2^-24,
 * exponent 31 encodes infinities (f == 0) and NaNs. */
double oracle_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(1024.0 + (double)f, e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double, from the format: 1 sign bit, 8 exponent bits (bias
 * 127, as for float), 7 fraction bits; exponent 0 encodes subnormals
 * f * 2^-133, exponent 255 infinities (f == 0) and NaNs. */
double oracle_bf16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 255;
    int f = h & 127;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(128.0 + (double)f, e - 134); /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Reduce a float to TF32: keep 10 explicit fraction bits.  For a finite
 * nonzero x with 2^e <= |x| < 2^(e+1), the TF32 spacing is q = 2^(e-10);
 * below the smallest normal (2^-126) the spacing stays at 2^-136, as for
 * any subnormal of an 8-bit-exponent format with 10 fraction bits.
 * mode 1: nearest, ties away from zero (C round()); mode 2: toward zero.
 * The result is exact in double; a rounding that carries past the largest
 * finite value gives infinity, as the format would. */
double oracle_tf32_value(float x, int mode)
{
    double d = (double)x;
    if (d == 0.0 || isnan(d) || isinf(d))
        return d;
    int e2;
    frexp(d, &e2);          /* d = f * 2^e2, 0.5 <= |f| < 1  =>  e = e2 - 1 */
    int e = e2 - 1;
    if (e < -126)
        e = -126;
    double q = ldexp(1.0, e - 10);
    double n = d / q;       /* exact: a power-of-two scaling */
    double r = (mode == ORACLE_OPERAND_TF32_TRUNCATE) ? trunc(n) : round(n);
    double v = r * q;
    if (fabs(v) >= ldexp(1.0, 128))
        return d > 0 ? INFINITY : -INFINITY;
    return v;
}

/* Widen one operand matrix into a dense row-major double array.
 * kind: one of the ORACLE_OPERAND_* codes.  src holds rows x cols logical
 * elements; element (r, c) is at src[r*ld + c], or at src[c*ld + r] when
 * trans != 0 (the TN store of B).  dst receives rows*cols doubles. */
void oracle_widen(int kind, const void *src, int64_t rows, int64_t cols,
                  int64_t ld, int trans, double *dst)
{
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            int64_t at = trans ? c * ld + r : r * ld + c;
            double v;
            if (kind == ORACLE_OPERAND_F16)
                v = oracle_f16_value(((const uint16_t *)src)[at]);
            else if (kind == ORACLE_OPERAND_BF16)
                v = oracle_bf16_value(((const uint16_t *)src)[at]);
            else if (kind == ORACLE_OPERAND_F32)
                v = (double)((const float *)src)[at];
            else
                v = oracle_tf32_value(((const float *)src)[at], kind);
            dst[r * cols + c] = v;
        }
    }
}

/* ------------------------------------------------------------------ */
/* The product                                                         */
/* ------------------------------------------------------------------ */

typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const double *A; /* M x K, row-major, dense */
    const double *B; /* K x N, row-major, dense */
    const double *C; /* M x N, row-major, dense; unused when beta == 0 */
    double *ref;
    double *abs;
    /* which outputs: mode 0 = rows list, 1 = column list, 2 = (i, j) list */
    int mode;
    int64_t count;
    const int64_t *idx_i;
    const int64_t *idx_j;
    /* work split */
    int64_t begin, end;
} oracle_job;

/* One full output row i, loop order k then j, double accumulators. */
static void one_row(const oracle_job *p, int64_t i, double *ref, double *abs_)
{
    int64_t N = p->N, K = p->K;
    for (int64_t j = 0; j < N; ++j) {
        ref[j] = 0.0;
        abs_[j] = 0.0;
    }
    if (p->alpha != 0.0) {
        for (int64_t k = 0; k < K; ++k) {
            double a = p->A[i * K + k];
            const double *brow = p->B + k * N;
            for (int64_t j = 0; j < N; ++j) {
                ref[j] += a * brow[j];
                abs_[j] += fabs(a) * fabs(brow[j]);
            }
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        double v = (p->alpha != 0.0 && K > 0) ? p->alpha * ref[j] : 0.0;
        if (p->beta != 0.0)
            v += p->beta * p->C[i * N + j];
        ref[j] = v;
    }
}

/* One output entry (i, j): a K-long dot product. */
static void one_entry(const oracle_job *p, int64_t i, int64_t j, double *ref,
                      double *abs_)
{
    int64_t N = p->N, K = p->K;
    double s = 0.0, t = 0.0;
    if (p->alpha != 0.0) {
        for (int64_t k = 0; k < K; ++k) {
            double a = p->A[i * K + k];
            double b = p->B[k * N + j];
            s += a * b;
            t += fabs(a) * fabs(b);
        }
    }
    double v = (p->alpha != 0.0 && K > 0) ? p->alpha * s : 0.0;
    if (p->beta != 0.0)
        v += p->beta * p->C[i * N + j];
    *ref = v;
    *abs_ = t;
}

static void *worker(void *arg)
{
    const oracle_job *p = (const oracle_job *)arg;
    for (int64_t u = p->begin; u < p->end; ++u) {
        if (p->mode == 0) {
            int64_t i = p->idx_i[u];
            one_row(p, i, p->ref + u * p->N, p->abs + u * p->N);
        } else if (p->mode == 1) {
            int64_t j = p->idx_j[u];
            for (int64_t i = 0; i < p->M; ++i)
                one_entry(p, i, j, p->ref + u * p->M + i, p->abs + u * p->M + i);
        } else {
            one_entry(p, p->idx_i[u], p->idx_j[u], p->ref + u, p->abs + u);
        }
    }
    return NULL;
}

static int run_jobs(oracle_job *proto, int nthreads)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > proto->count)
        nthreads = proto->count > 0 ? (int)proto->count : 1;
    if (nthreads > 256)
        nthreads = 256;
    oracle_job jobs[256];
    pthread_t tids[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].begin = proto->count * t / nthreads;
        jobs[t].end = proto->count * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    /* any job whose thread could not start runs here */
    for (int t = started + 1; t < nthreads; ++t)
        worker(&jobs[t]);
    return nthreads;
}

/* Evaluate reference outputs on dense double operands (from oracle_widen).
 *   mode 0: `count` full rows idx_i[0..count)        -> ref/abs: count x N
 *   mode 1: `count` full columns idx_j[0..count)     -> ref/abs: count x M
 *           (column u stored contiguously: ref[u*M + i])
 *   mode 2: `count` entries (idx_i[u], idx_j[u])     -> ref/abs: count
 * C may be NULL when beta == 0.  Returns the number of threads used. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, double alpha,
                const double *A, const double *B, double beta,
                const double *C, int mode, int64_t count,
                const int64_t *idx_i, const int64_t *idx_j, double *ref,
                double *abs_, int nthreads)
{
    oracle_job p;
    memset(&p, 0, sizeof(p));
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.A = A;
    p.B = B;
    p.C = C;
    p.ref = ref;
    p.abs = abs_;
    p.mode = mode;
    p.count = count;
    p.idx_i = idx_i;
    p.idx_j = idx_j;
    if (count <= 0)
        return 0;
    return run_jobs(&p, nthreads);
}
