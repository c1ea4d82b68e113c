/*
 * Attention-forward oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's
 * CPU-baseline leg may load or call this file. The product path (the CUDA
 * library) shares no code, header, table or helper with it, and never falls
 * back to it.
 *
 * What it computes is the plain definition that the blocked online softmax
 * reaches exactly (up to rounding order):
 *
 *     O   = softmax(scale * Q K^T  [causal: key j > query i masked]) V
 *     LSE = natural-log log-sum-exp of each row of scale * Q K^T
 *
 * per (batch, head), following "4.4 Writing GPU Kernels with Triton"
 * (llm-stack-book), Kernel 4 "A Simplified FlashAttention": the kernel's
 * docstring says the streamed result equals a full softmax-then-matmul, and its
 * self-check builds exactly that reference (scores, tril mask, softmax, @ V).
 * The softmax itself is the three-pass stable softmax of Kernel 2 "Fused
 * Softmax" on the same page: pass 1 row max, pass 2 sum of exp(x - max),
 * pass 3 divide.
 *
 * Every score row is materialised in full (length N, fp64), as the definition
 * reads. There is no blocking, no fusion and no reordering beyond that.
 *
 * Inputs are bf16 bit patterns (uint16) widened exactly to double, or doubles.
 * Causal masking is top-left aligned: query i sees keys 0..i (torch.tril).
 * A key index >= N does not exist; a row index >= N is not an output.
 *
 * Parity pins for every function here live in the CPU test suite (closed
 * forms, invariants, brute force, the worked exercise on the page).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE fp32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Three-pass stable softmax of one row x[0..n-1] into p[0..n-1]
 * ("4.4 Writing GPU Kernels with Triton", Kernel 2 "Fused Softmax":
 * max, subtract and exponentiate, sum, divide). Entries equal to -inf are
 * masked and get probability 0. Returns the natural-log log-sum-exp,
 * max + ln(sum); -inf if every entry is masked (then p is all zero).
 */
double oracle_softmax_row_f64(const double* x, int64_t n, double* p)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)            /* pass 1: row max */
        if (x[j] > m) m = x[j];
    if (m == -INFINITY) {                       /* no visible entry */
        for (int64_t j = 0; j < n; ++j) p[j] = 0.0;
        return -INFINITY;
    }
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {           /* pass 2: sum of exp(x - max) */
        double e = (x[j] == -INFINITY) ? 0.0 : exp(x[j] - m);
        p[j] = e;
        z += e;
    }
    for (int64_t j = 0; j < n; ++j)             /* pass 3: divide */
        p[j] = p[j] / z;
    return m + log(z);
}

/*
 * One query row of attention for one head.
 *   q    : d values of query row i
 *   k, v : N x d, row-major (key j at k + j*d)
 *   s, p : scratch of length N (the materialised score row and its softmax)
 *   o    : d outputs; returns LSE (natural log).
 */
static double attn_row(const double* q, const double* k, const double* v,
                       int64_t N, int d, double scale, int causal, int64_t i,
                       double* s, double* p, double* o)
{
    for (int64_t j = 0; j < N; ++j) {
        if (causal && j > i) { s[j] = -INFINITY; continue; }
        double dot = 0.0;
        for (int t = 0; t < d; ++t) dot += q[t] * k[j * (int64_t)d + t];
        s[j] = scale * dot;
    }
    double lse = oracle_softmax_row_f64(s, N, p);
    for (int t = 0; t < d; ++t) o[t] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (p[j] == 0.0) continue;
        const double* vj = v + j * (int64_t)d;
        for (int t = 0; t < d; ++t) o[t] += p[j] * vj[t];
    }
    return lse;
}

/*
 * Shared driver for both input precisions. Rows are flattened ids
 * r = bh * N + i with bh = b * H + h. With rows == NULL every row of every
 * head is computed and o / lse are [B*H*N*d] / [B*H*N]; otherwise o / lse are
 * [nrows*d] / [nrows] in the order given. Runs of rows from the same head
 * share one widening of that head's K and V, so pass rows grouped by head.
 */
typedef void (*widen_fn)(const void* src, int64_t off, int64_t n, double* dst);

static void widen_bf16(const void* src, int64_t off, int64_t n, double* dst)
{
    const uint16_t* s = (const uint16_t*)src + off;
    for (int64_t t = 0; t < n; ++t) dst[t] = bf16_bits_to_double(s[t]);
}

static void widen_f64(const void* src, int64_t off, int64_t n, double* dst)
{
    memcpy(dst, (const double*)src + off, (size_t)n * sizeof(double));
}

static int run_rows(widen_fn widen, const void* q, const void* k, const void* v,
                    int B, int H, int64_t N, int d, double scale, int causal,
                    const int64_t* rows, int64_t nrows, double* o, double* lse,
                    int nthreads)
{
    if (B < 1 || H < 1 || N < 1 || d < 1 || !q || !k || !v || !o || !lse) return 1;
    const int64_t total = (int64_t)B * H * N;
    if (!rows) nrows = total;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    double* kh = (double*)malloc((size_t)N * d * sizeof(double));
    double* vh = (double*)malloc((size_t)N * d * sizeof(double));
    if (!kh || !vh) { free(kh); free(vh); return 2; }
    int err = 0;

    int64_t start = 0;
    while (start < nrows) {
        int64_t r0 = rows ? rows[start] : start;
        if (r0 < 0 || r0 >= total) { err = 3; break; }
        int64_t bh = r0 / N;
        int64_t end = start + 1;                    /* same-head run [start, end) */
        while (end < nrows) {
            int64_t r = rows ? rows[end] : end;
            if (r < 0 || r >= total) { err = 3; break; }
            if (r / N != bh) break;
            ++end;
        }
        if (err) break;
        widen(k, bh * N * d, N * d, kh);
        widen(v, bh * N * d, N * d, vh);
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
        {
            double* s = (double*)malloc((size_t)N * sizeof(double));
            double* p = (double*)malloc((size_t)N * sizeof(double));
            double* qr = (double*)malloc((size_t)d * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
            for (int64_t idx = start; idx < end; ++idx) {
                int64_t r = rows ? rows[idx] : idx;
                int64_t i = r - bh * N;
                widen(q, r * d, d, qr);
                lse[idx] = attn_row(qr, kh, vh, N, d, scale, causal, i, s, p,
                                    o + idx * (int64_t)d);
            }
            free(s); free(p); free(qr);
        }
        start = end;
    }
    free(kh); free(vh);
    return err;
}

/* bf16 inputs (bit patterns), contiguous [B,H,N,d]. Returns 0 on success. */
int oracle_attn_fwd_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int B, int H, int64_t N, int d, double scale, int causal,
                         const int64_t* rows, int64_t nrows,
                         double* o, double* lse, int nthreads)
{
    return run_rows(widen_bf16, q, k, v, B, H, N, d, scale, causal,
                    rows, nrows, o, lse, nthreads);
}

/* fp64 inputs, contiguous [B,H,N,d]; same contract as the bf16 entry. */
int oracle_attn_fwd_f64(const double* q, const double* k, const double* v,
                        int B, int H, int64_t N, int d, double scale, int causal,
                        const int64_t* rows, int64_t nrows,
                        double* o, double* lse, int nthreads)
{
    return run_rows(widen_f64, q, k, v, B, H, N, d, scale, causal,
                    rows, nrows, o, lse, nthreads);
}

/* Threads the oracle would use with nthreads <= 0. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
