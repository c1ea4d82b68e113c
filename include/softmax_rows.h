/*
 * softmax_rows.h - C ABI of the fused row softmax (sm_103a), a second,
 * memory-bound workload of the same library.
 *
 * The operation is Kernel 2 "Fused Softmax" of "4.4 Writing GPU Kernels with
 * Triton" (llm-stack-book), also the fused softmax of "Triton"
 * (ai-infra-handbooks): for every row i of an M x N fp32 matrix,
 *
 *     y[i, j] = exp(x[i, j] - m_i) / sum_k exp(x[i, k] - m_i),   m_i = max_k x[i, k]
 *
 * reading each row from memory once and writing it once (the page's
 * "1 read + 1 write"). Rows longer than SOFTMAX_ROWS_ONCHIP_COLS do not fit
 * on chip and take the page's fallback, a loop over tiles with the online
 * softmax: one pass for the running max and sum, one pass to write, so two
 * reads and one write.
 *
 * Status codes are the attn_status values of attn.h.
 */
#ifndef BOS_SOFTMAX_ROWS_H
#define BOS_SOFTMAX_ROWS_H

#ifdef __cplusplus
extern "C" {
#endif

/* Widest row the single-pass kernel keeps in registers. */
#define SOFTMAX_ROWS_ONCHIP_COLS 16384

/*
 * Row softmax of x into y, asynchronous on `stream`.
 *
 *   x, y          : fp32 device memory, 4-byte aligned; y may equal x with the
 *                   same row stride (in place) but must not otherwise overlap it.
 *   rows, cols    : M >= 1 and N >= 1.
 *   x_row_stride,
 *   y_row_stride  : elements between consecutive rows, each >= cols.
 *   stream        : a cudaStream_t (NULL = the legacy default stream).
 *
 * Rows whose elements are all -inf come out as NaN, as exp(-inf - (-inf))
 * is undefined; +inf or NaN inputs give NaN rows. Nothing is allocated.
 * Returns ATTN_OK, or ATTN_ERR_NULLPTR, ATTN_ERR_BAD_SHAPE (rows or cols < 1,
 * a stride < cols, or sizes past the index space), ATTN_ERR_MISALIGNED,
 * ATTN_ERR_UNSUPPORTED_DEVICE, ATTN_ERR_LAUNCH; on an error nothing is launched.
 */
int softmax_rows_fwd(const float* x, float* y, int rows, int cols, long long x_row_stride,
                     long long y_row_stride, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BOS_SOFTMAX_ROWS_H */
