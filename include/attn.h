/*
 * attn.h - C ABI of the GB300 (sm_103a) attention-forward library.
 *
 * The operation is the forward pass of "4.4 Writing GPU Kernels with Triton"
 * (llm-stack-book), Kernel 4 "A Simplified FlashAttention", with the online
 * softmax of "The Online Softmax Recurrence" on the same page: per (batch,
 * head),
 *
 *     O[i, :] = sum_j softmax_j(scale * q_i . k_j) v_j
 *     LSE[i]  = ln sum_j exp(scale * q_i . k_j)            (natural log)
 *
 * with key j > i masked when causal is set (top-left aligned, as torch.tril).
 * The N x N score matrix is never written to memory: key/value tiles are
 * streamed through on-chip memory and each query row keeps a running max, a
 * running sum and an unnormalised accumulator, normalised once at the end.
 * LSE is saved in natural log (the kernel runs in base 2 internally), as the
 * page's "Base consistency" note asks, so a backward pass can rebuild P with a
 * plain exp.
 *
 * Nothing here allocates on behalf of the caller except attn_fwd_host, which
 * stages host buffers through stream-ordered device memory.
 */
#ifndef BOS_ATTN_H
#define BOS_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. Every entry point returns one; 0 means success. */
typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_NULLPTR = 1,            /* a required pointer is NULL */
    ATTN_ERR_BAD_SHAPE = 2,          /* B, H or N < 1, or the sizes overflow the index space */
    ATTN_ERR_UNSUPPORTED_D = 3,      /* d is not a multiple of 8 in [8, 256] ([8, 128] for attn_bwd) */
    ATTN_ERR_BAD_SCALE = 4,          /* scale is NaN or infinite */
    ATTN_ERR_MISALIGNED = 5,         /* q, k, v, o not 16-byte aligned, or lse not 4-byte aligned */
    ATTN_ERR_UNSUPPORTED_DEVICE = 6, /* the current device is not compute capability 10.3 */
    ATTN_ERR_LAUNCH = 7,             /* the kernel launch failed (cudaGetLastError) */
    ATTN_ERR_TIMEOUT = 8,            /* a bounded wait inside the kernel gave up */
    ATTN_ERR_CUDA = 9,               /* another CUDA runtime call failed */
    ATTN_ERR_BAD_ARG = 10,           /* causal not 0/1, or another malformed argument */
    ATTN_ERR_TOO_LARGE = 11,         /* the problem does not fit attn_fwd_host_noalloc's fixed scratch */
    ATTN_ERR_SCHED_BUSY = 12         /* (device status) a forward launch found its work-counter slot held by
                                        another launch still in flight and skipped its work */
} attn_status;

/*
 * attn_fwd - attention forward on device buffers, asynchronous on `stream`.
 *
 *   q, k, v : bf16, contiguous [B, H, N, d] (row i of head (b, h) at element
 *             ((b*H + h)*N + i)*d), device memory, 16-byte aligned. Read only.
 *   o       : bf16, contiguous [B, H, N, d], device memory, 16-byte aligned.
 *             Written, rounded to nearest even from the fp32 accumulator.
 *   lse     : fp32, contiguous [B, H, N], device memory, 4-byte aligned.
 *             Written with the natural-log log-sum-exp of each row.
 *   B, H, N : batch, heads, sequence length; each >= 1. N need not be a
 *             multiple of any tile size: keys past N do not exist and rows past
 *             N are neither read as outputs nor written.
 *   d       : head dimension, a multiple of 8 from 8 to 256. Kernels exist for
 *             64, 128 and 256 columns; any other d runs on the next one up,
 *             the missing columns read as zero by the tensor copies (they add
 *             nothing to q . k or to O) and never written, so no padded copy
 *             of the inputs is made ("Sizing the attention kernel" of "4.4
 *             Writing GPU Kernels with Triton": zero-padding the head dim is
 *             exact). The backward, attn_bwd, takes d up to 128.
 *   scale   : the multiplier of q . k (1/sqrt(d) in the pages; a C ABI has no
 *             default, so the caller passes it). Must be finite.
 *   causal  : 0 or 1. With 1, query i attends to keys 0..i.
 *   stream  : a cudaStream_t (NULL = the legacy default stream).
 *
 * The caller owns every buffer. The call validates all arguments on the host
 * first; on any error it returns a nonzero status and launches nothing and
 * writes nothing. On success the kernel is enqueued on `stream` and the call
 * returns without synchronising. Safe to call from several host threads.
 * May be captured in a CUDA graph (it allocates nothing and only enqueues
 * work on `stream`).
 *
 * Work distribution: each launch draws one of 4096 slots of work counters in a
 * static device array, round-robin, and its CTAs take work units from it. A
 * slot is held by the launch (tagged with the launch's unique grid id) from
 * its first CTA's start until its last CTA's end. A launch that finds its slot
 * still held by another launch in flight (more than 4096 forward launches
 * outstanding at once, or one graph instance, which keeps the slot it drew
 * at capture, replayed on two streams at the same time) does not share that
 * launch's counter: it skips its work, leaves its outputs incomplete and
 * records ATTN_ERR_SCHED_BUSY, which attn_device_status reports.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * attn_fwd_strided - attn_fwd on strided (non-contiguous) q, k, v and o, e.g.
 * the [B, N, H, d] layout a fused projection produces, or rows padded past d.
 * "Sizing the attention kernel" of "4.4 Writing GPU Kernels with Triton"
 * passes every tensor's batch, head, row and column strides to the kernel;
 * here the head dim must be contiguous (stride 1) and the other three are
 * given per tensor.
 *
 *   q_strides, k_strides, v_strides, o_strides : host arrays of 3 element
 *       strides {batch, head, row}; element (b, h, n, c) of q is at
 *       q + b*q_strides[0] + h*q_strides[1] + n*q_strides[2] + c. Each stride
 *       must be a positive multiple of 8 elements (16 bytes, the TMA rule for
 *       global strides) and at most 2^36; the row stride of q, k and v must be
 *       >= d; o must not map two elements to one address.
 *   lse : fp32 [B, H, N], contiguous, as attn_fwd.
 *   other arguments as attn_fwd (pointers 16-byte aligned, d a multiple of 8
 *   up to 256).
 *
 * Returns the attn_fwd codes; ATTN_ERR_NULLPTR for a NULL stride array,
 * ATTN_ERR_BAD_ARG for strides that break the rules above. attn_fwd itself is
 * this call with the dense strides {H*N*d, N*d, d}.
 */
int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                     const long long* q_strides, const long long* k_strides, const long long* v_strides,
                     const long long* o_strides, float scale, int causal, void* stream);

/* Element types of q, k, v and o for attn_fwd_ex. */
typedef enum attn_dtype {
    ATTN_DTYPE_BF16 = 0,   /* bfloat16: the type of attn_fwd */
    ATTN_DTYPE_F16 = 1     /* IEEE half: the pages' examples call the kernel on fp16 tensors */
} attn_dtype;

/*
 * attn_fwd_ex - attn_fwd for either element type, with optional strides.
 * dtype is ATTN_DTYPE_BF16 or ATTN_DTYPE_F16. q, k, v and o share it, and P
 * enters the second product in it as well; accumulation is fp32 and lse is
 * fp32 either way. Each *_strides is a host array of 3 element strides as in
 * attn_fwd_strided, or NULL for a dense [B, H, N, d] tensor. Returns the
 * attn_fwd_strided codes, and ATTN_ERR_BAD_ARG for an unknown dtype.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                const long long* q_strides, const long long* k_strides, const long long* v_strides,
                const long long* o_strides, float scale, int causal, int dtype, void* stream);

/*
 * attn_fwd_host - the same operation on HOST buffers, end to end.
 *
 *   q_h, k_h, v_h : bf16 host arrays, contiguous [B, H, N, d] (pinned memory
 *                   gives full copy bandwidth; pageable memory also works).
 *   o_h           : bf16 host array [B, H, N, d], written.
 *   lse_h         : fp32 host array [B, H, N], written.
 *   other arguments as for attn_fwd.
 *
 * Stages the arrays through device memory taken from a library-owned,
 * stream-ordered memory pool (the pool keeps its memory between calls, up to
 * the largest problem seen, until the process exits). Large problems are cut
 * into chunks of whole heads whose host-to-device copies, kernels and
 * device-to-host copies overlap on internal streams ordered after `stream`.
 * Synchronises `stream` before returning, so the host arrays are ready when it
 * returns ATTN_OK. Calls for the same device are serialised internally. Host
 * pointers need no particular alignment.
 */
int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                  int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * attn_fwd_host_noalloc - attn_fwd_host for callers that cannot allocate.
 *
 * The pages have no counterpart to this call. attn_fwd_host stages the host
 * arrays through device memory it allocates (from a memory pool) on every
 * call; some callers cannot allocate at that point (another framework's
 * caching allocator owns the device memory, or the thread must not take the
 * implicit synchronisation an allocation can bring). This entry point
 * computes the same result, byte for byte, with no cudaMalloc,
 * cudaMallocAsync or cudaFree: Q, K, V, O and LSE are staged through one
 * fixed device array of ATTN_NOALLOC_SCRATCH_BYTES.
 *
 *   arguments as for attn_fwd_host (host arrays owned by the caller; d a
 *   multiple of 8 from 8 to 256; the same status codes, checked in the same
 *   order).
 *
 * Limit: 4 * round_up(B*H*N*d*2, 256) + round_up(B*H*N*4, 256) bytes must fit
 * in ATTN_NOALLOC_SCRATCH_BYTES (e.g. B*H*N*d up to about 8M elements);
 * larger problems return ATTN_ERR_TOO_LARGE before anything is copied.
 * The array belongs to the library's module: a device holds it from when that
 * module is loaded on it until the process exits. Under CUDA's default lazy
 * loading that is this call's first use on the device; under
 * CUDA_MODULE_LOADING=EAGER it is the creation of the device's context.
 * The first call on a device also looks up the array's device address (with
 * that device current) and keeps it; make that first call before any stream
 * capture begins.
 * Every call shares the one array: calls whose work overlaps on the GPU (on
 * different streams, or from different host threads) race and must be
 * serialised by the caller. Nothing in the array needs clearing between calls:
 * each call copies in every byte the kernel reads. Synchronises `stream`
 * before returning, like attn_fwd_host.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u << 20)
int attn_fwd_host_noalloc(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                          int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * attn_device_status - failures that only the kernel can see.
 *
 * Every wait inside the kernel is bounded in wall time. A wait that runs out
 * records ATTN_ERR_TIMEOUT in a device-wide status word and the kernel returns
 * early (its outputs are then incomplete) after draining its own copies and
 * MMAs, so the CUDA context stays usable. This call synchronises `stream`,
 * returns that word (ATTN_OK if nothing failed since the last call) and clears
 * it. The word is shared by all launches on the current device.
 */
int attn_device_status(void* stream);

/*
 * attn_set_wait_limit_ns - wall-time limit of each wait inside the kernel, in
 * nanoseconds, for launches enqueued after the call (0 restores the default,
 * 2 s). Process-wide. Intended for tests of the failure path.
 */
int attn_set_wait_limit_ns(unsigned long long ns);

/*
 * attn_set_test_stall - test hook for the failure path. While `on` is nonzero,
 * every attn_fwd launch's MMA-issuing threads, and the S/dV-issuing thread of
 * every attn_bwd launch, first wait on a barrier that nothing signals; the wait runs out after the wait limit, the kernel drains and
 * returns, and attn_device_status reports ATTN_ERR_TIMEOUT. No fault, trap or
 * hang is involved. Process-wide; off by default.
 */
int attn_set_test_stall(int on);

/*
 * attn_set_test_sched_busy - test hook for the work-counter guard. While `on`
 * is nonzero, each forward launch's counter slot is marked as held by another
 * launch (a copy on `stream` before the launch; the mark is cleared by a copy
 * after it), so the launch skips its work and attn_device_status reports
 * ATTN_ERR_SCHED_BUSY. Process-wide; off by default.
 */
int attn_set_test_sched_busy(int on);

/* Human-readable text for a status code; never NULL, static storage. */
const char* attn_status_string(int status);

/* Version of this ABI (incremented on any incompatible change). */
int attn_abi_version(void);

/*
 * Backward pass of attn_fwd: Kernel 5 "FlashAttention Backward" of "4.4 Writing
 * GPU Kernels with Triton" (llm-stack-book). With P = exp(scale * q k^T - LSE)
 * rebuilt from the forward's natural-log LSE, D = rowsum(dO * O) and
 * dS = P * (dO v^T - D) * scale:
 *
 *     dq = dS k,   dk = dS^T q,   dv = P^T dO.
 *
 * A gradient g on the LSE output (dL/dLSE) may be passed as dlse; since the
 * derivative of LSE_i in the score S_ij is P_ij, it enters as D_i - g_i.
 *
 *   q, k, v, o, dout : bf16, contiguous [B, H, N, d], device memory, 16-byte
 *                      aligned; o and lse are attn_fwd's outputs for the same
 *                      q, k, v, scale and causal; dout is dL/dO.
 *   lse              : fp32 [B, H, N], device memory, 4-byte aligned.
 *   dlse             : fp32 [B, H, N] gradient on lse, device memory, 4-byte
 *                      aligned; NULL when the loss does not depend on lse.
 *   dq, dk, dv       : bf16 [B, H, N, d] outputs, 16-byte aligned.
 *   workspace        : device memory of workspace_bytes >=
 *                      attn_bwd_workspace_bytes(B, H, N, d), 256-byte aligned:
 *                      the fp32 dq accumulator (every key block adds its part
 *                      with bulk tensor reductions) and the fp32 row sums D.
 *                      Owned by the caller; nothing is allocated.
 *   B, H, N, d, scale, causal, stream: as attn_fwd, with d up to 128. Head
 *                      dims above 128 are not supported, by design: one CTA
 *                      per key block accumulates dK and dV (fp32, d columns
 *                      each) in tensor memory, and at d = 256 those two alone
 *                      take all 512 columns an SM has, before the columns of
 *                      S^T, dP^T and dQ; ATTN_ERR_UNSUPPORTED_D is returned.
 *
 * Asynchronous on stream. Returns the attn_fwd validation codes, or
 * ATTN_ERR_BAD_ARG when the workspace is smaller than needed; on an error
 * nothing is launched or written.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             const float* dlse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
             float scale, int causal, void* stream);

/*
 * attn_bwd_ex - attn_bwd for either element type: dtype is ATTN_DTYPE_BF16 or
 * ATTN_DTYPE_F16, shared by q, k, v, o, dout, dq, dk and dv (lse, dlse and the
 * workspace stay fp32). Returns the attn_bwd codes, and ATTN_ERR_BAD_ARG for
 * an unknown dtype.
 */
int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                const float* dlse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                int H, int N, int d, float scale, int causal, int dtype, void* stream);

/* Workspace bytes attn_bwd needs for these sizes (0 if B, H, N or d are out of range). */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

#ifdef __cplusplus
}
#endif

#endif /* BOS_ATTN_H */
