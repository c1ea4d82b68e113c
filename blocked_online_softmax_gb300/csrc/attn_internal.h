// Internal interface between the C-ABI host code and the device kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace bos {

struct AttnParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int B, H, N, d;
    float scale;
    int causal;
    int f16 = 0;   // q, k, v, o are fp16 (else bf16)
    // element strides of the batch, head and row dims of q, k, v, o (the head
    // dim is contiguous); set_contiguous fills the dense [B, H, N, d] ones
    long long sq[3], sk[3], sv[3], so[3];
};

inline void set_strides(long long (&s)[3], long long sb, long long sh, long long sn) {
    s[0] = sb;
    s[1] = sh;
    s[2] = sn;
}

inline void set_contiguous(AttnParams& p) {
    const long long sn = p.d, sh = (long long)p.N * p.d, sb = (long long)p.H * p.N * p.d;
    set_strides(p.sq, sb, sh, sn);
    set_strides(p.sk, sb, sh, sn);
    set_strides(p.sv, sb, sh, sn);
    set_strides(p.so, sb, sh, sn);
}

// Enqueues the forward kernel for validated arguments on `stream` (device `dev`
// is current). Returns an attn_status code.
int launch_attn_fwd(const AttnParams& p, cudaStream_t stream, int dev);

// attn_fwd_host's body: `p` holds HOST pointers (validated); stages them through
// device memory, overlapping copies and compute over chunks of heads, and
// synchronises `stream` before returning. Returns an attn_status code.
int host_forward(const AttnParams& p, cudaStream_t stream, int dev);

// Wall-time limit of every wait inside the kernel (0 restores the default).
void set_wait_limit_ns(uint64_t ns);

// Test hook: launches enqueued while on make the MMA thread wait on a barrier
// that nothing signals, so the bounded wait expires and the abort path runs.
void set_test_stall(int on);

// Test hook: launches enqueued while on find their work-counter slot held by
// another launch (a foreign tag is written into it before the launch and
// cleared after), so they take no units and record ATTN_ERR_SCHED_BUSY.
void set_test_sched_busy(int on);

// Synchronises `stream`, returns the sticky device status (an attn_status) and
// clears it.
int read_and_clear_device_status(cudaStream_t stream);

struct AttnBwdParams {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const void* dout;
    const float* lse;
    const float* dlse;   // optional gradient on lse (may be null)
    void* dq;
    void* dk;
    void* dv;
    void* workspace;     // fp32 dQ accumulator [B,H,N,d], then fp32 D [B,H,N]
    int B, H, N, d;
    float scale;
    int causal;
    int f16 = 0;         // q, k, v, o, dout and the gradients are fp16 (else bf16)
};

// Bytes of workspace attn_bwd needs (each part 256-byte aligned).
size_t attn_bwd_workspace(int B, int H, int N, int d);

// Enqueues the backward pass (preprocess, main kernel, dQ cast) for validated arguments.
int launch_attn_bwd(const AttnBwdParams& p, cudaStream_t stream, int dev);

// Row softmax (softmax_rows_fwd) for validated arguments on `stream`.
int launch_softmax_rows(const float* x, float* y, int rows, int cols, long long x_stride, long long y_stride,
                        cudaStream_t stream, int dev);

}  // namespace bos
