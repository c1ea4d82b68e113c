// Host side of the C ABI declared in include/attn.h: argument validation,
// device check, dispatch to the sm_103a kernel, and the host-buffer path.
//
// The operation is the forward pass of "4.4 Writing GPU Kernels with Triton"
// (llm-stack-book), Kernel 4 "A Simplified FlashAttention"; the page's wrapper
// `flash_attention` allocates O like q and an fp32 (B, H, N) LSE and launches
// one program per (query block, batch*head). Here the caller owns all buffers
// and every argument is checked before anything is launched.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "attn.h"
#include "attn_internal.h"
#include "softmax_rows.h"

namespace {

constexpr int kAbiVersion = 1;
constexpr int kMaxDevices = 64;

// Per-device cache of the compute-capability check: 0 unknown, 1 ok, 2 unsupported.
std::atomic<int> g_device_ok[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks that need no GPU. Returns ATTN_OK or the first failing status.
// max_d: the widest head dim the caller's kernels take (forward 256, backward 128).
int validate_host(const void* q, const void* k, const void* v, const void* o, const void* lse,
                  int B, int H, int N, int d, float scale, int causal, bool device_ptrs, int max_d = 256) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULLPTR;
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_BAD_SHAPE;
    const int64_t rows = (int64_t)B * H * N;
    // work units: 256 query rows (d <= 128) or 128 (d > 128)
    const int64_t unit_rows = d > 128 ? 128 : 256;
    const int64_t units = (int64_t)B * H * ((N + unit_rows - 1) / unit_rows);
    if ((int64_t)B * H > INT_MAX || rows > ((int64_t)1 << 40) || units > INT_MAX / 2)
        return ATTN_ERR_BAD_SHAPE;
    // a multiple of 8 (rows of Q, K, V, O must be 16-byte strided for TMA) up to max_d
    if (d < 8 || d > max_d || d % 8 != 0) return ATTN_ERR_UNSUPPORTED_D;
    if (!std::isfinite(scale)) return ATTN_ERR_BAD_SCALE;
    if (causal != 0 && causal != 1) return ATTN_ERR_BAD_ARG;
    if (device_ptrs) {
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
            return ATTN_ERR_MISALIGNED;
        if (!aligned(lse, 4)) return ATTN_ERR_MISALIGNED;
    }
    return ATTN_OK;
}

int check_device(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return ATTN_ERR_CUDA; }
    *dev_out = dev;
    const int known = (dev >= 0 && dev < kMaxDevices) ? g_device_ok[dev].load(std::memory_order_relaxed) : 0;
    if (known != 0) return known == 1 ? ATTN_OK : ATTN_ERR_UNSUPPORTED_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < kMaxDevices) g_device_ok[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
    return ok ? ATTN_OK : ATTN_ERR_UNSUPPORTED_DEVICE;
}

}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int N, int d, float scale, int causal, void* stream) {
    int st = validate_host(q, k, v, o, lse, B, H, N, d, scale, causal, true);
    if (st != ATTN_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != ATTN_OK) return st;
    bos::AttnParams p;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    p.B = B; p.H = H; p.N = N; p.d = d;
    p.scale = scale; p.causal = causal;
    bos::set_contiguous(p);
    return bos::launch_attn_fwd(p, static_cast<cudaStream_t>(stream), dev);
}

namespace {

// Strides (elements) of one [B, H, N, d] operand with a contiguous head dim:
// positive, and 16-byte multiples (the TMA rule for every global stride).
bool strides_ok(const long long* s) {
    for (int i = 0; i < 3; ++i)
        if (s[i] <= 0 || s[i] % 8 != 0 || s[i] > ((long long)1 << 36)) return false;
    return true;
}

// The output must not map two elements to one address: sorted by stride,
// every dim must start past the extent of the ones inside it.
bool non_overlapping(const long long* s, int B, int H, int N, int d) {
    long long st[3] = {s[0], s[1], s[2]}, ext[3] = {B, H, N};
    for (int i = 0; i < 3; ++i)            // ascending stride (3 elements: insertion sort)
        for (int j = i; j > 0 && st[j] < st[j - 1]; --j) {
            long long t = st[j]; st[j] = st[j - 1]; st[j - 1] = t;
            t = ext[j]; ext[j] = ext[j - 1]; ext[j - 1] = t;
        }
    long long span = d;                    // elements covered by the dims inside
    for (int i = 0; i < 3; ++i) {
        if (ext[i] == 1) continue;
        if (st[i] < span) return false;
        span = st[i] * (ext[i] - 1) + span;
    }
    return true;
}

}  // namespace

namespace {

// attn_fwd_strided's body, for either element type (f16: fp16, else bf16).
int fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                const long long* q_strides, const long long* k_strides, const long long* v_strides,
                const long long* o_strides, float scale, int causal, int f16, void* stream) {
    int st = validate_host(q, k, v, o, lse, B, H, N, d, scale, causal, true);
    if (st != ATTN_OK) return st;
    if (!q_strides || !k_strides || !v_strides || !o_strides) return ATTN_ERR_NULLPTR;
    if (!strides_ok(q_strides) || !strides_ok(k_strides) || !strides_ok(v_strides) || !strides_ok(o_strides))
        return ATTN_ERR_BAD_ARG;
    if (q_strides[2] < d || k_strides[2] < d || v_strides[2] < d || !non_overlapping(o_strides, B, H, N, d))
        return ATTN_ERR_BAD_ARG;
    int dev = 0;
    st = check_device(&dev);
    if (st != ATTN_OK) return st;
    bos::AttnParams p;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    p.B = B; p.H = H; p.N = N; p.d = d;
    p.scale = scale; p.causal = causal;
    p.f16 = f16;
    for (int i = 0; i < 3; ++i) {
        p.sq[i] = q_strides[i];
        p.sk[i] = k_strides[i];
        p.sv[i] = v_strides[i];
        p.so[i] = o_strides[i];
    }
    return bos::launch_attn_fwd(p, static_cast<cudaStream_t>(stream), dev);
}

}  // namespace

extern "C" int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int N, int d, const long long* q_strides, const long long* k_strides,
                                const long long* v_strides, const long long* o_strides, float scale, int causal,
                                void* stream) {
    return fwd_strided(q, k, v, o, lse, B, H, N, d, q_strides, k_strides, v_strides, o_strides, scale, causal, 0,
                       stream);
}

extern "C" int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                           int d, const long long* q_strides, const long long* k_strides,
                           const long long* v_strides, const long long* o_strides, float scale, int causal,
                           int dtype, void* stream) {
    if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_F16) return ATTN_ERR_BAD_ARG;
    // a NULL stride array means that tensor is dense [B, H, N, d]
    const long long dense[3] = {(long long)H * N * d, (long long)N * d, (long long)d};
    return fwd_strided(q, k, v, o, lse, B, H, N, d, q_strides ? q_strides : dense, k_strides ? k_strides : dense,
                       v_strides ? v_strides : dense, o_strides ? o_strides : dense, scale, causal,
                       dtype == ATTN_DTYPE_F16 ? 1 : 0, stream);
}

extern "C" int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                             float* lse_h, int B, int H, int N, int d, float scale, int causal,
                             void* stream_) {
    int st = validate_host(q_h, k_h, v_h, o_h, lse_h, B, H, N, d, scale, causal, false);
    if (st != ATTN_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != ATTN_OK) return st;
    bos::AttnParams p;
    p.q = q_h; p.k = k_h; p.v = v_h; p.o = o_h; p.lse = lse_h;
    p.B = B; p.H = H; p.N = N; p.d = d;
    p.scale = scale; p.causal = causal;
    bos::set_contiguous(p);
    return bos::host_forward(p, static_cast<cudaStream_t>(stream_), dev);
}

extern "C" size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
    static const char one = 0;
    if (validate_host(&one, &one, &one, &one, reinterpret_cast<const float*>(&one), B, H, N, d, 1.0f, 0, false,
                      128) != ATTN_OK)
        return 0;
    return bos::attn_bwd_workspace(B, H, N, d);
}

namespace {

// attn_bwd's body, for either element type (f16: fp16, else bf16).
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             const float* dlse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H,
             int N, int d, float scale, int causal, int f16, void* stream) {
    int st = validate_host(q, k, v, dq, lse, B, H, N, d, scale, causal, true, 128);
    if (st != ATTN_OK) return st;
    if (!o || !dout || !dk || !dv || !workspace) return ATTN_ERR_NULLPTR;
    if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(workspace, 256) ||
        !aligned(dlse, 4))
        return ATTN_ERR_MISALIGNED;
    if (workspace_bytes < bos::attn_bwd_workspace(B, H, N, d)) return ATTN_ERR_BAD_ARG;
    int dev = 0;
    st = check_device(&dev);
    if (st != ATTN_OK) return st;
    bos::AttnBwdParams p;
    p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse; p.dlse = dlse;
    p.dq = dq; p.dk = dk; p.dv = dv; p.workspace = workspace;
    p.B = B; p.H = H; p.N = N; p.d = d;
    p.scale = scale; p.causal = causal;
    p.f16 = f16;
    return bos::launch_attn_bwd(p, static_cast<cudaStream_t>(stream), dev);
}

}  // namespace

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, const float* dlse, void* dq, void* dk, void* dv, void* workspace,
                        size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, void* stream) {
    return bwd_impl(q, k, v, o, dout, lse, dlse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
                    0, stream);
}

extern "C" int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                           const float* lse, const float* dlse, void* dq, void* dk, void* dv, void* workspace,
                           size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, int dtype,
                           void* stream) {
    if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_F16) return ATTN_ERR_BAD_ARG;
    return bwd_impl(q, k, v, o, dout, lse, dlse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
                    dtype == ATTN_DTYPE_F16 ? 1 : 0, stream);
}

extern "C" int softmax_rows_fwd(const float* x, float* y, int rows, int cols, long long x_row_stride,
                                long long y_row_stride, void* stream) {
    if (!x || !y) return ATTN_ERR_NULLPTR;
    if (rows < 1 || cols < 1 || x_row_stride < cols || y_row_stride < cols) return ATTN_ERR_BAD_SHAPE;
    if ((long long)rows > (LLONG_MAX / 4) / x_row_stride || (long long)rows > (LLONG_MAX / 4) / y_row_stride)
        return ATTN_ERR_BAD_SHAPE;
    if (!aligned(x, 4) || !aligned(y, 4)) return ATTN_ERR_MISALIGNED;
    int dev = 0;
    const int st = check_device(&dev);
    if (st != ATTN_OK) return st;
    return bos::launch_softmax_rows(x, y, rows, cols, x_row_stride, y_row_stride, static_cast<cudaStream_t>(stream),
                                    dev);
}

extern "C" int attn_device_status(void* stream) {
    int dev = 0;
    const int st = check_device(&dev);
    if (st != ATTN_OK) return st;
    return bos::read_and_clear_device_status(static_cast<cudaStream_t>(stream));
}

extern "C" int attn_set_wait_limit_ns(unsigned long long ns) {
    bos::set_wait_limit_ns((uint64_t)ns);
    return ATTN_OK;
}

extern "C" int attn_set_test_stall(int on) {
    bos::set_test_stall(on);
    return ATTN_OK;
}

extern "C" int attn_set_test_sched_busy(int on) {
    bos::set_test_sched_busy(on);
    return ATTN_OK;
}

extern "C" const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULLPTR: return "a required pointer is NULL";
        case ATTN_ERR_BAD_SHAPE: return "B, H and N must be >= 1 and the sizes must fit the index space";
        case ATTN_ERR_UNSUPPORTED_D:
            return "head dimension d must be a multiple of 8 from 8 to 256 (to 128 for the backward)";
        case ATTN_ERR_BAD_SCALE: return "scale must be finite";
        case ATTN_ERR_MISALIGNED: return "q, k, v, o must be 16-byte aligned and lse 4-byte aligned";
        case ATTN_ERR_UNSUPPORTED_DEVICE: return "the current device is not compute capability 10.3 (sm_103a)";
        case ATTN_ERR_LAUNCH: return "kernel launch failed";
        case ATTN_ERR_TIMEOUT: return "a bounded wait inside the kernel timed out";
        case ATTN_ERR_CUDA: return "a CUDA runtime call failed";
        case ATTN_ERR_BAD_ARG: return "malformed argument (causal must be 0 or 1; strides positive multiples of 8, row stride >= d, output not self-overlapping; workspace large enough)";
        case ATTN_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of attn_fwd_host_noalloc (ATTN_NOALLOC_SCRATCH_BYTES)";
        case ATTN_ERR_SCHED_BUSY:
            return "a launch found its work-counter slot held by another launch in flight (more than 4096 "
                   "forward launches outstanding on the device); it skipped its work units";
        default: return "unknown status";
    }
}

extern "C" int attn_abi_version(void) { return kAbiVersion; }
