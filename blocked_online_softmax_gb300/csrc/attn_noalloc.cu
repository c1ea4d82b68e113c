// attn_fwd_host_noalloc: the host-buffer entry point without any device
// allocation. The pages have no counterpart; this exists for callers that
// cannot call cudaMalloc or cudaMallocAsync at the point where they need
// attention (for example code running while another framework's caching
// allocator owns the device memory, or latency-critical threads that must not
// take the implicit synchronisation an allocation can bring).
//
// Instead of stream-ordered staging memory, Q, K, V, O and LSE are staged
// through one file-scope device array of ATTN_NOALLOC_SCRATCH_BYTES. The array
// belongs to this translation unit's module: a device holds it from the moment
// that module is loaded on it until the process exits. With CUDA's default
// lazy module loading that is the first call of this entry point on the
// device (the address look-up below loads it); with CUDA_MODULE_LOADING=EAGER
// it is the creation of the device's context, whether or not this entry point
// is ever called.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"

namespace {

constexpr size_t kScratchBytes = (size_t)ATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch per device. In host code the symbol
// itself is only a host-side stand-in, so the address is looked up once per
// device, with that device current, and kept here.
char* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

int scratch_address(int dev, char** out) {
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<char*>(p);
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" int attn_fwd_host_noalloc(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                                     float* lse_h, int B, int H, int N, int d, float scale, int causal,
                                     void* stream_) {
    if (!q_h || !k_h || !v_h || !o_h || !lse_h) return ATTN_ERR_NULLPTR;
    // The same argument rules as attn_fwd_host, in the same order, before any
    // size arithmetic (so no product below can overflow).
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_BAD_SHAPE;
    if ((int64_t)B * H > INT_MAX || (int64_t)B * H * N > ((int64_t)1 << 40)) return ATTN_ERR_BAD_SHAPE;
    if (d < 8 || d > 256 || d % 8 != 0) return ATTN_ERR_UNSUPPORTED_D;
    if (!std::isfinite(scale)) return ATTN_ERR_BAD_SCALE;
    if (causal != 0 && causal != 1) return ATTN_ERR_BAD_ARG;
    // rows <= 2^40 and d <= 256: every byte count below stays under 2^50
    const uint64_t rows = (uint64_t)B * (uint64_t)H * (uint64_t)N;
    const uint64_t tbytes = rows * (uint64_t)d * 2u;         // one bf16 tensor
    const uint64_t lbytes = rows * 4u;                       // fp32 LSE
    if (4 * round256(tbytes) + round256(lbytes) > kScratchBytes) return ATTN_ERR_TOO_LARGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    char* base = nullptr;
    int rc = scratch_address(dev, &base);
    if (rc != ATTN_OK) return rc;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const size_t off_k = round256(tbytes), off_v = off_k + round256(tbytes), off_o = off_v + round256(tbytes),
                 off_l = off_o + round256(tbytes);
    // Nothing in the array needs clearing: every byte the kernel reads (Q, K, V)
    // is copied in by this call first, every byte copied out (O, LSE) is written
    // by the kernel, and rows past N are never touched (the tensor maps stop at N).
    if (cudaMemcpyAsync(base, q_h, tbytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(base + off_k, k_h, tbytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(base + off_v, v_h, tbytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        rc = ATTN_ERR_CUDA;
    if (rc == ATTN_OK)
        rc = attn_fwd(base, base + off_k, base + off_v, base + off_o, reinterpret_cast<float*>(base + off_l), B, H,
                      N, d, scale, causal, stream);
    if (rc == ATTN_OK &&
        (cudaMemcpyAsync(o_h, base + off_o, tbytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
         cudaMemcpyAsync(lse_h, base + off_l, lbytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess))
        rc = ATTN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    if (rc != ATTN_OK) cudaGetLastError();
    return rc;
}
