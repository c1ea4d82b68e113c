// Fused row softmax for GB300 (sm_103a): y = exp(x - rowmax) / rowsum, fp32.
//
// The operation is Kernel 2 "Fused Softmax" of "4.4 Writing GPU Kernels with
// Triton" (llm-stack-book) and the fused softmax of "Triton"
// (ai-infra-handbooks): each row is read from memory once, its max, its
// exponentials and their sum are formed on chip, and it is written once. The
// work is memory-bound (one exp2 and a few FP32 operations per 8 bytes moved),
// so the design is about streaming: coalesced 16-byte loads and stores, enough
// rows in flight per SM, and no second pass over memory.
//
//  * A row is handled by a group of G threads (one warp for rows up to 1024
//    columns, a 256-thread block up to 16384); each thread keeps up to K
//    four-float chunks of the row in registers, so the row is never re-read.
//    The reductions are warp shuffles, plus one shared-memory step across the
//    block's warps when G = 256. Masked columns load as -inf, which can never
//    be the max and whose exponential is 0 (the page's `other=-inf` trick).
//  * exp(x - m) is taken as exp2((x - m) * log2 e): the difference first, which
//    is exact in fp32 for x near the max (where the result matters), so logits
//    of any size keep full relative accuracy near the top of the row.
//  * Longer rows take the page's fallback ("a loop over tiles with online
//    softmax"): one CTA walks the row in tiles keeping a running max and a
//    running sum rescaled by exp2(m_old - m_new), merges the threads' pairs,
//    then walks the row again to write it: two reads and one write.
//  * Rows are distributed over a grid-stride loop, so any row count works.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "attn.h"
#include "attn_internal.h"
#include "softmax_rows.h"

namespace bos {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int G>
__device__ __forceinline__ float group_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (G > 32) {
        const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
        __syncthreads();                       // red[] may still be read from the previous reduction
        if (lane == 0) red[w] = v;
        __syncthreads();
        v = red[0];
#pragma unroll
        for (int i = 1; i < G / 32; ++i) v = fmaxf(v, red[i]);
    }
    return v;
}

template <int G>
__device__ __forceinline__ float group_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if constexpr (G > 32) {
        const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
        __syncthreads();
        if (lane == 0) red[w] = v;
        __syncthreads();
        v = red[0];
#pragma unroll
        for (int i = 1; i < G / 32; ++i) v += red[i];
    }
    return v;
}

// Single pass: a row of up to 4*G*K columns per group of G threads. Thread t of
// a group owns the four-float chunks t, t+G, t+2G, ... (coalesced across the
// group). kVec: rows start 16-byte aligned and cols % 4 == 0, so chunks are
// float4 loads/stores; otherwise elements are loaded one by one.
template <int G, int K, bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_rows_onchip(const float* __restrict__ x, float* __restrict__ y, int rows, int cols, long long xs,
                    long long ys) {
    constexpr int kGroups = kThreads / G;
    __shared__ float red[kThreads / 32];
    const int g = threadIdx.x / G, t = threadIdx.x % G;
    for (long long r0 = (long long)blockIdx.x * kGroups; r0 < rows; r0 += (long long)gridDim.x * kGroups) {
        const long long row = r0 + g;
        // with G = 256 the whole block is one group and takes part in every row
        // (a block-wide barrier inside the reductions), so the loop bound above
        // is uniform across the block; with G = 32 a warp past the end just idles
        const bool live = row < rows;
        const float* xr = x + (live ? row : 0) * xs;
        float v[4 * K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int c0 = (k * G + t) * 4;
            if (kVec) {
                float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                if (live && c0 < cols) q = *reinterpret_cast<const float4*>(xr + c0);
                v[4 * k] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[4 * k + e] = (live && c0 + e < cols) ? xr[c0 + e] : -INFINITY;
            }
        }
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4 * K; ++i) m = fmaxf(m, v[i]);
        m = group_max<G>(m, red);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4 * K; ++i) {
            v[i] = ex2f((v[i] - m) * kLog2e);       // exp(x - m); -inf columns give 0
            s += v[i];
        }
        s = group_sum<G>(s, red);
        const float inv = 1.f / s;
        if (!live) continue;
        float* yr = y + row * ys;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int c0 = (k * G + t) * 4;
            if (kVec) {
                if (c0 < cols)
                    *reinterpret_cast<float4*>(yr + c0) =
                        make_float4(v[4 * k] * inv, v[4 * k + 1] * inv, v[4 * k + 2] * inv, v[4 * k + 3] * inv);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (c0 + e < cols) yr[c0 + e] = v[4 * k + e] * inv;
            }
        }
    }
}

// Rows too long for registers: the online softmax over tiles of the row, then
// a second walk to write it. One block per row.
__global__ void __launch_bounds__(kThreads)
softmax_rows_online(const float* __restrict__ x, float* __restrict__ y, int rows, int cols, long long xs,
                    long long ys) {
    __shared__ float red_m[kThreads / 32], red_l[kThreads / 32];
    const int t = threadIdx.x, w = t / 32, lane = t % 32;
    for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
        const float* xr = x + row * xs;
        float* yr = y + row * ys;
        // running max m and sum l = sum exp(x - m) of this thread's elements
        float m = -INFINITY, l = 0.f;
        for (int c = t; c < cols; c += kThreads) {
            const float z = xr[c];
            if (z > m) {
                l = l * ex2f((m - z) * kLog2e) + 1.f;   // rescale the old sum to the new max
                m = z;
            } else if (z != -INFINITY) {                // (-inf adds nothing, also while m is still -inf)
                l += ex2f((z - m) * kLog2e);
            }
        }
        // merge (m, l) pairs: l = l_a e^(m_a - m) + l_b e^(m_b - m), m = max(m_a, m_b)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, o), lo = __shfl_xor_sync(0xffffffffu, l, o);
            const float mn = fmaxf(m, mo);
            l = (mn == -INFINITY) ? 0.f : l * ex2f((m - mn) * kLog2e) + lo * ex2f((mo - mn) * kLog2e);
            m = mn;
        }
        __syncthreads();
        if (lane == 0) { red_m[w] = m; red_l[w] = l; }
        __syncthreads();
        m = red_m[0];
        l = red_l[0];
        for (int i = 1; i < kThreads / 32; ++i) {
            const float mn = fmaxf(m, red_m[i]);
            l = (mn == -INFINITY) ? 0.f : l * ex2f((m - mn) * kLog2e) + red_l[i] * ex2f((red_m[i] - mn) * kLog2e);
            m = mn;
        }
        const float inv = 1.f / l;
        for (int c = t; c < cols; c += kThreads) yr[c] = ex2f((xr[c] - m) * kLog2e) * inv;
    }
}

std::atomic<int> g_sms[64];   // SM count per device, shared by host threads

template <int G, int K, bool kVec>
int launch_onchip(const float* x, float* y, int rows, int cols, long long xs, long long ys, cudaStream_t stream,
                  int sms) {
    constexpr int kGroups = kThreads / G;
    long long blocks = ((long long)rows + kGroups - 1) / kGroups;
    const long long cap = (long long)sms * 8;   // grid-stride beyond a few waves
    if (blocks > cap) blocks = cap;
    softmax_rows_onchip<G, K, kVec><<<(unsigned)blocks, kThreads, 0, stream>>>(x, y, rows, cols, xs, ys);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

template <int G, bool kVec>
int dispatch_k(const float* x, float* y, int rows, int cols, long long xs, long long ys, cudaStream_t stream,
               int sms) {
    const int chunks = (cols + 4 * G - 1) / (4 * G);   // four-float chunks per thread
    if (chunks <= 1) return launch_onchip<G, 1, kVec>(x, y, rows, cols, xs, ys, stream, sms);
    if (chunks <= 2) return launch_onchip<G, 2, kVec>(x, y, rows, cols, xs, ys, stream, sms);
    if (chunks <= 4) return launch_onchip<G, 4, kVec>(x, y, rows, cols, xs, ys, stream, sms);
    if (chunks <= 8 || G == 32) return launch_onchip<G, 8, kVec>(x, y, rows, cols, xs, ys, stream, sms);
    return launch_onchip<G, (G == 32 ? 8 : 16), kVec>(x, y, rows, cols, xs, ys, stream, sms);
}

}  // namespace

int launch_softmax_rows(const float* x, float* y, int rows, int cols, long long xs, long long ys,
                        cudaStream_t stream, int dev) {
    int sms = (dev >= 0 && dev < 64) ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    if (cols > SOFTMAX_ROWS_ONCHIP_COLS) {
        long long blocks = rows < (long long)sms * 8 ? rows : (long long)sms * 8;
        softmax_rows_online<<<(unsigned)blocks, kThreads, 0, stream>>>(x, y, rows, cols, xs, ys);
        return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
    }
    const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
                     cols % 4 == 0 && xs % 4 == 0 && ys % 4 == 0;
    if (cols <= 4 * 32 * 8) {   // one warp per row
        return vec ? dispatch_k<32, true>(x, y, rows, cols, xs, ys, stream, sms)
                   : dispatch_k<32, false>(x, y, rows, cols, xs, ys, stream, sms);
    }
    return vec ? dispatch_k<256, true>(x, y, rows, cols, xs, ys, stream, sms)
               : dispatch_k<256, false>(x, y, rows, cols, xs, ys, stream, sms);
}

}  // namespace bos
