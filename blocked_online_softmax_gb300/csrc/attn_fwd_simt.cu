// First, plain CUDA-core implementation of the attention forward pass.
//
// One CTA per (32-row query block, batch*head), four threads per query row,
// key/value blocks of 64 streamed through shared memory, and the online
// softmax of "4.4 Writing GPU Kernels with Triton" (llm-stack-book), Kernel 4
// "A Simplified FlashAttention": running max m, running sum l, unnormalised
// accumulator acc; alpha = exp2(m_old - m_new); one divide at the end; log2(e)
// folded into the scale; LSE converted back to natural log.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"
#include "attn_internal.h"

namespace bos {
namespace {

constexpr int kBM = 32;         // query rows per CTA
constexpr int kBN = 64;         // keys per streamed block
constexpr int kTPR = 4;         // threads per query row
constexpr int kThreads = kBM * kTPR;

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float2 t = __bfloat1622float2(h[e]);
        f[2 * e] = t.x;
        f[2 * e + 1] = t.y;
    }
}

// Thread c of a row owns the 8-element chunks c, c+4, c+8, ... of the head dim,
// so the four threads of a row read four different bank groups of a key row.
template <int D>
__global__ void __launch_bounds__(kThreads)
attn_fwd_simt_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ o,
                     float* __restrict__ lse, int N, float scale_log2, int causal) {
    constexpr int kChunks = D / 8 / kTPR;   // 8-element chunks per thread
    constexpr int kDP = kChunks * 8;        // dims per thread
    __shared__ __align__(16) __nv_bfloat16 ks[kBN][D];
    __shared__ __align__(16) __nv_bfloat16 vs[kBN][D];

    const int tid = threadIdx.x;
    const int r = tid / kTPR, c = tid % kTPR;
    const int64_t i = (int64_t)blockIdx.x * kBM + r;
    const int64_t bh = blockIdx.y;
    const __nv_bfloat16* qh = q + bh * (int64_t)N * D;
    const __nv_bfloat16* kh = k + bh * (int64_t)N * D;
    const __nv_bfloat16* vh = v + bh * (int64_t)N * D;

    float qf[kDP], acc[kDP];
#pragma unroll
    for (int u = 0; u < kChunks; ++u) {
        uint4 w = make_uint4(0, 0, 0, 0);
        if (i < N) w = *reinterpret_cast<const uint4*>(qh + i * D + (u * kTPR + c) * 8);
        unpack8(w, qf + u * 8);
    }
#pragma unroll
    for (int t = 0; t < kDP; ++t) acc[t] = 0.f;
    float m = -INFINITY, l = 0.f;

    const int64_t row_hi = (int64_t)(blockIdx.x + 1) * kBM;
    const int kv_end = causal ? (int)(row_hi < N ? row_hi : N) : N;
    for (int j0 = 0; j0 < kv_end; j0 += kBN) {
        __syncthreads();
        for (int idx = tid; idx < kBN * D / 8; idx += kThreads) {
            const int jr = idx / (D / 8), col = (idx % (D / 8)) * 8;
            const int64_t j = j0 + jr;
            uint4 kw = make_uint4(0, 0, 0, 0), vw = make_uint4(0, 0, 0, 0);
            if (j < N) {
                kw = *reinterpret_cast<const uint4*>(kh + j * D + col);
                vw = *reinterpret_cast<const uint4*>(vh + j * D + col);
            }
            *reinterpret_cast<uint4*>(&ks[jr][col]) = kw;
            *reinterpret_cast<uint4*>(&vs[jr][col]) = vw;
        }
        __syncthreads();

        float s[kBN];
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
            float part = 0.f;
#pragma unroll
            for (int u = 0; u < kChunks; ++u) {
                float kf[8];
                unpack8(*reinterpret_cast<const uint4*>(&ks[jj][(u * kTPR + c) * 8]), kf);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(qf[u * 8 + e], kf[e], part);
            }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            s[jj] = part * scale_log2;          // base-2 logits
        }
        float tile_max = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
            const int64_t j = j0 + jj;
            if (j >= N || (causal && j > i)) s[jj] = -INFINITY;
            tile_max = fmaxf(tile_max, s[jj]);
        }
        const float m_new = fmaxf(m, tile_max);
        // A row whose every key so far is masked keeps m = -inf; subtract 0 then.
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m - m_use);
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < kDP; ++t) acc[t] *= alpha;
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
            const float p = exp2f(s[jj] - m_use);
            sum += p;
#pragma unroll
            for (int u = 0; u < kChunks; ++u) {
                float vf[8];
                unpack8(*reinterpret_cast<const uint4*>(&vs[jj][(u * kTPR + c) * 8]), vf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[u * 8 + e] = fmaf(p, vf[e], acc[u * 8 + e]);
            }
        }
        l = l * alpha + sum;
        m = m_new;
    }

    if (i < N) {
        const float l_safe = (l > 0.f) ? l : 1.f;
        const float inv = 1.f / l_safe;
        __nv_bfloat16* oh = o + bh * (int64_t)N * D + i * D;
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
            __align__(16) __nv_bfloat162 outv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                outv[e] = __floats2bfloat162_rn(acc[u * 8 + 2 * e] * inv, acc[u * 8 + 2 * e + 1] * inv);
            *reinterpret_cast<uint4*>(oh + (u * kTPR + c) * 8) = *reinterpret_cast<uint4*>(outv);
        }
        if (c == 0) lse[bh * (int64_t)N + i] = (m + log2f(l_safe)) * 0.69314718055994531f;
    }
}

}  // namespace

int launch_attn_fwd(const AttnParams& p, cudaStream_t stream, int /*dev*/) {
    const float scale_log2 = p.scale * 1.44269504088896341f;
    dim3 grid((unsigned)((p.N + kBM - 1) / kBM), (unsigned)(p.B * p.H));
    const auto* q = static_cast<const __nv_bfloat16*>(p.q);
    const auto* k = static_cast<const __nv_bfloat16*>(p.k);
    const auto* v = static_cast<const __nv_bfloat16*>(p.v);
    auto* o = static_cast<__nv_bfloat16*>(p.o);
    if (p.d == 64)
        attn_fwd_simt_kernel<64><<<grid, kThreads, 0, stream>>>(q, k, v, o, p.lse, p.N, scale_log2, p.causal);
    else
        attn_fwd_simt_kernel<128><<<grid, kThreads, 0, stream>>>(q, k, v, o, p.lse, p.N, scale_log2, p.causal);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace bos
