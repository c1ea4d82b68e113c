// Attention backward for GB300 (sm_103a). Included once, from attn_fwd_sm103.cu,
// after the shared pieces (bounded waits, tensor maps); it is not a header for
// other files.
//
// The method is Kernel 5 "FlashAttention Backward" of "4.4 Writing GPU Kernels
// with Triton" (llm-stack-book): a preprocessing pass D_i = rowsum(dO_i * O_i),
// then one program per key/value block j that loops over the query blocks able
// to see it, recomputes P = exp(S - L) from the saved natural-log LSE, and
// forms
//     dV_j += P^T dO_i,   dP = dO_i V_j^T,   dS = P * (dP - D_i) * scale,
//     dK_j += dS^T Q_i,   dQ_i += dS K_j   (scattered with fp32 atomic adds),
// accumulating dK_j and dV_j privately and casting the fp32 dQ buffer to bf16
// at the end.
//
// GB300 design: one CTA per key block (192 threads): warps 0-3 compute P and
// dS (thread = key = tensor-memory lane), warp 4 loads with TMA, warp 5 issues
// the tcgen05 MMAs from one thread into one 512-column allocation:
//   T0 (cols 0-127)   : S^T = K Q_i^T (fp32), then P^T as bf16 pairs over its
//                       first 64 columns, then the dQ part dS K_j (fp32, d cols)
//   T1 (cols 128-255) : dP^T = V dO_i^T (fp32), then dS^T as bf16 pairs
//   T2 (cols 256-383) : dV_j (fp32, d cols)
//   T3 (cols 384-511) : dK_j (fp32, d cols)
// Working with the transposes keeps the key on the lane, so dV += P^T dO and
// dK += dS^T Q take P^T and dS^T straight from tensor memory (TS MMAs); dQ =
// dS K needs dS with the query on the lane, so the compute warps also write dS
// to shared memory as [query][key] (K-major, 128-byte swizzle, the layout the
// forward's shared-memory P uses), one 16-bit element per (query, own key).
// Each block's steps run in sequence (no overlap between query blocks beyond
// the TMA loads).

namespace bos {
namespace {

namespace bwd {

constexpr int kThreads = 192;
constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
constexpr uint32_t kT0 = 0, kT1 = 128, kT2 = 256, kT3 = 384;
constexpr float kLog2e = 1.4426950408889634f;

enum : int {
    kBarKV = 0,        // K_j and V_j have landed
    kBarQFull = 1,     // Q_i and dO_i have landed
    kBarQFree = 2,     // every MMA of block i is complete: Q_i, dO_i and the dS buffer are free (commit)
    kBarSFull = 3,     // S^T and dP^T of block i are complete (commit)
    kBarPReady = 4,    // P^T and dS^T of block i are written (128 arrivals)
    kBarDqReady = 5,   // the dQ part of block i is in T0 (commit; also covers dK, dV of block i)
    kBarDqRead = 6,    // the dQ part has been read out of T0 (128 arrivals)
    kBarLse = 7,       // LSE and D of block i are in shared memory (128 arrivals)
    kBarDrain = 8,
    kNumBars = 9,
};

template <int D>
struct Cfg {
    static constexpr int kTile = 128 * D * 2;                  // one bf16 128-row tile
    static constexpr int kBoxes = D / 64;
    static constexpr int kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffDO = 3 * kTile;
    static constexpr int kOffDS = 4 * kTile;                   // dS, [128 queries][128 keys] bf16: 32 KB
    static constexpr int kOffLse = kOffDS + 32768;             // [2][128] LSE * log2 e, then [2][128] D
    static constexpr int kOffBar = kOffLse + 2 * 2 * 128 * 4;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;    // tmem slot, abort flag
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
};

struct BwdArgs {
    int BH, N, d, nkv, causal;
    float scale, c2;                  // c2 = scale * log2 e
    const float* lse;                 // [BH, N] natural log, from the forward pass
    const float* dsum;                // [BH, N] D = rowsum(dO * O)
    float* dq_acc;                    // [BH, N, d] fp32, zeroed before the launch
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    uint64_t wait_limit_ns;
};

template <int D>
__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                         const CUtensorMap* tm_do, uint8_t* smem, uint64_t* bars, volatile int* abort_flag,
                         int bh, int j, int i0, int nq, const BwdArgs& a) {
    using C = Cfg<D>;
    mbar_arrive_expect_tx(&bars[kBarKV], 2 * C::kTile);
    for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_3d(smem + C::kOffK + b * 16384, tm_k, &bars[kBarKV], b * 64, j * 128, bh);
        tma_load_3d(smem + C::kOffV + b * 16384, tm_v, &bars[kBarKV], b * 64, j * 128, bh);
    }
    int last = -1;
    for (int it = 0; it < nq; ++it) {
        const int i = i0 + it;
        // Q_i and dO_i reuse one buffer: wait until block it-1's MMAs are done with it
        if (it > 0 && !wait_or_abort(&bars[kBarQFree], (uint32_t)((it - 1) & 1), a.wait_limit_ns, abort_flag)) break;
        mbar_arrive_expect_tx(&bars[kBarQFull], 2 * C::kTile);
        for (int b = 0; b < C::kBoxes; ++b) {
            tma_load_3d(smem + C::kOffQ + b * 16384, tm_q, &bars[kBarQFull], b * 64, i * 128, bh);
            tma_load_3d(smem + C::kOffDO + b * 16384, tm_do, &bars[kBarQFull], b * 64, i * 128, bh);
        }
        last = it;
    }
    // every copy this thread started must land before the CTA may exit
    mbar_wait(&bars[kBarKV], 0, kDrainLimitNs);
    if (last >= 0) mbar_wait(&bars[kBarQFull], (uint32_t)(last & 1), kDrainLimitNs);
}

template <int D>
__device__ void mma_issuer(uint32_t tm, uint8_t* smem, uint64_t* bars, volatile int* abort_flag, int nq,
                           const BwdArgs& a) {
    using C = Cfg<D>;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
    const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
    const uint32_t sDS = smem_u32(smem + C::kOffDS);
    // S^T, dP^T: M = 128 keys, N = 128 queries, K = d, both operands K-major
    constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
    // dV, dK: M = 128 keys, N = d, K = 128 queries; A from tensor memory, B (dO, Q) N-major
    constexpr uint32_t id_kv = idesc_bf16_f32(128, D, false, true);
    // dQ: M = 128 queries, N = d, K = 128 keys; A (dS in shared memory) K-major, B (K_j) N-major
    constexpr uint32_t id_q = idesc_bf16_f32(128, D, false, true);
    bool ok = wait_or_abort(&bars[kBarKV], 0, lim, abort_flag);
    for (int it = 0; ok && it < nq; ++it) {
        const uint32_t par = (uint32_t)(it & 1);
        if (!wait_or_abort(&bars[kBarQFull], par, lim, abort_flag)) break;
        // T0 is free once the compute warps have read the previous dQ part
        if (it > 0 && !wait_or_abort(&bars[kBarDqRead], par ^ 1, lim, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
            mma_ss(tm + kT0, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
            mma_ss(tm + kT1, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[kBarSFull]);
        if (!wait_or_abort(&bars[kBarPReady], par, lim, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 queries per step: 8 columns of bf16 pairs, 16 rows of dO / Q
            mma_ts(tm + kT2, tm + kT0 + kk * 8, sdesc_sw128(sDO + kk * 2048, 16384, 1024), id_kv,
                   (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_ts(tm + kT3, tm + kT1 + kk * 8, sdesc_sw128(sQ + kk * 2048, 16384, 1024), id_kv,
                   (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 keys per step: 32 bytes of each dS row, 16 rows of K_j
            mma_ss(tm + kT0, sdesc_sw128(sDS + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                   sdesc_sw128(sK + kk * 2048, 16384, 1024), id_q, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarDqReady]);
        mma_commit(&bars[kBarQFree]);
    }
    mma_commit(&bars[kBarDrain]);
    mbar_wait(&bars[kBarDrain], 0, kDrainLimitNs);
}

template <int D>
__device__ void compute_role(uint32_t tm, int w, int lane, uint8_t* smem, uint64_t* bars, volatile int* abort_flag,
                             int bh, int j, int i0, int nq, const BwdArgs& a) {
    using C = Cfg<D>;
    const uint64_t lim = a.wait_limit_ns;
    const int r = w * 32 + lane;                              // tensor-memory lane
    const uint32_t lane_base = tm + ((uint32_t)(w * 32) << 16);
    float* lse_s = reinterpret_cast<float*>(smem + C::kOffLse);         // [2][128]
    float* d_s = lse_s + 2 * 128;                                        // [2][128]
    // this thread's key in the [query][key] dS buffer: box r / 64, 16-byte chunk
    // (r % 64) / 8 (swizzled with the query row), element r % 8
    uint8_t* ds_col = smem + C::kOffDS + (r >> 6) * 16384 + (r & 7) * 2;
    const int ds_chunk = (r & 63) >> 3;
    const int key = j * 128 + r;
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool got = wait_or_abort(bar, parity, lim, abort_flag);
        return __all_sync(0xffffffffu, got);
    };
    bool ok = true;
    for (int it = 0; it < nq; ++it) {
        const uint32_t par = (uint32_t)(it & 1);
        const int q0 = (i0 + it) * 128;
        // this block's LSE (to base 2) and D, one query per thread, into shared memory
        {
            const int q = q0 + r;
            const int b = it & 1;
            lse_s[b * 128 + r] = (q < a.N) ? a.lse[(int64_t)bh * a.N + q] * kLog2e : INFINITY;
            d_s[b * 128 + r] = (q < a.N) ? a.dsum[(int64_t)bh * a.N + q] : 0.f;
            mbar_arrive(&bars[kBarLse]);
        }
        if (!wait_warp(&bars[kBarLse], par) || !wait_warp(&bars[kBarSFull], par)) { ok = false; break; }
        tc_fence_after();
        const float* lse_b = lse_s + (it & 1) * 128;
        const float* d_b = d_s + (it & 1) * 128;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {                      // 32 queries per chunk
            uint32_t sv[32], dpv[32];
            tmem_ld32(lane_base + kT0 + ch * 32, sv);
            tmem_ld32(lane_base + kT1 + ch * 32, dpv);
            uint32_t pk[16], dk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float pp[2], dd[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int qc = ch * 32 + 2 * e + h;
                    const int q = q0 + qc;
                    const bool valid = key < a.N && (!a.causal || q >= key);
                    const float p = valid ? ex2(fmaf(__uint_as_float(sv[2 * e + h]), a.c2, -lse_b[qc])) : 0.f;
                    pp[h] = p;
                    dd[h] = p * (__uint_as_float(dpv[2 * e + h]) - d_b[qc]) * a.scale;
                }
                pk[e] = pack_bf16(pp[0], pp[1]);
                dk[e] = pack_bf16(dd[0], dd[1]);
            }
            tmem_st16(lane_base + kT0 + ch * 16, pk);         // P^T over S^T columns already read
            tmem_st16(lane_base + kT1 + ch * 16, dk);         // dS^T over dP^T columns already read
#pragma unroll
            for (int e = 0; e < 32; ++e) {                    // dS[query][key r], queries 32ch..32ch+31
                const int qr = ch * 32 + e;
                const uint32_t pair = dk[e >> 1];
                *reinterpret_cast<uint16_t*>(ds_col + qr * 128 + ((ds_chunk ^ (qr & 7)) << 4)) =
                    (uint16_t)((e & 1) ? (pair >> 16) : (pair & 0xffffu));
            }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[kBarPReady]);
        // the dQ part: lane r is now query q0 + r
        if (!wait_warp(&bars[kBarDqReady], par)) { ok = false; break; }
        tc_fence_after();
        {
            const int q = q0 + r;
            float* dst = a.dq_acc + ((int64_t)bh * a.N + q) * a.d;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(lane_base + kT0 + c0, v);
                if (q < a.N) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        if (c0 + e < a.d)
                            atomicAdd(reinterpret_cast<float4*>(dst + c0 + e),
                                      make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                                  __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])));
                }
            }
        }
        tc_fence_before();
        mbar_arrive(&bars[kBarDqRead]);
    }
    if (!ok) return;
    // dK_j and dV_j are final once the last block's dQ part was ready (same commit).
    // The tensor-memory loads are warp-collective: every lane takes part, and
    // only the stores depend on the lane's key being inside the sequence.
    tc_fence_after();
    {
        __nv_bfloat16* dkr = a.dk + ((int64_t)bh * a.N + key) * a.d;
        __nv_bfloat16* dvr = a.dv + ((int64_t)bh * a.N + key) * a.d;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t kv[32], vv[32];
            tmem_ld32(lane_base + kT3 + c0, kv);
            tmem_ld32(lane_base + kT2 + c0, vv);
            if (key >= a.N) continue;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                if (c0 + e >= a.d) break;
                uint4 wk, wv;
                wk.x = pack_bf16(__uint_as_float(kv[e]), __uint_as_float(kv[e + 1]));
                wk.y = pack_bf16(__uint_as_float(kv[e + 2]), __uint_as_float(kv[e + 3]));
                wk.z = pack_bf16(__uint_as_float(kv[e + 4]), __uint_as_float(kv[e + 5]));
                wk.w = pack_bf16(__uint_as_float(kv[e + 6]), __uint_as_float(kv[e + 7]));
                wv.x = pack_bf16(__uint_as_float(vv[e]), __uint_as_float(vv[e + 1]));
                wv.y = pack_bf16(__uint_as_float(vv[e + 2]), __uint_as_float(vv[e + 3]));
                wv.z = pack_bf16(__uint_as_float(vv[e + 4]), __uint_as_float(vv[e + 5]));
                wv.w = pack_bf16(__uint_as_float(vv[e + 6]), __uint_as_float(vv[e + 7]));
                *reinterpret_cast<uint4*>(dkr + c0 + e) = wk;
                *reinterpret_cast<uint4*>(dvr + c0 + e) = wv;
            }
        }
    }
}

}  // namespace bwd

// One CTA per (key block j, batch*head); heavier key blocks (small j under causal masking) first.
template <int D>
__global__ void __launch_bounds__(bwd::kThreads, 1)
attn_bwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const bwd::BwdArgs a) {
    using C = bwd::Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int j = blockIdx.x / a.BH, bh = blockIdx.x % a.BH;
    const int i0 = a.causal ? j : 0;
    const int nq = a.nkv - i0;

    if (threadIdx.x == 0) {
        mbar_init(&bars[bwd::kBarKV], 1);
        mbar_init(&bars[bwd::kBarQFull], 1);
        mbar_init(&bars[bwd::kBarQFree], 1);
        mbar_init(&bars[bwd::kBarSFull], 1);
        mbar_init(&bars[bwd::kBarPReady], 128);
        mbar_init(&bars[bwd::kBarDqReady], 1);
        mbar_init(&bars[bwd::kBarDqRead], 128);
        mbar_init(&bars[bwd::kBarLse], 128);
        mbar_init(&bars[bwd::kBarDrain], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == bwd::kWarpProducer && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
    }
    if (warp == bwd::kWarpMma) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_slot[0];

    if (warp < 4) {
        bwd::compute_role<D>(tm, warp, lane, smem, bars, abort_flag, bh, j, i0, nq, a);
    } else if (warp == bwd::kWarpProducer) {
        if (lane == 0) bwd::producer<D>(&tm_q, &tm_k, &tm_v, &tm_do, smem, bars, abort_flag, bh, j, i0, nq, a);
        __syncwarp();
    } else {
        if (lane == 0) bwd::mma_issuer<D>(tm, smem, bars, abort_flag, nq, a);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == bwd::kWarpMma) tmem_dealloc(tm, 512);
}

// D = rowsum(dO * O) in fp32 per row, and the fp32 dQ buffer zeroed: one warp per row.
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                           const __nv_bfloat16* __restrict__ dout,
                                                           float* __restrict__ dsum, float* __restrict__ dq_acc,
                                                           int64_t rows, int d) {
    const int lane = threadIdx.x % 32;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; row < rows;
         row += (int64_t)gridDim.x * blockDim.x / 32) {
        const __nv_bfloat16* orow = o + row * d;
        const __nv_bfloat16* grow = dout + row * d;
        float s = 0.f;
        for (int c = lane; c < d; c += 32) s += __bfloat162float(orow[c]) * __bfloat162float(grow[c]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) dsum[row] = s;
        for (int c = lane; c < d; c += 32) dq_acc[row * d + c] = 0.f;
    }
}

// dQ: the fp32 accumulation buffer to bf16.
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const float* __restrict__ dq_acc,
                                                            __nv_bfloat16* __restrict__ dq, int64_t n) {
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x)
        dq[idx] = __float2bfloat16_rn(dq_acc[idx]);
}

}  // namespace
}  // namespace bos
