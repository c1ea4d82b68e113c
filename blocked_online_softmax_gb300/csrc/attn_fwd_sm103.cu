// Attention forward for GB300 (sm_103a): TMA-fed shared-memory ring, tcgen05
// MMAs accumulating in tensor memory, and the blocked online softmax.
//
// The method is that of "4.4 Writing GPU Kernels with Triton" (llm-stack-book),
// Kernel 4 "A Simplified FlashAttention" and "The Online Softmax Recurrence":
// keys and values stream through on-chip memory in blocks; each query row keeps
// a running max m, a running sum l and an unnormalised accumulator O; a new
// block's scores s give p = exp2(s*scale*log2e - m), l = alpha*l + sum(p),
// O = alpha*O + p.V with alpha = exp2(m_old - m_new); one divide at the end;
// LSE = (m + log2 l) * ln2 in natural log. The score matrix never leaves the SM.
//
// GB300 design (what differs from the page's Triton kernel):
//  * Work unit = 256 query rows of one (batch, head) = two 128-row Q tiles that
//    share every K/V tile. CTAs are persistent (one per SM) and walk a static
//    list of units: for causal masking the list is heaviest-first over all heads
//    and dealt to CTAs in snake order, which balances the triangle of work.
//  * Warp roles (384 threads): warp 0 issues TMA loads (Q per unit, then K_j,
//    V_j into a multi-stage ring); warp 1 issues tcgen05 MMAs from one thread;
//    warp 2 owns the tensor-memory allocation; warpgroups 1 and 2 run the
//    softmax of Q tile 0 and Q tile 1, one thread per query row.
//  * Tensor memory (512 columns x 128 lanes): S_t = Q_t K^T (fp32, 128 cols per
//    tile), P_t (bf16, written over the first 64 columns of S_t) and O_t (fp32,
//    d columns). O += P V takes P straight from tensor memory.
//  * MMA order PV_0(i), S_0(i+1), PV_1(i), S_1(i+1): while one softmax
//    warpgroup works on its tile, the tensor core runs the other tile's MMAs.
//  * Key blocks are visited from the last to the first, so the only masked
//    blocks (the causal diagonal, the ragged tail past N) come first and the
//    steady-state loop has no masking. Causal: blocks past a tile's diagonal are
//    skipped, as in the page's loop bound.
//  * The running max is only moved (and O, l rescaled) when a block's max
//    exceeds it by more than 8 in log2 units; otherwise exponentials are taken
//    against the older, smaller max (p <= 2^8). O/l and LSE are unchanged in
//    exact arithmetic, and the O rescale through tensor memory becomes rare.
//  * Every wait is bounded in wall time: on expiry the kernel records a status,
//    drains its own copies and MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace bos {
namespace {

using namespace ptx;

constexpr int kBM = 128;                  // query rows per Q tile (tensor-memory lanes)
constexpr int kBN = 128;                  // keys per K/V tile
constexpr int kUnitRows = 2 * kBM;        // query rows per work unit
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f; // log2 units
constexpr uint32_t kTmemCols = 512;
// tensor-memory column of S_t (P_t overlays its first 64 columns) and of O_t
__host__ __device__ constexpr uint32_t tmem_s_col(int t) { return (uint32_t)t * 128u; }
__host__ __device__ constexpr uint32_t tmem_o_col(int t) { return 256u + (uint32_t)t * 128u; }
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;         // 1 s

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kBN * D * 2;          // one bf16 Q, K or V tile
    static constexpr int kStages = (D == 128) ? 4 : 8;      // K/V ring depth
    static constexpr int kBoxes = D / 64;                   // 64-column TMA boxes per tile
    static constexpr int kOffKV = 2 * kTileBytes;           // after the two Q tiles
    static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
    // barriers: q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], drain, never
    static constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 2 + 1 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
};

struct KernelArgs {
    int BH, N, U, causal;
    float scale_log2;
    __nv_bfloat16* o;
    float* lse;
    uint64_t wait_limit_ns;
    int test_stall;   // test hook: the MMA thread first waits on a barrier nothing signals
};

}  // namespace

// Sticky device-side status: 0, or the attn_status of the first failure.
__device__ int g_attn_device_status;

namespace {

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicCAS(&g_attn_device_status, 0, (int)ATTN_ERR_TIMEOUT);
            return false;
        }
    }
}

// Decoded work unit.
struct Unit {
    int bh, row0, n, first0;   // n key tiles for Q tile 1; Q tile 0 starts at iteration first0
};

__device__ __forceinline__ Unit decode_unit(int k, const KernelArgs& a) {
    Unit u;
    int q;
    if (a.causal) {            // heaviest first over all heads
        q = a.U - 1 - k / a.BH;
        u.bh = k % a.BH;
    } else {                   // head-major (every unit costs the same)
        u.bh = k / a.U;
        q = k % a.U;
    }
    u.row0 = q * kUnitRows;
    const int nkv = (a.N + kBN - 1) / kBN;
    int c0 = nkv, c1 = nkv;
    if (a.causal) {
        c0 = min(u.row0 / kBN + 1, nkv);
        c1 = min(u.row0 / kBN + 2, nkv);
    }
    u.n = c1;
    u.first0 = c1 - c0;
    return u;
}

// k-th unit of this CTA: snake order over the grid.
__device__ __forceinline__ int unit_index(int r) {
    const int G = gridDim.x, g = blockIdx.x;
    return r * G + ((r & 1) ? (G - 1 - g) : g);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ roles

template <int D>
__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                         uint8_t* sQ, uint8_t* sKV, uint64_t* bars, volatile int* abort_flag,
                         const KernelArgs& a) {
    using C = Cfg<D>;
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = bars + 2 + C::kStages;
    const int total = a.BH * a.U;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;             // stages with a load whose completion is not yet observed
    uint32_t issued_parity = 0;           // parity of that load's phase, per stage
    int q_parity = -1;                    // parity of the last Q load's phase, -1 before the first
    bool ok = true;
    // One K/V tile into the next ring stage.
    auto load_kv = [&](const CUtensorMap* tm, int j, int bh) -> bool {
        if (!wait_or_abort(&kv_empty[stage], phase ^ 1, a.wait_limit_ns, abort_flag)) return false;
        mbar_arrive_expect_tx(&kv_full[stage], C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(sKV + stage * C::kTileBytes + b * 16384, tm, &kv_full[stage], b * 64, j * kBN, bh);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        return true;
    };
    int it = 0;
    for (int r = 0; ok; ++r, ++it) {
        const int k = unit_index(r);
        if (k >= total) break;
        const Unit u = decode_unit(k, a);
        // The first K/V pair of a unit goes ahead of its Q tiles: Q must wait until the
        // previous unit's last S = Q K^T has read the Q buffer, the ring need not.
        for (int i = 0; i < u.n && ok; ++i) {
            const int j = u.n - 1 - i;
            if (!load_kv(tm_k, j, u.bh) || !load_kv(tm_v, j, u.bh)) { ok = false; break; }
            if (i == 0) {
                if (!wait_or_abort(q_empty, (it & 1) ^ 1, a.wait_limit_ns, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(q_full, 2 * C::kTileBytes);
                q_parity = it & 1;
                for (int t = 0; t < 2; ++t)
                    for (int b = 0; b < C::kBoxes; ++b)
                        tma_load_3d(sQ + t * C::kTileBytes + b * 16384, tm_q, q_full, b * 64, u.row0 + t * kBM,
                                    u.bh);
            }
        }
    }
    // Every copy this thread started must land before the CTA may exit (on the
    // normal path they already have).
    for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait(&kv_full[s], (issued_parity >> s) & 1u, kDrainLimitNs);
    if (q_parity >= 0) mbar_wait(q_full, (uint32_t)q_parity, kDrainLimitNs);
}

template <int D>
__device__ __forceinline__ void issue_s(uint32_t tmem, int t, const uint8_t* sQ, const uint8_t* sK) {
    using C = Cfg<D>;
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
    const uint32_t qa = smem_u32(sQ + t * C::kTileBytes), ka = smem_u32(sK);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;   // 64-column box, 32-byte K step
        mma_ss(tmem + tmem_s_col(t), sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc,
               kk > 0 ? 1u : 0u);
    }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem, int t, const uint8_t* sV, bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, false, true);
    const uint32_t va = smem_u32(sV);
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)   // 16 keys per step: 8 P columns, 16 V rows (2048 bytes)
        mma_ts(tmem + tmem_o_col(t), tmem + tmem_s_col(t) + kk * 8, sdesc_sw128(va + kk * 2048, 16384, 1024), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
}

template <int D>
__device__ void mma_issuer(uint32_t tmem, const uint8_t* sQ, const uint8_t* sKV, uint64_t* bars,
                           volatile int* abort_flag, const KernelArgs& a) {
    using C = Cfg<D>;
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = bars + 2 + C::kStages;
    uint64_t* s_full = bars + 2 + 2 * C::kStages;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_full = p_full + 2;
    uint64_t* drain = o_full + 2;
    uint64_t* never = o_full + 3;
    const uint64_t lim = a.wait_limit_ns;
    const int total = a.BH * a.U;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t p_phase[2] = {0, 0};
    bool ok = true;
    auto next_stage = [&](int& st) -> bool {
        st = stage;
        const bool got = wait_or_abort(&kv_full[stage], phase, lim, abort_flag);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        return got;
    };
    if (a.test_stall && !wait_or_abort(never, 0, lim, abort_flag)) ok = false;
    int it = 0;
    for (int r = 0; ok; ++r, ++it) {
        const int k = unit_index(r);
        if (k >= total) break;
        const Unit u = decode_unit(k, a);
        if (!wait_or_abort(q_full, it & 1, lim, abort_flag)) { ok = false; break; }
        tc_fence_after();
        int kst, vst;
        if (!next_stage(kst)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* sK = sKV + kst * C::kTileBytes;
        if (u.first0 == 0) { issue_s<D>(tmem, 0, sQ, sK); mma_commit(&s_full[0]); }
        issue_s<D>(tmem, 1, sQ, sK);
        mma_commit(&s_full[1]);
        mma_commit(&kv_empty[kst]);
        if (u.n == 1) mma_commit(q_empty);
        for (int i = 0; i < u.n; ++i) {
            if (!next_stage(vst)) { ok = false; break; }
            const uint8_t* sV = sKV + vst * C::kTileBytes;
            if (i >= u.first0) {
                if (!wait_or_abort(&p_full[0], p_phase[0], lim, abort_flag)) { ok = false; break; }
                p_phase[0] ^= 1;
                tc_fence_after();
                issue_pv<D>(tmem, 0, sV, i > u.first0);
                if (i == u.n - 1) mma_commit(&o_full[0]);
            }
            const bool more = (i + 1 < u.n);
            if (more) {
                if (!next_stage(kst)) { ok = false; break; }
                tc_fence_after();
                sK = sKV + kst * C::kTileBytes;
                if (i + 1 >= u.first0) { issue_s<D>(tmem, 0, sQ, sK); mma_commit(&s_full[0]); }
            }
            if (!wait_or_abort(&p_full[1], p_phase[1], lim, abort_flag)) { ok = false; break; }
            p_phase[1] ^= 1;
            tc_fence_after();
            issue_pv<D>(tmem, 1, sV, i > 0);
            mma_commit(&kv_empty[vst]);
            if (i == u.n - 1) mma_commit(&o_full[1]);
            if (more) {
                issue_s<D>(tmem, 1, sQ, sK);
                mma_commit(&s_full[1]);
                mma_commit(&kv_empty[kst]);
                if (i + 1 == u.n - 1) mma_commit(q_empty);
            }
        }
    }
    // Every MMA this thread issued must complete before tensor memory is freed.
    mma_commit(drain);
    mbar_wait(drain, 0, kDrainLimitNs);
}

template <int D>
__device__ void softmax_role(uint32_t tmem, int t, int wq, int lane, uint64_t* bars, volatile int* abort_flag,
                             const KernelArgs& a) {
    using C = Cfg<D>;
    uint64_t* s_full = bars + 2 + 2 * C::kStages;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_full = p_full + 2;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t tS = lane_base + tmem_s_col(t);
    const uint32_t tO = lane_base + tmem_o_col(t);
    const int row_in_tile = wq * 32 + lane;
    const float c = a.scale_log2;
    const int total = a.BH * a.U;
    uint32_t s_phase = 0, o_phase = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int k = unit_index(r);
        if (k >= total) break;
        const Unit u = decode_unit(k, a);
        const int tile_row0 = u.row0 + t * kBM;
        const int row = tile_row0 + row_in_tile;
        const int first = (t == 0) ? u.first0 : 0;
        float m_ref = -INFINITY;   // max the exponentials are taken against (base-2 units)
        float l = 0.f;
        for (int i = first; i < u.n; ++i) {
            const int j = u.n - 1 - i;
            bool got = wait_or_abort(&s_full[t], s_phase, lim, abort_flag);
            got = __all_sync(0xffffffffu, got);
            if (!got) { ok = false; break; }
            s_phase ^= 1;
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128(tS, sr);
            const int key0 = j * kBN;
            const bool need_mask = (key0 + kBN > a.N) || (a.causal && key0 + kBN - 1 > tile_row0);
            float m_tile;
            if (need_mask) {
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int cc = 0; cc < 128; ++cc) {
                    const int key = key0 + cc;
                    float x = __uint_as_float(sr[cc]) * c;
                    if (key >= a.N || (a.causal && key > row)) x = -INFINITY;
                    sr[cc] = __float_as_uint(x);
                    mx[cc & 3] = fmaxf(mx[cc & 3], x);
                }
                m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            } else {
                float mx[4], mn[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) mx[q] = mn[q] = __uint_as_float(sr[q]);
#pragma unroll
                for (int cc = 4; cc < 128; ++cc) {
                    const float s = __uint_as_float(sr[cc]);
                    mx[cc & 3] = fmaxf(mx[cc & 3], s);
                    mn[cc & 3] = fminf(mn[cc & 3], s);
                }
                const float smax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const float smin = fminf(fminf(mn[0], mn[1]), fminf(mn[2], mn[3]));
                m_tile = (c >= 0.f) ? smax * c : smin * c;
            }
            float alpha = 1.f;
            if (m_ref == -INFINITY) {
                m_ref = m_tile;
            } else if (m_tile > m_ref + kRescaleThreshold) {
                alpha = ex2(m_ref - m_tile);
                m_ref = m_tile;
            }
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
            float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {           // 32 keys -> 16 packed bf16 pairs per chunk
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c0 = ch * 32 + 2 * e;
                    float p0, p1;
                    if (need_mask) {
                        p0 = ex2(__uint_as_float(sr[c0]) - m_use);
                        p1 = ex2(__uint_as_float(sr[c0 + 1]) - m_use);
                    } else {
                        p0 = ex2(fmaf(__uint_as_float(sr[c0]), c, -m_use));
                        p1 = ex2(fmaf(__uint_as_float(sr[c0 + 1]), c, -m_use));
                    }
                    sum[e & 3] += p0;
                    sum[(e + 2) & 3] += p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                tmem_st16(tS + ch * 16, pk);
            }
            l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t orow[32];
                    tmem_ld32(tO + ch * 32, orow);
#pragma unroll
                    for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st32(tO + ch * 32, orow);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
        }
        if (!ok) break;
        // epilogue: O / l -> bf16, LSE in natural log
        bool got = wait_or_abort(&o_full[t], o_phase, lim, abort_flag);
        got = __all_sync(0xffffffffu, got);
        if (!got) { ok = false; break; }
        o_phase ^= 1;
        tc_fence_after();
        const float l_safe = (l > 0.f) ? l : 1.f;
        const float inv = 1.f / l_safe;
        __nv_bfloat16* orow_ptr = a.o + ((int64_t)u.bh * a.N + row) * D;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t ov[32];
            tmem_ld32(tO + ch * 32, ov);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pk[e] = pack_bf16(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
            if (row < a.N) {
                uint4* dst = reinterpret_cast<uint4*>(orow_ptr + ch * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
        }
        if (row < a.N) a.lse[(int64_t)u.bh * a.N + row] = (m_ref + log2f(l_safe)) * 0.69314718055994531f;
        tc_fence_before();
    }
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const KernelArgs a) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + C::kOffKV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        mbar_init(bars + 0, 1);                                  // q_full
        mbar_init(bars + 1, 1);                                  // q_empty
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bars + 2 + s, 1);                          // kv_full
            mbar_init(bars + 2 + C::kStages + s, 1);             // kv_empty
        }
        uint64_t* s_full = bars + 2 + 2 * C::kStages;
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full + t, 1);                            // s_full
            mbar_init(s_full + 2 + t, kBM);                      // p_full: every softmax thread arrives
            mbar_init(s_full + 4 + t, 1);                        // o_full
        }
        mbar_init(s_full + 6, 1);                                // drain
        mbar_init(s_full + 7, 1);                                // never (test hook)
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) producer<D>(&tm_q, &tm_k, &tm_v, sQ, sKV, bars, abort_flag, a);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<D>(tmem, sQ, sKV, bars, abort_flag, a);
        __syncwarp();
    } else if (warp >= 4) {
        softmax_role<D>(tmem, (warp - 4) / 4, warp % 4, lane, bars, abort_flag, a);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// [BH, N, D] bf16 viewed as a 3-D tensor (D innermost); 64x128 boxes, 128-byte
// swizzle; rows past N read as zero.
bool encode_qkv_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int BH, int N, int D) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kBN, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint64_t g_wait_limit_ns = kDefaultWaitLimitNs;
int g_test_stall = 0;

template <int D>
int launch_d(const AttnParams& p, cudaStream_t stream, int dev) {
    using C = Cfg<D>;
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return ATTN_ERR_CUDA;
    const int BH = p.B * p.H;
    CUtensorMap mq, mk, mv;
    if (!encode_qkv_map(enc, &mq, p.q, BH, p.N, D) || !encode_qkv_map(enc, &mk, p.k, BH, p.N, D) ||
        !encode_qkv_map(enc, &mv, p.v, BH, p.N, D))
        return ATTN_ERR_BAD_SHAPE;
    static int sms_cache[64] = {0};
    static int attr_done[64] = {0};
    int sms = (dev >= 0 && dev < 64) ? sms_cache[dev] : 0;
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) sms_cache[dev] = sms;
    }
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        if (cudaFuncSetAttribute(attn_fwd_sm103_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_LAUNCH;
        }
        if (dev >= 0 && dev < 64) attr_done[dev] = 1;
    }
    KernelArgs a;
    a.BH = BH;
    a.N = p.N;
    a.U = (p.N + kUnitRows - 1) / kUnitRows;
    a.causal = p.causal;
    a.scale_log2 = (float)((double)p.scale * 1.4426950408889634);
    a.o = static_cast<__nv_bfloat16*>(p.o);
    a.lse = p.lse;
    a.wait_limit_ns = g_wait_limit_ns;
    a.test_stall = g_test_stall;
    const int64_t units = (int64_t)BH * a.U;
    const int grid = (int)(units < sms ? units : sms);
    attn_fwd_sm103_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, a);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_attn_fwd(const AttnParams& p, cudaStream_t stream, int dev) {
    return p.d == 64 ? launch_d<64>(p, stream, dev) : launch_d<128>(p, stream, dev);
}

void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns ? ns : kDefaultWaitLimitNs; }

void set_test_stall(int on) { g_test_stall = on ? 1 : 0; }

int read_and_clear_device_status(cudaStream_t stream) {
    int h = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_attn_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_attn_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return h;
}

}  // namespace bos
