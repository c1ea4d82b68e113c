// Attention forward for head dimension 64 (sm_103a). Included once, from
// attn_fwd_sm103.cu, after the shared pieces (scheduler, waits, softmax
// arithmetic); it is not a header for other files.
//
// Same method and work split as the d = 128 kernel (two 128-row Q tiles per
// unit, one MMA stream and one softmax warpgroup per tile), but with d = 64 a
// tile's S (128 columns), P (128 keys as 64 columns of bf16 pairs) and O (64
// columns) fit side by side in its 256 tensor-memory columns. P therefore has
// its own columns and both halves of O += P V are TS MMAs; S(i+1) only waits
// until the softmax has read S(i) into registers, so the tensor core computes
// the next scores while the softmax works on the current block. Each stream
// issues S(0), S(1), PV(0), S(2), PV(1), ... and the K/V ring is loaded one K
// ahead of V in that order. Q is double-buffered; O is staged for its TMA
// stores in a buffer of its own.

namespace bos {
namespace {

namespace d64 {

constexpr int kD = 64;
constexpr uint32_t kTmemS = 0;       // S_t, fp32, 128 columns
constexpr uint32_t kTmemP = 128;     // P_t, bf16 pairs, 64 columns
constexpr uint32_t kTmemO = 192;     // O_t, fp32, 64 columns

enum : int {
    kBarQFull = 0,      // [2] per Q buffer: the unit's two Q tiles have landed
    kBarQEmpty = 2,     // [2] per Q buffer: both streams' last S of the unit is complete (two commits)
    kBarSFull = 4,      // [2] S_t complete (MMA commit)
    kBarSFree = 6,      // [2] the softmax has read S_t into registers (128 arrivals)
    kBarPHalf = 8,      // [2] keys 0-63 of P_t are in tensor memory (128 arrivals)
    kBarPFull = 10,     // [2] keys 64-127 of P_t are in tensor memory (128 arrivals)
    kBarPaDone = 12,    // [2] PV_t for keys 0-63 complete (MMA commit)
    kBarPbDone = 14,    // [2] PV_t for keys 64-127 complete: O_t current (MMA commit)
    kBarDrain = 16,     // [2]
    kBarNever = 18,     // never signalled (test hook)
    kBarUnitFull = 19,  // [kUnitRing]
    kBarUnitEmpty = 23, // [kUnitRing]
    kBarKV = 27,        // kv_full[kStages], then kv_empty[kStages]
};

struct Cfg {
    static constexpr int kTileBytes = kBN * kD * 2;         // one bf16 Q, K, V or O tile: 16 KB
    static constexpr int kStages = 8;
    // shared memory: Q [2 buffers][2 tiles] | O staging [2 tiles] | K/V ring | barriers | misc
    static constexpr int kOffEpi = 4 * kTileBytes;
    static constexpr int kOffKV = kOffEpi + 2 * kTileBytes;
    static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
    static constexpr int kNumBars = kBarKV + 2 * kStages;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slots [2], abort flag, unit ring [4]
    static constexpr int kSmemBytes = kOffMisc + 32 + 1024;  // + alignment slack
};

__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint8_t* sQ,
                         uint8_t* sKV, uint64_t* bars, const UnitRing& ring, volatile int* abort_flag,
                         volatile int* member, const KernelArgs& a) {
    uint64_t* kv_full = bars + kBarKV;
    uint64_t* kv_empty = bars + kBarKV + Cfg::kStages;
    const int total = a.BH * a.U;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;   // ring loads whose completion is not yet observed
    int q_parity[2] = {-1, -1};                    // per Q buffer: parity of its last load, -1 before any
    bool ok = true;
    auto load_kv = [&](const CUtensorMap* tm, int j, int h, int b) -> bool {
        if (!wait_or_abort(&kv_empty[stage], phase ^ 1, a.wait_limit_ns, abort_flag)) return false;
        mbar_arrive_expect_tx(&kv_full[stage], Cfg::kTileBytes);
        tma_load_4d(sKV + stage * Cfg::kTileBytes, tm, &kv_full[stage], 0, j * kBN, h, b);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == Cfg::kStages) { stage = 0; phase ^= 1; }
        return true;
    };
    for (int r = 0; ok; ++r) {
        const int sl = r % kUnitRing;
        if (!wait_or_abort(&bars[kBarUnitEmpty + sl], (uint32_t)((r / kUnitRing) & 1) ^ 1, a.wait_limit_ns,
                           abort_flag)) {
            ok = false;
            break;
        }
        int k;   // the first unit of CTA g is g; a CTA whose counter slot is held elsewhere takes none
        if (r == 0) {
            *member = sched_claim(a.sched) ? 1 : 0;
            k = *member ? (int)blockIdx.x : total;
        } else {
            k = (int)gridDim.x + (int)atomicAdd(a.sched, 1u);
        }
        ring.idx[sl] = k;
        mbar_arrive(&bars[kBarUnitFull + sl]);
        if (k >= total) break;
        const Unit u = decode_unit(k, a);
        const int qb = r & 1;
        if (!wait_or_abort(&bars[kBarQEmpty + qb], ((r >> 1) & 1) ^ 1, a.wait_limit_ns, abort_flag)) {
            ok = false;
            break;
        }
        mbar_arrive_expect_tx(&bars[kBarQFull + qb], 2 * Cfg::kTileBytes);
        q_parity[qb] = (r >> 1) & 1;
        for (int t = 0; t < 2; ++t)
            tma_load_4d(sQ + (qb * 2 + t) * Cfg::kTileBytes, tm_q, &bars[kBarQFull + qb], 0, u.row0 + t * kBM,
                        u.h, u.b);
        // key block i is j = n-1-i; K runs one block ahead of V
        if (!load_kv(tm_k, u.n - 1, u.h, u.b)) { ok = false; break; }
        for (int i = 0; i < u.n && ok; ++i) {
            if (i + 1 < u.n && !load_kv(tm_k, u.n - 2 - i, u.h, u.b)) { ok = false; break; }
            if (!load_kv(tm_v, u.n - 1 - i, u.h, u.b)) { ok = false; break; }
        }
    }
    for (int s = 0; s < Cfg::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait(&kv_full[s], (issued_parity >> s) & 1u, kDrainLimitNs);
    for (int qb = 0; qb < 2; ++qb)
        if (q_parity[qb] >= 0) mbar_wait(&bars[kBarQFull + qb], (uint32_t)q_parity[qb], kDrainLimitNs);
}

// S_t = Q_t K^T (K = 64: four steps of 16 within one 128-byte swizzled row).
template <bool kF16>
__device__ __forceinline__ void issue_s(uint32_t tm, const uint8_t* sQt, const uint8_t* sK) {
    constexpr uint32_t idesc = idesc_f32acc(kBM, kBN, false, false, kF16);
    const uint32_t qa = smem_u32(sQt), ka = smem_u32(sK);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss(tm + kTmemS, sdesc_sw128(qa + kk * 32, 16, 1024), sdesc_sw128(ka + kk * 32, 16, 1024), idesc,
               kk > 0 ? 1u : 0u);
}

// O_t (+)= P_t[:, keys 64h .. 64h+63] * V[those keys, :], P from its tensor-memory columns.
template <bool kF16>
__device__ __forceinline__ void issue_pv(uint32_t tm, const uint8_t* sV, int h, bool accumulate) {
    constexpr uint32_t idesc = idesc_f32acc(kBM, kD, false, true, kF16);
    const uint32_t va = smem_u32(sV);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {   // 16 keys per step: 8 P columns, 16 V rows (2048 bytes)
        const int step = h * 4 + kk;
        mma_ts(tm + kTmemO, tm + kTmemP + step * 8, sdesc_sw128(va + step * 2048, 16384, 1024), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
    }
}

template <bool kF16>
__device__ void mma_issuer(uint32_t tm, int t, const uint8_t* sQ, const uint8_t* sKV, uint64_t* bars,
                           const UnitRing& ring, volatile int* abort_flag, const KernelArgs& a) {
    uint64_t* kv_full = bars + kBarKV;
    uint64_t* kv_empty = bars + kBarKV + Cfg::kStages;
    uint64_t* s_full = bars + kBarSFull + t;
    uint64_t* s_free = bars + kBarSFree + t;
    uint64_t* p_half = bars + kBarPHalf + t;
    uint64_t* p_full = bars + kBarPFull + t;
    uint64_t* pa_done = bars + kBarPaDone + t;
    uint64_t* pb_done = bars + kBarPbDone + t;
    const uint64_t lim = a.wait_limit_ns;
    const int total = a.BH * a.U;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t s_count = 0;    // S blocks issued so far
    uint32_t pv_count = 0;   // PV blocks issued so far
    bool ok = true;
    if (t == 0 && a.test_stall && !wait_or_abort(bars + kBarNever, 0, lim, abort_flag)) ok = false;
    auto next_stage = [&](int& st) -> bool {
        st = stage;
        if (!wait_or_abort(&kv_full[stage], phase, lim, abort_flag)) return false;
        if (++stage == Cfg::kStages) { stage = 0; phase ^= 1; }
        return true;
    };
    for (int r = 0; ok; ++r) {
        int k;
        if (!ring.get(r, k, lim, abort_flag)) { ok = false; break; }
        ring.release(r);
        if (k >= total) break;
        const Unit u = decode_unit(k, a);
        const int first = (t == 0) ? u.first0 : 0;   // Q tile 0 skips the block past its diagonal
        const int qb = r & 1;
        const uint8_t* sQt = sQ + (qb * 2 + t) * Cfg::kTileBytes;
        if (!wait_or_abort(&bars[kBarQFull + qb], (r >> 1) & 1, lim, abort_flag)) { ok = false; break; }
        for (int i = -1; i < u.n; ++i) {
            if (i + 1 < u.n) {   // S(i+1), once the softmax has read the previous S out of S_t
                int kst;
                if (!next_stage(kst)) { ok = false; break; }
                if (i + 1 >= first) {
                    if (s_count > 0 && !wait_or_abort(s_free, (s_count - 1) & 1, lim, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s<kF16>(tm, sQt, sKV + kst * Cfg::kTileBytes);
                    mma_commit(s_full);
                    ++s_count;
                }
                mma_commit(&kv_empty[kst]);
                if (i + 1 == u.n - 1) mma_commit(&bars[kBarQEmpty + qb]);
            }
            if (i < 0) continue;
            int vst;   // PV(i), one half of P at a time
            if (!next_stage(vst)) { ok = false; break; }
            if (i >= first) {
                const uint32_t par = pv_count & 1;
                if (!wait_or_abort(p_half, par, lim, abort_flag)) { ok = false; break; }
                tc_fence_after();
                issue_pv<kF16>(tm, sKV + vst * Cfg::kTileBytes, 0, i > first);
                mma_commit(pa_done);
                if (!wait_or_abort(p_full, par, lim, abort_flag)) { ok = false; break; }
                tc_fence_after();
                issue_pv<kF16>(tm, sKV + vst * Cfg::kTileBytes, 1, true);
                mma_commit(pb_done);
                ++pv_count;
            }
            mma_commit(&kv_empty[vst]);
        }
    }
    mma_commit(&bars[kBarDrain + t]);
    mbar_wait(&bars[kBarDrain + t], 0, kDrainLimitNs);
}

// Keys 64h .. 64h+63 of P_t (chunks 2h and 2h+1) into P_t's tensor-memory columns.
template <bool kF16>
__device__ __forceinline__ void p_half_to_tmem(const uint32_t (&sr)[128], int h, uint64_t c2, uint64_t negm2,
                                               uint64_t (&acc)[4], uint32_t tP) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[16];
        exp_pack<kF16>(sr, 2 * h + cc, c2, negm2, acc, pk);
        tmem_st16(tP + (2 * h + cc) * 16, pk);
    }
}

template <bool kF16>
__device__ void softmax_role(uint32_t tm, int t, int wq, int lane, uint64_t* bars, const UnitRing& ring,
                             volatile int* abort_flag, uint8_t* sEpi, const CUtensorMap* tm_o, const KernelArgs& a) {
    uint64_t* s_full = bars + kBarSFull + t;
    uint64_t* s_free = bars + kBarSFree + t;
    uint64_t* p_half = bars + kBarPHalf + t;
    uint64_t* p_full = bars + kBarPFull + t;
    uint64_t* pa_done = bars + kBarPaDone + t;
    uint64_t* pb_done = bars + kBarPbDone + t;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t lane_base = tm + ((uint32_t)(wq * 32) << 16);
    const uint32_t tS = lane_base + kTmemS;
    const uint32_t tP = lane_base + kTmemP;
    const uint32_t tO = lane_base + kTmemO;
    const int row_in_tile = wq * 32 + lane;
    uint8_t* sEpit = sEpi + t * Cfg::kTileBytes;
    const uint32_t erow = smem_u32(sEpit + row_in_tile * 128);   // this row of the staging buffer
    uint8_t* ewarp = sEpit + wq * 32 * 128;   // this warp's 32 rows (4 KB, 1024-byte aligned)
    const int swz = row_in_tile & 7;
    const float c = a.scale_log2;
    // with c == 0 every score is replaced by 0 (mask_row) and scaled by 1
    const float cs = (c == 0.f) ? 1.f : c;
    const uint64_t c2 = f2_pack(cs, cs);
    const int total = a.BH * a.U;
    uint32_t s_phase = 0;
    uint32_t blocks = 0;       // blocks of this tile processed so far; PV of block g completes pa/pb phase g
    bool ok = true;
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool got = wait_or_abort(bar, parity, lim, abort_flag);
        return __all_sync(0xffffffffu, got);
    };
    for (int r = 0; ok; ++r) {
        int k;
        bool got = ring.get(r, k, lim, abort_flag);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        __syncwarp();
        if (lane == 0) ring.release(r);
        if (k >= total) break;
        const Unit u = decode_unit(k, a);
        const int tile_row0 = u.row0 + t * kBM;
        const int row = tile_row0 + row_in_tile;
        const int first = (t == 0) ? u.first0 : 0;
        float m_ref = -INFINITY;   // max the exponentials are taken against (base-2 units)
        float l = 0.f;     // sum of the fp32 probabilities (LSE)
        float l_o = 0.f;   // the same plus each block's top-term rounding error (normalises O)
        for (int i = first; i < u.n; ++i) {
            const int j = u.n - 1 - i;
            if (!wait_warp(s_full, s_phase)) { ok = false; break; }
            s_phase ^= 1;
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128(tS, sr);
            tc_fence_before();
            mbar_arrive(s_free);       // the stream may now write S(i+1) over S_t
            const int key0 = j * kBN;
            const bool need_mask = (key0 + kBN > a.N) || (a.causal && key0 + kBN - 1 > tile_row0);
            if (need_mask || c == 0.f) {
                const int last = a.causal ? min(a.N, row + 1) : a.N;
                mask_row(sr, c, need_mask ? max(0, min(kBN, last - key0)) : kBN);
            }
            const float r_ext = (cs >= 0.f) ? row_extreme<true>(sr) : row_extreme<false>(sr);
            const float m_tile = r_ext * cs;
            // PV of the previous block (phase blocks-1) must be complete before a
            // half of P_t is rewritten (pa: keys 0-63, pb: keys 64-127 and O_t).
            const bool prev = blocks > 0;
            const uint32_t par = (blocks - 1) & 1;
            float alpha = 1.f;
            if (m_ref == -INFINITY) {
                m_ref = m_tile;
            } else if (m_tile > m_ref + rescale_threshold<kF16>()) {
                alpha = ex2(m_ref - m_tile);
                m_ref = m_tile;
            }
            const float negm = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const uint64_t negm2 = f2_pack(negm, negm);
            const float top_err = top_rounding_error<kF16>(r_ext, cs, negm);
            uint64_t acc[4] = {0, 0, 0, 0};   // +0.0f pairs
            if (prev && !wait_warp(pa_done, par)) { ok = false; break; }
            tc_fence_after();
            p_half_to_tmem<kF16>(sr, 0, c2, negm2, acc, tP);
            // Rescale O_t after the first half of the exponentials, so the wait for
            // the previous block's PV overlaps them; it must land before PV(i).
            bool pb_seen = false;
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                if (prev && !wait_warp(pb_done, par)) { ok = false; break; }
                pb_seen = true;
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < kD / 32; ++ch) {
                    uint32_t orow[32];
                    tmem_ld32(tO + ch * 32, orow);
#pragma unroll
                    for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st32(tO + ch * 32, orow);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_half);
            if (prev && !pb_seen && !wait_warp(pb_done, par)) { ok = false; break; }
            tc_fence_after();
            p_half_to_tmem<kF16>(sr, 1, c2, negm2, acc, tP);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_full);
            ++blocks;
            const uint64_t s01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
            float sum0, sum1;
            f2_unpack(s01, sum0, sum1);
            l = l * alpha + (sum0 + sum1);
            l_o = l_o * alpha + (sum0 + sum1) + top_err;
        }
        if (!ok) break;
        // epilogue: O / l -> bf16 through the staging buffer and TMA, LSE in natural log
        if (!wait_warp(pb_done, (blocks - 1) & 1)) { ok = false; break; }   // the unit's last PV is complete
        tc_fence_after();
        const float l_safe = (l > 0.f) ? l : 1.f;
        const float inv = 1.f / ((l_o > 0.f) ? l_o : 1.f);
        uint32_t ov[kD];
        uint32_t (&h0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ov[0]);
        uint32_t (&h1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ov[32]);
        tmem_ld32(tO, h0);
        tmem_ld32(tO + 32, h1);
        tc_fence_before();
        if (lane == 0) bulk_wait_read0();   // the previous unit's store has read the staging rows
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) {     // 16-byte chunk = 8 output columns
            const int col = q * 8;
            uint4 w;
            w.x = pack2<kF16>(__uint_as_float(ov[col + 0]) * inv, __uint_as_float(ov[col + 1]) * inv);
            w.y = pack2<kF16>(__uint_as_float(ov[col + 2]) * inv, __uint_as_float(ov[col + 3]) * inv);
            w.z = pack2<kF16>(__uint_as_float(ov[col + 4]) * inv, __uint_as_float(ov[col + 5]) * inv);
            w.w = pack2<kF16>(__uint_as_float(ov[col + 6]) * inv, __uint_as_float(ov[col + 7]) * inv);
            st_shared16(erow + ((q ^ swz) << 4), w);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {   // this warp's 32 rows; the next epilogue waits for the read
            tma_store_4d(tm_o, ewarp, 0, tile_row0 + wq * 32, u.h, u.b);
            bulk_commit();
        }
        __syncwarp();
        if (row < a.N) a.lse[(int64_t)u.bh * a.N + row] = (m_ref + log2f(l_safe)) * 0.69314718055994531f;
    }
    if (lane == 0) bulk_wait0();   // this warp's O stores are complete
}

__device__ void init_barriers(uint64_t* bars) {
    for (int qb = 0; qb < 2; ++qb) {
        mbar_init(&bars[kBarQFull + qb], 1);
        mbar_init(&bars[kBarQEmpty + qb], 2);                // one commit per MMA stream
    }
    for (int t = 0; t < 2; ++t) {
        mbar_init(&bars[kBarSFull + t], 1);
        mbar_init(&bars[kBarSFree + t], kBM);
        mbar_init(&bars[kBarPHalf + t], kBM);
        mbar_init(&bars[kBarPFull + t], kBM);
        mbar_init(&bars[kBarPaDone + t], 1);
        mbar_init(&bars[kBarPbDone + t], 1);
        mbar_init(&bars[kBarDrain + t], 1);
    }
    mbar_init(&bars[kBarNever], 1);
    for (int sl = 0; sl < kUnitRing; ++sl) {
        mbar_init(&bars[kBarUnitFull + sl], 1);
        mbar_init(&bars[kBarUnitEmpty + sl], kUnitReaders);
    }
    for (int s = 0; s < Cfg::kStages; ++s) {
        mbar_init(&bars[kBarKV + s], 1);
        mbar_init(&bars[kBarKV + Cfg::kStages + s], 2);      // one commit per MMA stream
    }
}

}  // namespace d64

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_d64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const KernelArgs a) {
    using C = d64::Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem;
    uint8_t* sEpi = smem + C::kOffEpi;
    uint8_t* sKV = smem + C::kOffKV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);   // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile int* member = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 12);   // holds the counter slot
    const UnitRing ring{bars + d64::kBarUnitFull, bars + d64::kBarUnitEmpty,
                        reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16)};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        d64::init_barriers(bars);
        *abort_flag = 0;
        *member = 0;
        fence_mbar_init();
    }
    if (warp == kWarpProducer && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    if (warp == kWarpMma0) {
        tmem_alloc(tmem_slot, kTmemColsPerTile);
        tmem_alloc(tmem_slot + 1, kTmemColsPerTile);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem0 = tmem_slot[0], tmem1 = tmem_slot[1];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < kWarpProducer) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        d64::softmax_role<kF16>(warp < 4 ? tmem0 : tmem1, warp / 4, warp % 4, lane, bars, ring, abort_flag, sEpi, &tm_o, a);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (warp == kWarpProducer) {
            if (lane == 0) d64::producer(&tm_q, &tm_k, &tm_v, sQ, sKV, bars, ring, abort_flag, member, a);
            __syncwarp();
        } else if (warp == kWarpMma0 || warp == kWarpMma1) {
            const int t = warp - kWarpMma0;
            if (lane == 0) d64::mma_issuer<kF16>(t ? tmem1 : tmem0, t, sQ, sKV, bars, ring, abort_flag, a);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma0) {
        tmem_dealloc(tmem0, kTmemColsPerTile);
        tmem_dealloc(tmem1, kTmemColsPerTile);
    }
    if (threadIdx.x == 0 && *member) sched_release(a.sched);
}

}  // namespace
}  // namespace bos
