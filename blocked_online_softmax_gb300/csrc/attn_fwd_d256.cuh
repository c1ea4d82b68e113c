// Attention forward for head dimensions 136-256 (sm_103a). Included once, from
// attn_fwd_sm103.cu, after the shared pieces (scheduler, waits, softmax
// arithmetic); it is not a header for other files.
//
// Same method as the d = 128 kernel ("4.4 Writing GPU Kernels with Triton",
// Kernel 4 "A Simplified FlashAttention"), laid out for a 256-column O. A
// 128-row tile's O alone takes 256 of the 512 tensor-memory columns, so a CTA
// holds one Q tile (work unit = 128 query rows of one (batch, head)) and the
// other 256 columns hold S twice: S(g) is computed into buffer g % 2 while
// the softmax works on S(g-1) in the other. The softmax writes P(g) back as
// bf16 pairs over the first 64 columns of its own S buffer, so O += P V is a
// tensor-memory-A MMA whose N is the whole head width: 128 x 256 x 16 steps
// run at the tensor core's full rate even from one issuing thread. One MMA
// stream issues S(0), S(1), PV(0), S(2), PV(1), ...; S(g+2) overwrites buffer
// g % 2 only after PV(g) has read P(g) (in-order execution of one thread's
// MMAs).
//
// Shared memory: Q (64 KB), a ring of four 32 KB slots, O staging (32 KB).
// K tiles travel as two d-halves and V tiles as two key-halves, one slot
// each, in the order the stream reads them (K one block ahead of V), and each
// half is released as soon as the MMAs reading it complete.
//
// Head dims below 256 run on the same code: the tensor maps describe the
// caller's d columns, 64-column boxes past d are neither loaded nor stored,
// the S contraction stops at the last loaded box (columns in it past d load as
// zero) and PV's N covers the loaded boxes only.

namespace bos {
namespace {

namespace d256 {

constexpr int kD = 256;
constexpr int kThreads = 192;        // warps 0-3 softmax (thread = query row), 4 producer, 5 MMA + TMEM owner
constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSBuf = 128;  // S buffer b at column 128 b (fp32; P(g) over its first 64 columns)
constexpr uint32_t kTmemO = 256;     // O, fp32, up to 256 columns
constexpr int kUnitReaders = 1 + 4;  // the MMA thread and the four softmax warps

enum : int {
    kBarQFull = 0,      // the unit's Q tile has landed (TMA transaction count)
    kBarQEmpty = 1,     // the unit's last S is complete (MMA commit)
    kBarSFull = 2,      // [2] S(g) complete in buffer g % 2 (MMA commit)
    kBarPFull = 4,      // [2] P(g) is in buffer g % 2 and O is rescaled (128 arrivals)
    kBarPvDone = 6,     // PV(g) complete (MMA commit, one phase per block)
    kBarDrain = 7,      // every MMA of the stream complete (final commit)
    kBarNever = 8,      // never signalled (test hook)
    kBarUnitFull = 9,   // [kUnitRing]
    kBarUnitEmpty = 13, // [kUnitRing]
    kBarKV = 17,        // kv_full[kStages], then kv_empty[kStages]
};

struct Cfg {
    static constexpr int kBoxBytes = kBN * 64 * 2;           // 128 rows x 64 columns bf16: 16 KB
    static constexpr int kSlotBytes = 2 * kBoxBytes;         // half a K tile (128 keys x 128 d) or half a V
                                                             // tile (64 keys x 256 d): 32 KB
    static constexpr int kStages = 4;
    static constexpr int kEpiBytes = 32 * 64 * 2;            // one warp's 32 rows x 64 columns of O: 4 KB
    // shared memory: Q (4 boxes) | ring | O staging [4 warps][2] | barriers | misc
    static constexpr int kOffKV = 4 * kBoxBytes;
    static constexpr int kOffEpi = kOffKV + kStages * kSlotBytes;
    static constexpr int kOffBar = kOffEpi + 4 * 2 * kEpiBytes;
    static constexpr int kNumBars = kBarKV + 2 * kStages;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, unit ring [4]
    static constexpr int kSmemBytes = kOffMisc + 32 + 1024;  // + alignment slack
};
static_assert(Cfg::kSmemBytes <= 232448, "shared memory per CTA");

// Work unit k: 128 query rows. Causal: heaviest first within each group of
// heads (as the d <= 128 kernels order their 256-row units); non-causal:
// head-major.
__device__ __forceinline__ Unit decode_tile_unit(int k, const KernelArgs& a) {
    Unit u;
    int q;
    if (a.causal) {
        const int gu = a.group * a.U;
        const int h0 = (k / gu) * a.group;
        const int gh = min(a.group, a.BH - h0);
        const int kk = k - (k / gu) * gu;
        q = a.U - 1 - kk / gh;
        u.bh = h0 + kk % gh;
    } else {
        u.bh = k / a.U;
        q = k % a.U;
    }
    u.b = u.bh / a.H;
    u.h = u.bh - u.b * a.H;
    u.row0 = q * kBM;
    const int nkv = (a.N + kBN - 1) / kBN;
    u.n = a.causal ? min(q + 1, nkv) : nkv;
    u.first0 = 0;
    return u;
}

// 64-column boxes of the head dimension that hold columns < d.
__device__ __forceinline__ int head_boxes(const KernelArgs& a) { return (a.d + 63) / 64; }

__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint8_t* sQ,
                         uint8_t* sKV, uint64_t* bars, const UnitRing& ring, volatile int* abort_flag,
                         volatile int* member, const KernelArgs& a) {
    uint64_t* kv_full = bars + kBarKV;
    uint64_t* kv_empty = bars + kBarKV + Cfg::kStages;
    const int total = a.BH * a.U;
    const int nb = head_boxes(a);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;   // ring loads whose completion is not yet observed
    int q_parity = -1;                             // parity of the last Q load's phase, -1 before any
    bool ok = true;
    auto take_slot = [&](uint32_t bytes) -> uint8_t* {
        if (!wait_or_abort(&kv_empty[stage], phase ^ 1, a.wait_limit_ns, abort_flag)) return nullptr;
        mbar_arrive_expect_tx(&kv_full[stage], bytes);
        return sKV + stage * Cfg::kSlotBytes;
    };
    auto advance = [&]() {
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == Cfg::kStages) { stage = 0; phase ^= 1; }
    };
    // half hf of K tile j: head columns 128 hf .. 128 hf + 127 (the boxes below d)
    auto load_k = [&](int j, int hf, const Unit& u) -> bool {
        const int b0 = 2 * hf, b1 = min(2 * hf + 2, nb);
        uint8_t* dst = take_slot((uint32_t)((b1 - b0) * Cfg::kBoxBytes));
        if (!dst) return false;
        for (int bx = b0; bx < b1; ++bx)
            tma_load_4d(dst + (bx - b0) * Cfg::kBoxBytes, tm_k, &kv_full[stage], bx * 64, j * kBN, u.h, u.b);
        advance();
        return true;
    };
    // half hf of V tile j: keys 64 hf .. 64 hf + 63 of the block, every head column below d
    auto load_v = [&](int j, int hf, const Unit& u) -> bool {
        uint8_t* dst = take_slot((uint32_t)(nb * Cfg::kBoxBytes / 2));
        if (!dst) return false;
        for (int bx = 0; bx < nb; ++bx)
            tma_load_4d(dst + bx * (Cfg::kBoxBytes / 2), tm_v, &kv_full[stage], bx * 64, j * kBN + hf * 64, u.h,
                        u.b);
        advance();
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
        const Unit u = decode_tile_unit(k, a);
        // Q once the previous unit's last S is done with the buffer
        if (!wait_or_abort(&bars[kBarQEmpty], (r & 1) ^ 1, a.wait_limit_ns, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kBarQFull], (uint32_t)(nb * Cfg::kBoxBytes));
        q_parity = r & 1;
        for (int bx = 0; bx < nb; ++bx)
            tma_load_4d(sQ + bx * Cfg::kBoxBytes, tm_q, &bars[kBarQFull], bx * 64, u.row0, u.h, u.b);
        // key block i is j = n-1-i; the stream reads K(0), K(1), V(0), K(2), V(1), ...
        if (!load_k(u.n - 1, 0, u) || !load_k(u.n - 1, 1, u)) { ok = false; break; }
        for (int i = 0; i < u.n && ok; ++i) {
            if (i + 1 < u.n && (!load_k(u.n - 2 - i, 0, u) || !load_k(u.n - 2 - i, 1, u))) { ok = false; break; }
            if (!load_v(u.n - 1 - i, 0, u) || !load_v(u.n - 1 - i, 1, u)) { ok = false; break; }
        }
    }
    // Every copy this thread started must land before the CTA may exit.
    for (int s = 0; s < Cfg::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait(&kv_full[s], (issued_parity >> s) & 1u, kDrainLimitNs);
    if (q_parity >= 0) mbar_wait(&bars[kBarQFull], (uint32_t)q_parity, kDrainLimitNs);
}

// Part of S(g) = Q K^T into the accumulator at `d_tmem`: the 16-column steps of
// head-dimension boxes box0 .. box1-1, Q from its buffer, K from the half-tile
// slot `sKh` that holds those boxes. The first half starts the accumulation.
template <bool kF16>
__device__ __forceinline__ void issue_s_half(uint32_t d_tmem, const uint8_t* sQ, const uint8_t* sKh, int box0,
                                             int box1, bool first_half) {
    constexpr uint32_t idesc = idesc_f32acc(kBM, kBN, false, false, kF16);
    const uint32_t qa = smem_u32(sQ), ka = smem_u32(sKh);
#pragma unroll 1
    for (int bx = box0; bx < box1; ++bx) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // 32-byte K step within a 128-byte swizzled row
            const uint32_t qoff = bx * Cfg::kBoxBytes + kk * 32;
            const uint32_t koff = (bx - box0) * Cfg::kBoxBytes + kk * 32;
            mma_ss(d_tmem, sdesc_sw128(qa + qoff, 16, 1024), sdesc_sw128(ka + koff, 16, 1024), idesc,
                   (first_half && bx == box0 && kk == 0) ? 0u : 1u);
        }
    }
}

// O (+)= P(g)[:, keys 64 hf .. 64 hf + 63] * V half: P from the buffer's
// tensor-memory columns, V (MN-major, nb boxes of 64 keys x 64 columns, 8 KB
// apart) from shared memory; N = 64 nb.
__device__ __forceinline__ void issue_pv_half(uint32_t tm, uint32_t sbuf, const uint8_t* sVh, int hf, uint32_t idesc,
                                              bool accumulate) {
    const uint32_t va = smem_u32(sVh);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)   // 16 keys per step: 8 P columns, 16 V rows (2048 bytes)
        mma_ts(tm + kTmemO, tm + sbuf + (hf * 4 + kk) * 8, sdesc_sw128(va + kk * 2048, Cfg::kBoxBytes / 2, 1024),
               idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// The MMA stream, one thread: for each unit S(0), S(1), PV(0), S(2), PV(1), ...,
// PV(n-1), with the CTA's blocks numbered g = 0, 1, ... across units (S(g) in
// buffer g % 2).
template <bool kF16>
__device__ void mma_issuer(uint32_t tm, const uint8_t* sQ, const uint8_t* sKV, uint64_t* bars, const UnitRing& ring,
                           volatile int* abort_flag, const KernelArgs& a) {
    uint64_t* kv_full = bars + kBarKV;
    uint64_t* kv_empty = bars + kBarKV + Cfg::kStages;
    const uint64_t lim = a.wait_limit_ns;
    const int total = a.BH * a.U;
    const int nb = head_boxes(a);
    const uint32_t idesc_pv = idesc_f32acc(kBM, 64 * nb, false, true, kF16);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t s_count = 0;    // S blocks issued so far (g of the next S)
    uint32_t pv_count = 0;   // PV blocks issued so far (g of the next PV)
    bool ok = true;
    if (a.test_stall && !wait_or_abort(bars + kBarNever, 0, lim, abort_flag)) ok = false;
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
        const Unit u = decode_tile_unit(k, a);
        for (int i = -1; i < u.n; ++i) {
            if (i + 1 < u.n) {   // S(i+1)
                int k0, k1;
                if (!next_stage(k0) || !next_stage(k1)) { ok = false; break; }
                if (i + 1 == 0 && !wait_or_abort(&bars[kBarQFull], r & 1, lim, abort_flag)) { ok = false; break; }
                const uint32_t sbuf = (s_count & 1) * kTmemSBuf;
                tc_fence_after();
                issue_s_half<kF16>(tm + sbuf, sQ, sKV + k0 * Cfg::kSlotBytes, 0, min(2, nb), true);
                mma_commit(&kv_empty[k0]);
                issue_s_half<kF16>(tm + sbuf, sQ, sKV + k1 * Cfg::kSlotBytes, 2, nb, false);
                mma_commit(&kv_empty[k1]);
                mma_commit(&bars[kBarSFull + (s_count & 1)]);
                if (i + 1 == u.n - 1) mma_commit(&bars[kBarQEmpty]);
                ++s_count;
            }
            if (i < 0) continue;
            int v0, v1;   // PV(i)
            if (!next_stage(v0) || !next_stage(v1)) { ok = false; break; }
            const uint32_t pb = pv_count & 1;
            if (!wait_or_abort(&bars[kBarPFull + pb], (pv_count >> 1) & 1, lim, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_pv_half(tm, pb * kTmemSBuf, sKV + v0 * Cfg::kSlotBytes, 0, idesc_pv, i > 0);
            mma_commit(&kv_empty[v0]);
            issue_pv_half(tm, pb * kTmemSBuf, sKV + v1 * Cfg::kSlotBytes, 1, idesc_pv, true);
            mma_commit(&kv_empty[v1]);
            mma_commit(&bars[kBarPvDone]);
            ++pv_count;
        }
    }
    // Every MMA this thread issued must complete before tensor memory is freed.
    mma_commit(&bars[kBarDrain]);
    mbar_wait(&bars[kBarDrain], 0, kDrainLimitNs);
}

// Softmax warpgroup (thread = query row = TMEM lane). Per block g: read S(g),
// mask, exponentiate against the reference max, write P(g) over the buffer,
// wait for PV(g-1) (so O may be rescaled, and so this role never falls two
// phases behind the PV barrier), rescale O when the max moved, hand P(g) to
// the stream. After a unit's last block: O / l as bf16, one 64-column slice at
// a time, through two 4 KB staging buffers per warp and TMA; LSE.
template <bool kF16>
__device__ void softmax_role(uint32_t tm, int wq, int lane, uint64_t* bars, const UnitRing& ring,
                             volatile int* abort_flag, uint8_t* sEpi, const CUtensorMap* tm_o, const KernelArgs& a) {
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t lane_base = tm + ((uint32_t)(wq * 32) << 16);
    const uint32_t tO = lane_base + kTmemO;
    const int row_in_tile = wq * 32 + lane;
    uint8_t* ewarp = sEpi + wq * 2 * Cfg::kEpiBytes;   // this warp's two staging buffers (1024-byte aligned)
    const int swz = lane & 7;
    const int nb = head_boxes(a);
    const float c = a.scale_log2;
    const float cs = (c == 0.f) ? 1.f : c;   // with c == 0 every score is replaced by 0 (mask_row), scaled by 1
    const uint64_t c2 = f2_pack(cs, cs);
    const int total = a.BH * a.U;
    uint32_t blocks = 0;   // g of the next block
    uint32_t slices = 0;   // O slices stored so far; consecutive slices alternate staging buffers
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
        const Unit u = decode_tile_unit(k, a);
        const int tile_row0 = u.row0;
        const int row = tile_row0 + row_in_tile;
        float m_ref = -INFINITY;   // max the exponentials are taken against (base-2 units)
        float l = 0.f;     // sum of the fp32 probabilities (LSE)
        float l_o = 0.f;   // the same plus each block's top-term rounding error (normalises O)
        for (int i = 0; i < u.n; ++i) {
            const int j = u.n - 1 - i;
            const uint32_t g = blocks;
            const uint32_t tS = lane_base + (g & 1) * kTmemSBuf;
            if (!wait_warp(&bars[kBarSFull + (g & 1)], (g >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128(tS, sr);
            const int key0 = j * kBN;
            const bool need_mask = (key0 + kBN > a.N) || (a.causal && key0 + kBN - 1 > tile_row0);
            if (need_mask || c == 0.f) {
                const int last = a.causal ? min(a.N, row + 1) : a.N;
                mask_row(sr, c, need_mask ? max(0, min(kBN, last - key0)) : kBN);
            }
            const float r_ext = (cs >= 0.f) ? row_extreme<true>(sr) : row_extreme<false>(sr);
            const float m_tile = r_ext * cs;
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
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {   // all 128 keys as bf16 pairs over the buffer's first 64 columns
                uint32_t pk[16];
                exp_pack<kF16>(sr, ch, c2, negm2, acc, pk);
                tmem_st16(tS + ch * 16, pk);
            }
            if (g > 0 && !wait_warp(&bars[kBarPvDone], (g - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int ch = 0; ch < 2 * nb; ++ch) {
                    uint32_t orow[32];
                    tmem_ld32(tO + ch * 32, orow);
#pragma unroll
                    for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st32(tO + ch * 32, orow);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars[kBarPFull + (g & 1)]);
            ++blocks;
            const uint64_t s01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
            float sum0, sum1;
            f2_unpack(s01, sum0, sum1);
            l = l * alpha + (sum0 + sum1);
            l_o = l_o * alpha + (sum0 + sum1) + top_err;
        }
        if (!ok) break;
        // epilogue: the unit's last PV must be complete
        if (!wait_warp(&bars[kBarPvDone], (blocks - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const float l_safe = (l > 0.f) ? l : 1.f;
        const float inv = 1.f / ((l_o > 0.f) ? l_o : 1.f);
#pragma unroll 1
        for (int s = 0; s < nb; ++s) {
            uint32_t o0[32], o1[32];   // this slice's 64 columns of O
            tmem_ld32(tO + s * 64, o0);
            tmem_ld32(tO + s * 64 + 32, o1);
            uint8_t* ebuf = ewarp + (slices++ & 1) * Cfg::kEpiBytes;
            const uint32_t erow = smem_u32(ebuf + lane * 128);
            if (lane == 0) bulk_wait_read1();   // the store before last (same buffer) is done reading
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q) {   // 16-byte chunk = 8 output columns
                const uint32_t* ov = (q < 4) ? o0 + q * 8 : o1 + (q - 4) * 8;
                uint4 w;
                w.x = pack2<kF16>(__uint_as_float(ov[0]) * inv, __uint_as_float(ov[1]) * inv);
                w.y = pack2<kF16>(__uint_as_float(ov[2]) * inv, __uint_as_float(ov[3]) * inv);
                w.z = pack2<kF16>(__uint_as_float(ov[4]) * inv, __uint_as_float(ov[5]) * inv);
                w.w = pack2<kF16>(__uint_as_float(ov[6]) * inv, __uint_as_float(ov[7]) * inv);
                st_shared16(erow + ((q ^ swz) << 4), w);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {   // this warp's 32 rows (rows past N are clipped)
                tma_store_4d(tm_o, ebuf, s * 64, tile_row0 + wq * 32, u.h, u.b);
                bulk_commit();
            }
            __syncwarp();
        }
        tc_fence_before();
        if (row < a.N) a.lse[(int64_t)u.bh * a.N + row] = (m_ref + log2f(l_safe)) * 0.69314718055994531f;
    }
    if (lane == 0) bulk_wait0();   // this warp's O stores are complete
}

__device__ void init_barriers(uint64_t* bars) {
    mbar_init(&bars[kBarQFull], 1);
    mbar_init(&bars[kBarQEmpty], 1);
    for (int b = 0; b < 2; ++b) {
        mbar_init(&bars[kBarSFull + b], 1);
        mbar_init(&bars[kBarPFull + b], kBM);
    }
    mbar_init(&bars[kBarPvDone], 1);
    mbar_init(&bars[kBarDrain], 1);
    mbar_init(&bars[kBarNever], 1);
    for (int sl = 0; sl < kUnitRing; ++sl) {
        mbar_init(&bars[kBarUnitFull + sl], 1);
        mbar_init(&bars[kBarUnitEmpty + sl], kUnitReaders);
    }
    for (int s = 0; s < Cfg::kStages; ++s) {
        mbar_init(&bars[kBarKV + s], 1);
        mbar_init(&bars[kBarKV + Cfg::kStages + s], 1);     // one MMA stream
    }
}

}  // namespace d256

template <bool kF16>
__global__ void __launch_bounds__(d256::kThreads, 1)
attn_fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const KernelArgs a) {
    using C = d256::Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + C::kOffKV;
    uint8_t* sEpi = smem + C::kOffEpi;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile int* member = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 12);   // holds the counter slot
    const UnitRing ring{bars + d256::kBarUnitFull, bars + d256::kBarUnitEmpty,
                        reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16)};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        d256::init_barriers(bars);
        *abort_flag = 0;
        *member = 0;
        fence_mbar_init();
    }
    if (warp == d256::kWarpProducer && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    if (warp == d256::kWarpMma) {
        tmem_alloc(tmem_slot, d256::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot[0];
    // programmatic stream serialization, as in the other forward kernels
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < d256::kWarpProducer) {
        d256::softmax_role<kF16>(tmem, warp, lane, bars, ring, abort_flag, sEpi, &tm_o, a);
    } else if (warp == d256::kWarpProducer) {
        if (lane == 0) d256::producer(&tm_q, &tm_k, &tm_v, sQ, sKV, bars, ring, abort_flag, member, a);
        __syncwarp();
    } else {
        if (lane == 0) d256::mma_issuer<kF16>(tmem, sQ, sKV, bars, ring, abort_flag, a);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == d256::kWarpMma) tmem_dealloc(tmem, d256::kTmemCols);
    if (threadIdx.x == 0 && *member) sched_release(a.sched);
}

}  // namespace
}  // namespace bos
