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
//    share every K/V tile. CTAs are persistent (one per SM) and take units from
//    a per-launch global counter; units are numbered heaviest first (for causal
//    masking, within groups of heads whose K and V fit a slice of L2), so the
//    triangle of work balances itself and SMs that run slower simply take
//    fewer units.
//  * Warp roles (384 threads): warpgroups 0 and 1 run the softmax of Q tile 0
//    and Q tile 1, one thread per query row, with 208 registers each after a
//    setmaxnreg split; warp 8 takes units and issues TMA loads (Q per unit, then
//    K_j, V_j into a multi-stage ring); warps 9 and 10 each issue the tcgen05
//    MMAs of one Q tile from one thread. A stream executes its MMAs in issue
//    order, and each tile's products wait on its own softmax; with a stream
//    per tile, one tile's waits do not hold back the other tile's MMAs.
//  * Tensor memory: one 256-column allocation per Q tile holding S_t = Q_t K^T
//    (fp32, 128 columns) and O_t (fp32, d columns). Keys 0-63 of P_t are written
//    back as bf16 over S_t's first 32 columns and multiplied from there (TS
//    MMA); keys 64-127 go to a swizzled shared-memory buffer (SS MMA). Because
//    only the first half aliases S_t, each stream issues S(i), PV_lo(i), S(i+1),
//    PV_hi(i): the next scores are computed while the softmax is still
//    exponentiating the second half of the block.
//  * Key blocks are visited from the last to the first, so the masked blocks
//    (the causal diagonal, the ragged tail past N) come first. Causal: blocks
//    past a tile's diagonal are skipped, as in the page's loop bound.
//  * The running max is only moved (and O, l rescaled) when a block's max
//    exceeds it by more than 32 in log2 units (8 with fp16 P); otherwise
//    exponentials are taken against the older, smaller max (p <= 2^32). O/l
//    and LSE are unchanged in exact arithmetic, and the O rescale through
//    tensor memory becomes rare even for large logits.
//  * Epilogue: O / l as bf16 through the tile's shared P buffer, one TMA store
//    per warp (32 rows), fp32 LSE with plain stores.
//  * Every wait is bounded in wall time: on expiry the kernel records a status,
//    drains its own copies and MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
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
// warps 0-3: softmax of Q tile 0, warps 4-7: softmax of Q tile 1 (warp w reads
// TMEM lanes 32*(w%4)..+31, so each warpgroup covers the 128 rows of its tile);
// warpgroup 2: warp 8 TMA producer, warp 9 MMA issuer and TMEM owner.
// Registers after launch (384 x 168): 128 x (208 + 208 + 88) = 64512.
constexpr int kThreads = 384;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma0 = 9;         // MMA stream of Q tile 0; also owns TMEM allocation
constexpr int kWarpMma1 = 10;        // MMA stream of Q tile 1
constexpr int kRegsSoftmax = 208;
constexpr int kRegsControl = 88;
// Stale-max threshold (log2 units): the reference max moves (and O, l are
// rescaled) only when a block's max exceeds it by more than this, so every
// probability is at most 2^T. bf16 P reaches 2^127, so it takes T = 32: O and
// l then stay finite in fp32 while N * 2^32 * max|V| < 2^128 (max|V| below
// ~10^24 at N = 2^16). fp16 P ends below 2^16, so it keeps T = 8.
template <bool kF16>
constexpr float rescale_threshold() { return kF16 ? 8.0f : 32.0f; }
// Each Q tile has its own 256-column TMEM allocation: S at column 0 (P overlays
// its first 64 columns as packed bf16), O at column 128. MMAs issued by one
// thread run in issue order; one thread issuing 128 x 128 x 16 MMAs back to
// back keeps the tensor core at 94-100 % of its rate (measured on this GPU),
// and two threads issuing at once share it.
constexpr uint32_t kTmemColsPerTile = 256;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 128;
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;         // 1 s

// Barriers (mbarriers in shared memory), by index.
enum : int {
    kBarQFull = 0,      // the unit's two Q tiles have landed (TMA transaction count)
    kBarQEmpty = 1,     // both streams' last S of the unit is complete (two MMA commits)
    kBarSFull = 2,      // [2] S_t complete (MMA commit)
    kBarPHalf = 4,      // [2] keys 0-63 of P_t are in tensor memory (128 arrivals)
    kBarPFull = 6,      // [2] keys 64-127 of P_t are in shared memory (128 arrivals)
    kBarPbDone = 8,     // [2] PV_t for keys 64-127 complete: O_t current, P_t's shared half free (MMA commit)
    kBarDrain = 10,     // [2] every MMA of stream t complete (final commit)
    kBarNever = 12,     // never signalled (test hook)
    kBarUnitFull = 13,  // [kUnitRing] the producer has written the next unit index (1 arrival)
    kBarUnitEmpty = 17, // [kUnitRing] every role has read it (2 MMA threads + 8 softmax warps)
    kBarKV = 21,        // kv_full[kStages], then kv_empty[kStages]
};
constexpr int kUnitRing = 4;              // unit indices handed from the producer to the other roles
constexpr int kUnitReaders = 2 + 8;

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kBN * D * 2;          // one bf16 Q, K or V tile
    static constexpr int kPbBytes = kBM * 64 * 2;           // keys 64-127 of P_t (bf16), one 128-byte row per query
    // K/V ring depth. V_i's stage stays busy until the PV of keys 64-127, which a
    // stream issues after S(i+1); with four 32 KB stages (d = 128) every load has
    // about a block of lead.
    static constexpr int kStages = 4;
    static constexpr int kBoxes = D / 64;                   // 64-column TMA boxes per tile
    // shared memory: Q tiles [2] | second halves of P [2] | K/V ring | barriers | misc
    static constexpr int kOffPb = 2 * kTileBytes;
    static constexpr int kOffKV = kOffPb + 2 * kPbBytes;
    static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
    static constexpr int kNumBars = kBarKV + 2 * kStages;
    // tmem slots [2], abort flag, member flag, unit ring indices [4], decoded units [4][8]
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 32 + kUnitRing * 32 + 1024;  // + alignment slack
};

struct KernelArgs {
    int BH, H, N, U, causal;
    int d;       // the caller's head dim (the kernel's width may be larger)
    int group;   // causal: heads per scheduling group (units run heaviest first within a group)
    float scale_log2;
    __nv_bfloat16* o;
    float* lse;
    uint64_t wait_limit_ns;
    int test_stall;   // test hook: the MMA thread first waits on a barrier nothing signals
    unsigned int* sched;   // this launch's work counter and exit counter (both zero at launch)
};

}  // namespace

// Sticky device-side status: 0, or the attn_status of the first failure.
__device__ int g_attn_device_status;

// Work counters. Each launch draws the next slot round-robin; a slot is four
// words: units taken, CTAs finished, and the 64-bit tag of the launch that
// holds it (its %gridid + 1; 0 = free). A CTA claims the slot before it takes
// a unit; the last CTA out returns the counters to zero and frees the slot. A
// launch that finds its slot still held by another launch (only possible with
// more than kSchedSlots launches in flight on the device) takes no units and
// records ATTN_ERR_SCHED_BUSY instead of sharing the other launch's counter.
constexpr int kSchedSlots = 4096;
constexpr int kSchedWords = 4;
__device__ __align__(16) unsigned int g_attn_sched[kSchedWords * kSchedSlots];

namespace {

// Bounded wait that also gives up as soon as another role has aborted. The
// waiting thread sleeps inside try_wait (up to ~0.5 ms per try) instead of
// spinning, so waiting warps leave the issue slots to the softmax warps that
// share their SM sub-partition.
constexpr uint32_t kSuspendNs = 500000;

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint32_t hint = (uint32_t)(limit_ns < kSuspendNs ? limit_ns : kSuspendNs);
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, hint)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicCAS(&g_attn_device_status, 0, (int)ATTN_ERR_TIMEOUT);
            return false;
        }
    }
}

// The launch's tag in its work-counter slot: unique per launch in this context.
__device__ __forceinline__ unsigned long long launch_tag() {
    unsigned long long g;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
    return g + 1ull;
}

// Claims this launch's counter slot (one thread per CTA, before its first
// unit). False if another launch still holds it; the status is then recorded.
__device__ __forceinline__ bool sched_claim(unsigned int* slot) {
    const unsigned long long me = launch_tag();
    const unsigned long long held =
        atomicCAS(reinterpret_cast<unsigned long long*>(slot + 2), 0ull, me);
    if (held == 0ull || held == me) return true;
    atomicCAS(&g_attn_device_status, 0, (int)ATTN_ERR_SCHED_BUSY);
    return false;
}

// Called once by every CTA that claimed the slot, after all its work: the last
// one zeroes the counters, then frees the slot for a later launch.
__device__ __forceinline__ void sched_release(unsigned int* slot) {
    __threadfence();
    if (atomicAdd(slot + 1, 1u) == gridDim.x - 1) {
        atomicExch(slot, 0u);
        atomicExch(slot + 1, 0u);
        __threadfence();
        atomicExch(reinterpret_cast<unsigned long long*>(slot + 2), 0ull);
    }
}

// Decoded work unit.
struct Unit {
    int bh, b, h, row0, n, first0;   // n key tiles for Q tile 1; Q tile 0 starts at iteration first0
};

__device__ __forceinline__ Unit decode_unit(int k, const KernelArgs& a) {
    Unit u;
    int q;
    if (a.causal) {            // heaviest first within each group of heads
        const int gu = a.group * a.U;
        const int h0 = (k / gu) * a.group;
        const int gh = min(a.group, a.BH - h0);
        const int kk = k - (k / gu) * gu;
        q = a.U - 1 - kk / gh;
        u.bh = h0 + kk % gh;
    } else {                   // head-major (every unit costs the same)
        u.bh = k / a.U;
        q = k % a.U;
    }
    u.b = u.bh / a.H;
    u.h = u.bh - u.b * a.H;
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

// The unit ring: the producer takes each unit index from the launch's global
// counter (units are numbered heaviest first, so CTAs that run faster simply
// take more of them; a CTA's first unit is its own index, which saves a global
// atomic on the start-up path) and hands it to the MMA and softmax roles in order.
// Index >= total means no work is left. Where `unit` is set, the producer
// also writes the decoded unit into the slot, so a reader can take it from
// shared memory instead of repeating the integer divisions at a unit
// change-over; the softmax warps and the MMA threads both do.
struct UnitRing {
    uint64_t* full;      // [kUnitRing] the producer has written the slot (1 arrival)
    uint64_t* empty;     // [kUnitRing] every reader has read it (kUnitReaders arrivals)
    volatile int* idx;   // [kUnitRing]
    volatile int* unit;  // [kUnitRing][8]: bh, b, h, row0, n, first0 of a unit < total (or null)
    // reader side: the r-th unit index of this CTA, or false if a wait failed
    __device__ __forceinline__ bool get(int r, int& k, uint64_t lim, volatile int* abort_flag) const {
        const int sl = r % kUnitRing;
        if (!wait_or_abort(&full[sl], (uint32_t)((r / kUnitRing) & 1), lim, abort_flag)) return false;
        k = idx[sl];
        return true;
    }
    // the decoded unit of slot r (after get, before release; only for an index < total)
    __device__ __forceinline__ Unit decoded(int r) const {
        const volatile int* p = unit + (r % kUnitRing) * 8;
        Unit u;
        u.bh = p[0];
        u.b = p[1];
        u.h = p[2];
        u.row0 = p[3];
        u.n = p[4];
        u.first0 = p[5];
        return u;
    }
    // producer side: the unit for slot sl, written before the slot's arrival
    __device__ __forceinline__ void put_decoded(int sl, const Unit& u) const {
        volatile int* p = unit + sl * 8;
        p[0] = u.bh;
        p[1] = u.b;
        p[2] = u.h;
        p[3] = u.row0;
        p[4] = u.n;
        p[5] = u.first0;
    }
    __device__ __forceinline__ void release(int r) const { mbar_arrive(&empty[r % kUnitRing]); }
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two values rounded to the forward's element type (bf16, or fp16 with kF16),
// lo in the low half.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (kF16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        return pack_bf16(lo, hi);
    }
}

// ------------------------------------------------------------------ roles

template <int D>
__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                         uint8_t* sQ, uint8_t* sKV, uint64_t* bars, const UnitRing& ring, volatile int* abort_flag,
                         volatile int* member, const KernelArgs& a) {
    using C = Cfg<D>;
    uint64_t* kv_full = bars + kBarKV;
    uint64_t* kv_empty = bars + kBarKV + C::kStages;
    const int total = a.BH * a.U;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;             // stages with a load whose completion is not yet observed
    uint32_t issued_parity = 0;           // parity of that load's phase, per stage
    int q_parity = -1;                    // parity of the last Q load's phase, -1 before any
    bool ok = true;
    // One K/V tile into the next ring stage.
    auto load_kv = [&](const CUtensorMap* tm, int j, const Unit& u) -> bool {
        if (!wait_or_abort(&kv_empty[stage], phase ^ 1, a.wait_limit_ns, abort_flag)) return false;
        mbar_arrive_expect_tx(&kv_full[stage], C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
            tma_load_4d(sKV + stage * C::kTileBytes + b * 16384, tm, &kv_full[stage], b * 64, j * kBN, u.h, u.b);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        return true;
    };
    for (int r = 0; ok; ++r) {
        const int sl = r % kUnitRing;
        if (!wait_or_abort(&bars[kBarUnitEmpty + sl], (uint32_t)((r / kUnitRing) & 1) ^ 1, a.wait_limit_ns,
                           abort_flag)) {
            ok = false;
            break;
        }
        // the first unit of CTA g is g (the grid never exceeds the unit count); the
        // counter hands out the rest. A CTA whose slot is held by another launch
        // takes no unit.
        int k;
        if (r == 0) {
            *member = sched_claim(a.sched) ? 1 : 0;
            k = *member ? (int)blockIdx.x : total;
        } else {
            k = (int)gridDim.x + (int)atomicAdd(a.sched, 1u);
        }
        Unit u{};
        if (k < total) {
            u = decode_unit(k, a);
            ring.put_decoded(sl, u);
        }
        ring.idx[sl] = k;
        mbar_arrive(&bars[kBarUnitFull + sl]);
        if (k >= total) break;
        // Q tiles first, once both streams' last S of the previous unit is done
        // with the buffer, then the unit's K/V stream.
        if (!wait_or_abort(&bars[kBarQEmpty], (r & 1) ^ 1, a.wait_limit_ns, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kBarQFull], 2 * C::kTileBytes);
        q_parity = r & 1;
        for (int t = 0; t < 2; ++t)
            for (int b = 0; b < C::kBoxes; ++b)
                tma_load_4d(sQ + t * C::kTileBytes + b * 16384, tm_q, &bars[kBarQFull], b * 64, u.row0 + t * kBM,
                            u.h, u.b);
        for (int i = 0; i < u.n && ok; ++i) {
            const int j = u.n - 1 - i;
            if (!load_kv(tm_k, j, u) || !load_kv(tm_v, j, u)) { ok = false; break; }
        }
    }
    // Every copy this thread started must land before the CTA may exit (on the
    // normal path they already have).
    for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait(&kv_full[s], (issued_parity >> s) & 1u, kDrainLimitNs);
    if (q_parity >= 0) mbar_wait(&bars[kBarQFull], (uint32_t)q_parity, kDrainLimitNs);
}

// S_t = Q_t K^T into the tile's TMEM allocation `tm`.
template <int D, bool kF16>
__device__ __forceinline__ void issue_s(uint32_t tm, const uint8_t* sQt, const uint8_t* sK) {
    constexpr uint32_t idesc = idesc_f32acc(kBM, kBN, false, false, kF16);
    const uint32_t qa = smem_u32(sQt), ka = smem_u32(sK);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;   // 64-column box, 32-byte K step
        mma_ss(tm + kTmemS, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc,
               kk > 0 ? 1u : 0u);
    }
}

// O_t (+)= P_t[:, keys 0-63] * V[keys 0-63, :], P from tensor memory (packed
// bf16 pairs over the first 32 columns of S_t).
template <int D, bool kF16>
__device__ __forceinline__ void issue_pv_lo(uint32_t tm, const uint8_t* sV, bool accumulate) {
    constexpr uint32_t idesc = idesc_f32acc(kBM, D, false, true, kF16);
    const uint32_t va = smem_u32(sV);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)       // 16 keys per step: 8 P columns, 16 V rows (2048 bytes)
        mma_ts(tm + kTmemO, tm + kTmemS + kk * 8, sdesc_sw128(va + kk * 2048, 16384, 1024), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
}

// O_t += P_t[:, keys 64-127] * V[keys 64-127, :], P from shared memory
// (K-major, 128-byte swizzle, one 128-byte row per query).
template <int D, bool kF16>
__device__ __forceinline__ void issue_pv_hi(uint32_t tm, const uint8_t* sPbt, const uint8_t* sV) {
    constexpr uint32_t idesc = idesc_f32acc(kBM, D, false, true, kF16);
    const uint32_t pa = smem_u32(sPbt), va = smem_u32(sV);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss(tm + kTmemO, sdesc_sw128(pa + kk * 32, 16, 1024), sdesc_sw128(va + (kk + 4) * 2048, 16384, 1024),
               idesc, 1u);
}

// One MMA stream: Q tile t's S_t = Q_t K^T and O_t += P_t V, issued by one
// thread into the tile's own TMEM allocation, in the order
//     S(i), PV_lo(i), S(i+1), PV_hi(i), PV_lo(i+1), S(i+2), ...
// PV_lo(i) reads keys 0-63 of P(i) from the first 32 columns of S_t, so S(i+1)
// may only overwrite S_t after it, and in-order execution within the stream
// guarantees that. Keys 64-127 of P(i) live in shared memory, so S(i+1) does
// not wait for the softmax to finish block i: the tensor core computes the next
// scores while the softmax is still writing the second half of P.
// Both streams walk the same K/V ring (K_j, V_j alternating); a stage is free
// once both have committed it.
template <int D, bool kF16>
__device__ void mma_issuer(uint32_t tm, int t, const uint8_t* sQ, const uint8_t* sPb, const uint8_t* sKV,
                           uint64_t* bars, const UnitRing& ring, volatile int* abort_flag, const KernelArgs& a) {
    using C = Cfg<D>;
    uint64_t* kv_full = bars + kBarKV;
    uint64_t* kv_empty = bars + kBarKV + C::kStages;
    uint64_t* s_full = bars + kBarSFull + t;
    uint64_t* p_half = bars + kBarPHalf + t;
    uint64_t* p_full = bars + kBarPFull + t;
    uint64_t* pb_done = bars + kBarPbDone + t;
    const uint64_t lim = a.wait_limit_ns;
    const int total = a.BH * a.U;
    const uint8_t* sQt = sQ + t * C::kTileBytes;
    const uint8_t* sPbt = sPb + t * C::kPbBytes;
    int stage = 0;
    uint32_t phase = 0, ph_phase = 0, pf_phase = 0;
    bool ok = true;
    if (t == 0 && a.test_stall && !wait_or_abort(bars + kBarNever, 0, lim, abort_flag)) ok = false;
    // the next ring stage in load order, once its tile has landed
    auto next_stage = [&](int& st) -> bool {
        st = stage;
        if (!wait_or_abort(&kv_full[stage], phase, lim, abort_flag)) return false;
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        return true;
    };
    // PV_hi of block `i` (if Q tile t takes part in it), then release V_i's stage
    auto finish_block = [&](int i, int first, int vst) -> bool {
        if (i >= first) {
            if (!wait_or_abort(p_full, pf_phase, lim, abort_flag)) return false;
            pf_phase ^= 1;
            tc_fence_after();
            issue_pv_hi<D, kF16>(tm, sPbt, sKV + vst * C::kTileBytes);
            mma_commit(pb_done);
        }
        mma_commit(&kv_empty[vst]);
        return true;
    };
    for (int r = 0; ok; ++r) {
        int k;
        if (!ring.get(r, k, lim, abort_flag)) { ok = false; break; }
        const Unit u = (k < total) ? ring.decoded(r) : Unit{};
        ring.release(r);
        if (k >= total) break;
        const int first = (t == 0) ? u.first0 : 0;   // Q tile 0 skips the block past its diagonal
        if (!wait_or_abort(&bars[kBarQFull], r & 1, lim, abort_flag)) { ok = false; break; }
        int vprev = -1;                                // V stage of block i-1
        for (int i = 0; i < u.n; ++i) {
            const bool active = (i >= first);
            int kst, vst;
            if (!next_stage(kst)) { ok = false; break; }
            if (active) {
                tc_fence_after();
                issue_s<D, kF16>(tm, sQt, sKV + kst * C::kTileBytes);
                mma_commit(s_full);
            }
            mma_commit(&kv_empty[kst]);
            if (i == u.n - 1) mma_commit(&bars[kBarQEmpty]);
            if (vprev >= 0 && !finish_block(i - 1, first, vprev)) { ok = false; break; }
            if (!next_stage(vst)) { ok = false; break; }
            if (active) {
                if (!wait_or_abort(p_half, ph_phase, lim, abort_flag)) { ok = false; break; }
                ph_phase ^= 1;
                tc_fence_after();
                issue_pv_lo<D, kF16>(tm, sKV + vst * C::kTileBytes, i > first);
            }
            vprev = vst;
        }
        if (!ok) break;
        if (!finish_block(u.n - 1, first, vprev)) { ok = false; break; }
    }
    // Every MMA this thread issued must complete before tensor memory is freed.
    mma_commit(&bars[kBarDrain + t]);
    mbar_wait(&bars[kBarDrain + t], 0, kDrainLimitNs);
}

// Packed fp32 pair helpers (sm_100 family: one instruction for two lanes of work).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Running max (kMax) or min of 32 raw scores into 8 chains.
template <bool kMax>
__device__ __forceinline__ void chunk_extreme(const uint32_t* x, float (&m)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float a = __uint_as_float(x[q]), b = __uint_as_float(x[q + 8]);
        const float cc = __uint_as_float(x[q + 16]), d = __uint_as_float(x[q + 24]);
        m[q] = kMax ? max3(m[q], max3(a, b, cc), d) : min3(m[q], min3(a, b, cc), d);
    }
}

template <bool kMax>
__device__ __forceinline__ float reduce8(const float (&m)[8]) {
    const float a = kMax ? max3(m[0], m[1], m[2]) : min3(m[0], m[1], m[2]);
    const float b = kMax ? max3(m[3], m[4], m[5]) : min3(m[3], m[4], m[5]);
    return kMax ? max3(a, b, fmaxf(m[6], m[7])) : min3(a, b, fminf(m[6], m[7]));
}

// Row max (scale c >= 0) or row min (c < 0) of 128 raw scores, 8 chains deep.
template <bool kMax>
__device__ __forceinline__ float row_extreme(const uint32_t (&sr)[128]) {
    float m[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) m[q] = kMax ? -INFINITY : INFINITY;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) chunk_extreme<kMax>(&sr[ch * 32], m);
    return reduce8<kMax>(m);
}

// Masks a score row in place so the unmasked max and exponent code serves
// masked blocks too (one copy of that code stays hot in the instruction
// cache; separate masked copies ran once per unit and were fetched cold each
// time). Columns >= lim become the raw value whose scaled score is -inf
// (-inf for c > 0, +inf for c < 0). With c == 0 every valid score scales to
// 0 whatever it is, so valid columns become 0, masked ones -inf, and the
// caller scales the row by 1 instead (it calls this for every block then).
__device__ __forceinline__ void mask_row(uint32_t (&sr)[128], float c, int lim) {
    const uint32_t masked = (c < 0.f) ? 0x7f800000u : 0xff800000u;
    const uint32_t keep = (c == 0.f) ? 0u : 0xffffffffu;
#pragma unroll
    for (int e = 0; e < 128; ++e) sr[e] = (e < lim) ? (sr[e] & keep) : masked;
}

// Rounding error of a block's largest probability in the element type P is
// multiplied in. The PV product uses the rounded P, so adding this error to the
// normaliser of O keeps the dominant term's weight exact in O = PV / l: a near
// one-hot row (large logits) then reproduces its V row to within O's own
// rounding, where the plain fp32 sum would leave the top term off by up to half
// a bf16 unit in the last place. r_ext is the block's raw extreme score; the
// exponent is formed exactly as exp_pack forms every element's.
template <bool kF16>
__device__ __forceinline__ float top_rounding_error(float r_ext, float cs, float negm) {
    const float p = ex2(fmaf(r_ext, cs, negm));
    float pr;
    if constexpr (kF16) {
        pr = __half2float(__float2half_rn(p));
    } else {
        pr = __bfloat162float(__float2bfloat16_rn(p));
    }
    return pr - p;
}

// exp2 of 32 scores (keys 32*ch .. 32*ch+31): x = s * c - m in one packed FMA per
// pair, p = 2^x (masked columns hold the raw value whose x is -inf, see
// mask_row), packed into 16 bf16 pairs (key 2e in the low half of pk[e]); the
// fp32 probabilities are added pairwise into acc[4].
template <bool kF16>
__device__ __forceinline__ void exp_pack(const uint32_t (&sr)[128], int ch, uint64_t c2, uint64_t negm2,
                                         uint64_t (&acc)[4], uint32_t (&pk)[16]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int c0 = ch * 32 + 2 * e;
        const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), c2, negm2);
        float x0, x1;
        f2_unpack(x2, x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
        pk[e] = pack2<kF16>(p0, p1);
    }
}

// Keys 0-63 of P_t: chunks 0 and 1 into tensor memory (over S_t's first 32 columns).
template <bool kF16>
__device__ __forceinline__ void p_lo_to_tmem(const uint32_t (&sr)[128], uint64_t c2, uint64_t negm2,
                                             uint64_t (&acc)[4], uint32_t tS) {
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        uint32_t pk[16];
        exp_pack<kF16>(sr, ch, c2, negm2, acc, pk);
        tmem_st16(tS + ch * 16, pk);
    }
}

// Keys 64-127 of P_t: chunks 2 and 3 into this row of the shared-memory half,
// K-major with the 128-byte swizzle (16-byte chunk q of the row at q ^ (row & 7)).
template <bool kF16>
__device__ __forceinline__ void p_hi_to_smem(const uint32_t (&sr)[128], uint64_t c2, uint64_t negm2,
                                             uint64_t (&acc)[4], uint32_t prow, int swz) {
#pragma unroll
    for (int ch = 2; ch < 4; ++ch) {
        uint32_t pk[16];
        exp_pack<kF16>(sr, ch, c2, negm2, acc, pk);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c16 = (ch - 2) * 4 + q;
            st_shared16(prow + ((c16 ^ swz) << 4), make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
        }
    }
}

// Softmax warpgroup of Q tile t (thread = query row = TMEM lane). After a unit's
// last block it also writes the unit's O tile: O / l as bf16, 32 columns at a
// time through the tile's shared half of P (free once the last PV is done).
// Each warp stores its own 32 rows with TMA (rows past N are clipped), so the
// epilogue needs no barrier wider than a warp.
template <int D, bool kF16>
__device__ void softmax_role(uint32_t tm, int t, int wq, int lane, uint64_t* bars, const UnitRing& ring,
                             volatile int* abort_flag, uint8_t* sPb, const CUtensorMap* tm_o, const KernelArgs& a) {
    using C = Cfg<D>;
    uint64_t* s_full = bars + kBarSFull + t;
    uint64_t* p_half = bars + kBarPHalf + t;
    uint64_t* p_full = bars + kBarPFull + t;
    uint64_t* pb_done = bars + kBarPbDone + t;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t lane_base = tm + ((uint32_t)(wq * 32) << 16);
    const uint32_t tS = lane_base + kTmemS;
    const uint32_t tO = lane_base + kTmemO;
    const int row_in_tile = wq * 32 + lane;
    uint8_t* sPbt = sPb + t * C::kPbBytes;
    const uint32_t prow = smem_u32(sPbt + row_in_tile * 128);   // this row of the shared half of P
    uint8_t* pwarp = sPbt + wq * 32 * 128;   // this warp's 32 rows (4 KB, 1024-byte aligned)
    const int swz = row_in_tile & 7;
    const float c = a.scale_log2;
    // with c == 0 every score is replaced by 0 (mask_row) and scaled by 1
    const float cs = (c == 0.f) ? 1.f : c;
    const uint64_t c2 = f2_pack(cs, cs);
    const int total = a.BH * a.U;
    uint32_t s_phase = 0, pb_phase = 0;
    bool store_pending = false;   // an O store of this warp may still be reading the P buffer
    bool ok = true;
    // bounded wait shared by the whole warp
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool got = wait_or_abort(bar, parity, lim, abort_flag);
        return __all_sync(0xffffffffu, got);
    };
    for (int r = 0; ok; ++r) {
        int k;
        bool got = ring.get(r, k, lim, abort_flag);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const Unit u = (k < total) ? ring.decoded(r) : Unit{};
        __syncwarp();
        if (lane == 0) ring.release(r);
        if (k >= total) break;
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
            const int key0 = j * kBN;
            const bool need_mask = (key0 + kBN > a.N) || (a.causal && key0 + kBN - 1 > tile_row0);
            // valid keys of this row in this block: key < N and, causal, key <= row
            tmem_ld128(tS, sr);
            if (need_mask || c == 0.f) {
                const int last = a.causal ? min(a.N, row + 1) : a.N;
                mask_row(sr, c, need_mask ? max(0, min(kBN, last - key0)) : kBN);
            }
            const float r_ext = (cs >= 0.f) ? row_extreme<true>(sr) : row_extreme<false>(sr);
            const float m_tile = r_ext * cs;
            // PV_hi of the previous block must be complete before O_t is rescaled
            // or the shared half of P_t is rewritten.
            bool pb_pending = (i > first);
            // Move the reference max only when the block's max exceeds it by more
            // than the threshold; then rescale O_t and l.
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
            // keys 0-63 into tensor memory; the MMA takes them (and then computes the
            // next block's scores) while keys 64-127 are being exponentiated
            p_lo_to_tmem<kF16>(sr, c2, negm2, acc, tS);
            // Rescale O_t after the first half of the exponentials, so the wait for
            // the previous block's PV_hi overlaps them; it must land before PV_lo(i).
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                if (pb_pending) {
                    if (!wait_warp(pb_done, pb_phase)) { ok = false; break; }
                    pb_phase ^= 1;
                    pb_pending = false;
                    tc_fence_after();
                }
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
            mbar_arrive(p_half);
            if (pb_pending) {
                if (!wait_warp(pb_done, pb_phase)) { ok = false; break; }
                pb_phase ^= 1;
            }
            if (store_pending) {   // the previous unit's O stores must have read this buffer
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
                store_pending = false;
            }
            p_hi_to_smem<kF16>(sr, c2, negm2, acc, prow, swz);
            fence_proxy_async_smem();
            mbar_arrive(p_full);
            const uint64_t s01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
            float sum0, sum1;
            f2_unpack(s01, sum0, sum1);
            l = l * alpha + (sum0 + sum1);
            l_o = l_o * alpha + (sum0 + sum1) + top_err;
        }
        if (!ok) break;
        // epilogue: O / l -> bf16 through shared memory and TMA, LSE in natural log
        if (!wait_warp(pb_done, pb_phase)) { ok = false; break; }   // the unit's last PV is complete
        pb_phase ^= 1;
        tc_fence_after();
        const float l_safe = (l > 0.f) ? l : 1.f;
        const float inv = 1.f / ((l_o > 0.f) ? l_o : 1.f);
        // 32 columns at a time through the two 2 KB halves of this warp's 4 KB
        // of the shared part of P (rows of 64 bytes with the 64-byte swizzle:
        // 16-byte chunk c of row r at c ^ ((r >> 1) & 3)), so each quarter is
        // written while the store of the one before reads the other half. The
        // loop stays rolled: this once-per-unit code stays small in the
        // instruction cache.
        const uint32_t orow = smem_u32(pwarp) + lane * 64;   // this row in each half
        const int oswz = (lane >> 1) & 3;
#pragma unroll 1
        for (int qt = 0; qt < D / 32; ++qt) {
            uint32_t ov[32];                                  // this quarter's 32 columns of O
            tmem_ld32(tO + qt * 32, ov);
            if (qt >= 2) {   // the store two quarters back must have read this half
                if (lane == 0) bulk_wait_read1();
                __syncwarp();
            }
            const uint32_t half = (uint32_t)(qt & 1) * 2048u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {     // 16-byte chunk = 8 output columns
                const uint32_t* o8 = ov + c * 8;
                uint4 w;
                w.x = pack2<kF16>(__uint_as_float(o8[0]) * inv, __uint_as_float(o8[1]) * inv);
                w.y = pack2<kF16>(__uint_as_float(o8[2]) * inv, __uint_as_float(o8[3]) * inv);
                w.z = pack2<kF16>(__uint_as_float(o8[4]) * inv, __uint_as_float(o8[5]) * inv);
                w.w = pack2<kF16>(__uint_as_float(o8[6]) * inv, __uint_as_float(o8[7]) * inv);
                st_shared16(orow + half + ((c ^ oswz) << 4), w);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && qt * 32 < a.d) {   // this warp's 32 rows; quarters past d hold no columns
                tma_store_4d(tm_o, pwarp + half, qt * 32, tile_row0 + wq * 32, u.h, u.b);
                bulk_commit();
            }
            __syncwarp();
        }
        tc_fence_before();
        store_pending = true;   // the last slice's read is waited for before the buffer is next written
        if (row < a.N) a.lse[(int64_t)u.bh * a.N + row] = (m_ref + log2f(l_safe)) * 0.69314718055994531f;
    }
    if (lane == 0) bulk_wait0();   // this warp's O stores are complete
}

// ------------------------------------------------------------------ kernel

// Instantiated for D = 128 only; head dims up to 64 run on attn_fwd_d64_kernel.
// kF16: Q, K, V, O (and P on the tensor cores) are fp16 instead of bf16.
template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const KernelArgs a) {
    static_assert(D == 128, "the d = 64 path is attn_fwd_d64_kernel");
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem;
    uint8_t* sPb = smem + C::kOffPb;
    uint8_t* sKV = smem + C::kOffKV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);   // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile int* member = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 12);   // holds the counter slot
    const UnitRing ring{bars + kBarUnitFull, bars + kBarUnitEmpty,
                        reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16),
                        reinterpret_cast<volatile int*>(smem + C::kOffMisc + 32)};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        mbar_init(&bars[kBarQFull], 1);
        mbar_init(&bars[kBarQEmpty], 2);                         // one commit per MMA stream
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars[kBarSFull + t], 1);                  // MMA commit
            mbar_init(&bars[kBarPHalf + t], kBM);                // every softmax thread arrives
            mbar_init(&bars[kBarPFull + t], kBM);
            mbar_init(&bars[kBarPbDone + t], 1);                 // MMA commit
            mbar_init(&bars[kBarDrain + t], 1);
        }
        mbar_init(&bars[kBarNever], 1);
        for (int sl = 0; sl < kUnitRing; ++sl) {
            mbar_init(&bars[kBarUnitFull + sl], 1);
            mbar_init(&bars[kBarUnitEmpty + sl], kUnitReaders);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars[kBarKV + s], 1);                     // kv_full
            mbar_init(&bars[kBarKV + C::kStages + s], 2);        // kv_empty: one commit per MMA stream
        }
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
    // Launched with programmatic stream serialization: the set-up above may run
    // while the previous kernel in the stream finishes; nothing in global memory
    // is read or written before that kernel has completed. A later launch of
    // this kernel may likewise start its set-up on SMs this grid has left.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < kWarpProducer) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        softmax_role<D, kF16>(warp < 4 ? tmem0 : tmem1, warp / 4, warp % 4, lane, bars, ring, abort_flag, sPb, &tm_o, a);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (warp == kWarpProducer) {
            if (lane == 0) producer<D>(&tm_q, &tm_k, &tm_v, sQ, sKV, bars, ring, abort_flag, member, a);
            __syncwarp();
        } else if (warp == kWarpMma0 || warp == kWarpMma1) {
            const int t = warp - kWarpMma0;
            if (lane == 0) mma_issuer<D, kF16>(t ? tmem1 : tmem0, t, sQ, sPb, sKV, bars, ring, abort_flag, a);
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
    // The last CTA out returns the launch's counters to zero for the next launch
    // that draws this slot.
    if (threadIdx.x == 0 && *member) sched_release(a.sched);
}
}  // namespace
}  // namespace bos

#include "attn_fwd_d64.cuh"
#include "attn_fwd_d256.cuh"

namespace bos {
namespace {

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

// bf16 (fp16 with f16) [B, H, N, d] with element strides st = {batch, head,
// row} (d contiguous) viewed as a 4-D tensor (column, row, head, batch); boxes
// of 64 columns x `rows` rows with the 128-byte swizzle (or 32 columns with the
// 64-byte swizzle); loads read rows past N (and columns past d) as zero, stores
// drop them.
bool encode_qkv_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int B, int H, int N, int d,
                    const long long (&st)[3], int rows, bool f16 = false, int cols = 64) {
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    cuuint32_t box[4] = {(cuuint32_t)cols, (cuuint32_t)rows, 1, 1};
    cuuint32_t elem[4] = {1, 1, 1, 1};
    return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(base), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// L2 bytes the K and V of one causal scheduling group of heads may take.
constexpr double kGroupKvBytes = 32.0 * 1024 * 1024;

uint64_t g_wait_limit_ns = kDefaultWaitLimitNs;
int g_test_stall = 0;
int g_test_sched_busy = 0;
std::atomic<unsigned int> g_sched_next{0};

template <int D, bool kF16>
int launch_d(const AttnParams& p, cudaStream_t stream, int dev) {
    constexpr int kSmemBytes =
        (D == 64) ? d64::Cfg::kSmemBytes : (D == 256) ? d256::Cfg::kSmemBytes : Cfg<128>::kSmemBytes;
    auto* const kernel = (D == 64) ? attn_fwd_d64_kernel<kF16>
                         : (D == 256) ? attn_fwd_d256_kernel<kF16>
                                      : attn_fwd_sm103_kernel<128, kF16>;
    // rows per work unit: two 128-row Q tiles, or one for d > 128
    constexpr int kRowsPerUnit = (D == 256) ? kBM : kUnitRows;
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return ATTN_ERR_CUDA;
    const int BH = p.B * p.H;
    CUtensorMap mq, mk, mv, mo;
    // Q, K and V move in 128-row boxes (V in 64-row key halves for d > 128); O is
    // stored 32 rows (one warp) at a time, 32 columns at a time for d = 128
    // (the maps describe the caller's d columns; boxes are 64 wide, so columns
    // from d up to the kernel's width D load as zero and are not stored)
    if (!encode_qkv_map(enc, &mq, p.q, p.B, p.H, p.N, p.d, p.sq, kBM, kF16) ||
        !encode_qkv_map(enc, &mk, p.k, p.B, p.H, p.N, p.d, p.sk, kBN, kF16) ||
        !encode_qkv_map(enc, &mv, p.v, p.B, p.H, p.N, p.d, p.sv, D == 256 ? kBN / 2 : kBN, kF16) ||
        !encode_qkv_map(enc, &mo, p.o, p.B, p.H, p.N, p.d, p.so, 32, kF16, D == 128 ? 32 : 64))
        return ATTN_ERR_BAD_SHAPE;
    // per-device caches, shared by host threads (the values are idempotent)
    static std::atomic<int> sms_cache[64];
    static std::atomic<int> attr_done[64];
    static std::atomic<unsigned int*> sched_cache[64];
    int sms = (dev >= 0 && dev < 64) ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) sms_cache[dev].store(sms, std::memory_order_relaxed);
    }
    unsigned int* sched = (dev >= 0 && dev < 64) ? sched_cache[dev].load(std::memory_order_relaxed) : nullptr;
    if (sched == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_attn_sched) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        sched = static_cast<unsigned int*>(ptr);
        if (dev >= 0 && dev < 64) sched_cache[dev].store(sched, std::memory_order_relaxed);
    }
    if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_LAUNCH;
        }
        if (dev >= 0 && dev < 64) attr_done[dev].store(1, std::memory_order_relaxed);
    }
    KernelArgs a;
    a.BH = BH;
    a.H = p.H;
    a.N = p.N;
    a.U = (p.N + kRowsPerUnit - 1) / kRowsPerUnit;
    a.causal = p.causal;
    a.d = p.d;
    // Causal units run heaviest first within groups of heads whose K and V
    // together fit kGroupKvBytes, so the K/V tiles a group re-reads stay in L2
    // (ordering over every head at once kept all heads' K/V in flight).
    {
        const double kv_head = 4.0 * (double)p.N * (double)D;   // bf16 K and V of one head, at the kernel's width
        const double g = kGroupKvBytes / kv_head;
        a.group = g >= (double)BH ? BH : (g < 1.0 ? 1 : (int)g);
    }
    a.scale_log2 = (float)((double)p.scale * 1.4426950408889634);
    a.o = static_cast<__nv_bfloat16*>(p.o);
    a.lse = p.lse;
    a.wait_limit_ns = g_wait_limit_ns;
    a.test_stall = g_test_stall;
    a.sched = sched + kSchedWords * (g_sched_next.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
    // test hook: the drawn slot is marked as held by another launch for the
    // duration of this one, so every CTA finds it busy
    static const unsigned long long kForeignTag = ~0ull;
    if (g_test_sched_busy &&
        cudaMemcpyAsync(a.sched + 2, &kForeignTag, sizeof(kForeignTag), cudaMemcpyHostToDevice, stream) !=
            cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    const int64_t units = (int64_t)BH * a.U;
    const int grid = (int)(units < sms ? units : sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(D == 256 ? d256::kThreads : kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mo, a) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
    }
    if (g_test_sched_busy && cudaMemsetAsync(a.sched + 2, 0, sizeof(unsigned long long), stream) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace

int launch_attn_fwd(const AttnParams& p, cudaStream_t stream, int dev) {
    // head dims below a kernel's width run on it with the missing columns
    // zero-filled by TMA on load and clipped on store
    if (p.f16) {
        if (p.d <= 64) return launch_d<64, true>(p, stream, dev);
        if (p.d <= 128) return launch_d<128, true>(p, stream, dev);
        return launch_d<256, true>(p, stream, dev);
    }
    if (p.d <= 64) return launch_d<64, false>(p, stream, dev);
    if (p.d <= 128) return launch_d<128, false>(p, stream, dev);
    return launch_d<256, false>(p, stream, dev);
}

void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns ? ns : kDefaultWaitLimitNs; }

void set_test_stall(int on) { g_test_stall = on ? 1 : 0; }

void set_test_sched_busy(int on) { g_test_sched_busy = on ? 1 : 0; }

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

#include "attn_bwd.cuh"
