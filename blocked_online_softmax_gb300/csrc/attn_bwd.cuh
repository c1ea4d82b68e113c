// Attention backward for GB300 (sm_103a). Included once, at the end of
// attn_fwd_sm103.cu, after the shared pieces (bounded waits, tensor maps, the
// host-side map encoder); it is not a header for other files.
//
// The method is Kernel 5 "FlashAttention Backward" of "4.4 Writing GPU Kernels
// with Triton" (llm-stack-book): a preprocessing pass D_i = rowsum(dO_i * O_i),
// then one program per key/value block j that loops over the query blocks able
// to see it, recomputes P = exp(S - L) from the saved natural-log LSE, and
// forms
//     dV_j += P^T dO_i,   dP = dO_i V_j^T,   dS = P * (dP - D_i) * scale,
//     dK_j += dS^T Q_i,   dQ_i += dS K_j   (added into an fp32 buffer),
// accumulating dK_j and dV_j privately and casting the fp32 dQ buffer to bf16
// at the end. An optional gradient g on the LSE output enters as D_i - g_i
// (the derivative of LSE_i in S_ij is P_ij).
//
// GB300 design: one CTA (512 threads) per (key block j of 128 keys, batch*head),
// looping over the query blocks i of 128 queries that can see block j.
// MMAs issued by one thread execute in issue order, so the five products of a
// block are split over two issuing warps, each with its own 256-column
// allocation, by what they wait on: X waits only for P, Y for dS and for the
// dQ read-out, and neither chain holds back the other's MMAs.
//   X (warp 13): S^T = K Q_i^T into X[0,128); P^T comes back over those
//                columns as bf16 pairs; dV_j += P^T dO_i into X[128,128+d).
//   Y (warp 14): dP^T = V dO_i^T into Y[0,128); dS^T comes back over those
//                columns; dK_j += dS^T Q_i into Y[128,128+d); then
//                dQ_i = dS K_j (fp32, query on the lane) into Y[0,128) for
//                d = 128 (after dK has read dS^T, in issue order) or into
//                Y[192,256) for d = 64.
// Working with the transposes keeps the key on the tensor-memory lane, so the
// dV and dK products take P^T and dS^T straight from tensor memory.
// Two compute warpgroups (thread = key = lane), warps 0-3 for queries 0-63 and
// warps 8-11 for queries 64-127 of each block, form P = exp2(S c - L2) as soon
// as S^T lands (X can then start dV and the next block's S^T), then dS = P (dP
// scale - D scale) once dP^T lands. Both are elementwise in the query, so the
// groups need no exchange; each packs its bf16 pairs over columns it has read
// itself (see pcol). dS also goes to shared memory, each thread writing its
// key's row of 64 queries with 16-byte stores ([key][query], 128-byte
// swizzle): the A operand of the dQ product, read query-major (MN-major).
// Warps 4-7 (thread = query = lane) take the dQ part out of tensor memory,
// write it to shared memory (an 8 KB slot per warp, 128-byte swizzle) and add
// it into the fp32 dQ buffer with TMA bulk tensor reductions, so the adds move
// as whole lines; per-thread atomics (one row per lane, or one line per warp
// with the head dim on the lane) were measured slower. They also stage each
// block's -LSE (base 2) and -D (times scale) in shared memory two blocks ahead,
// their global loads issued a block before the store; negated, each pair of
// queries costs the compute warps one packed f32x2 FMA per step.
// Warp 12 issues the TMA loads: K_j and V_j once, Q_i into two stages and dO_i
// into one (its next load has the dS and dK/dQ steps of a block to land).

namespace bos {
namespace {

namespace bwd {

// Warps 0-3 and 8-11: compute (queries 0-63 and 64-127 of every block); 4-7:
// dQ; 12: TMA producer; 13, 14: MMA issuers; 15 idle. Registers after launch
// (512 x 128), redistributed per warpgroup with setmaxnreg:
// 128 x (kRegsCompute x 2 + kRegsDq + kRegsControl) = 65536.
constexpr int kThreads = 512;
constexpr int kWarpDq = 4;          // warps 4-7
constexpr int kWarpCompute1 = 8;    // warps 8-11: the second half of each block's queries
constexpr int kWarpProducer = 12;
constexpr int kWarpMmaX = 13;       // also allocates both tensor-memory regions
constexpr int kWarpMmaY = 14;
constexpr int kRegsCompute = 112;
constexpr int kRegsDq = 184;
constexpr int kRegsControl = 104;
static_assert(2 * kRegsCompute + kRegsDq + kRegsControl == 512, "register split must use the launch's file");
constexpr uint32_t kCols = 256;     // columns of each allocation
constexpr uint32_t kAcc = 128;      // dV (in X) and dK (in Y) start at this column
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSmem = 232448;    // 227 KB per CTA

enum : int {
    kBarKV = 0,        // K_j and V_j have landed
    kBarQFull = 1,     // [2] Q_i of a stage has landed
    kBarQEmpty = 3,    // [2] a Q stage is free: X's S and Y's dK of its block are complete (2 commits)
    kBarDoFull = 5,    // dO_i has landed
    kBarDoEmpty = 6,   // the dO buffer is free: X's dV and Y's dP of its block are complete (2 commits)
    kBarSFull = 7,     // S^T of the block is complete (X commit)
    kBarPReady = 8,    // P^T is written (256 arrivals: both compute warpgroups)
    kBarDpFull = 9,    // dP^T of the block is complete (Y commit)
    kBarDsReady = 10,  // dS^T (tensor memory) and dS (shared memory) are written (256 arrivals)
    kBarDqReady = 11,  // the block's dQ part is complete (Y commit)
    kBarDqRead = 12,   // the dQ part has been read out of tensor memory (128 arrivals)
    kBarLseFull = 13,  // [2] LSE and D of a block are staged (128 arrivals)
    kBarDrainX = 15,   // every MMA of X is complete
    kBarDrainY = 16,   // every MMA of Y is complete
    kBarDsHalf = 17,   // dS^T of queries 0-63 is written (128 arrivals, the first compute warpgroup): Y may start dK
    kBarNever = 18,    // test hook: nothing arrives on it
    kNumBars = 19,
};

template <int D>
struct Cfg {
    static constexpr int kTile = 128 * D * 2;                  // one bf16 128-row tile
    static constexpr int kBoxes = D / 64;
    static constexpr int kOffK = 0, kOffV = kTile;
    static constexpr int kOffQ = 2 * kTile;                    // Q stage s at kOffQ + s * kTile
    static constexpr int kOffDO = 4 * kTile;
    static constexpr int kOffDS = 5 * kTile;                   // dS, [128 keys][128 queries] bf16: 32 KB
    static constexpr int kOffDQ = kOffDS + 32768;              // dQ staging: 8 KB per dQ warp
    static constexpr int kOffLse = kOffDQ + 32768;             // [2][128] -LSE log2 e, then [2][128] -D scale
    static constexpr int kOffBar = kOffLse + 2048;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;    // two tensor-memory slots, abort flag
    static constexpr int kUsed = kOffMisc + 16;
    // 1 KB to align the tiles by hand when it fits; otherwise the kernel checks
    // that the dynamic shared memory it was given starts 1024-byte aligned
    static constexpr int kPad = (kUsed + 1024 <= kMaxSmem) ? 1024 : 0;
    static constexpr int kSmemBytes = kUsed + kPad;
    static constexpr uint32_t kTdQ = (D == 64) ? 192u : 0u;    // dQ columns in Y
    static_assert(kSmemBytes <= kMaxSmem, "shared memory over the per-CTA limit");
};

// Packed bf16 pairs of P^T / dS^T in tensor memory. Each compute warpgroup
// writes over the S^T / dP^T columns of its own queries (group h reads columns
// 64h..64h+63), so neither overwrites a column the other has yet to read:
// 32-query chunk ch (queries 32ch..32ch+31) lands at columns pcol(ch)..+15,
// and the 16-query MMA step kk reads its 8 columns at pcol_step(kk).
__host__ __device__ constexpr uint32_t pcol(int ch) { return (uint32_t)(ch * 16 + (ch >= 2 ? 32 : 0)); }
__host__ __device__ constexpr uint32_t pcol_step(int kk) { return (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)); }

struct BwdArgs {
    int BH, H, N, d, nkv, causal;
    float scale, c2;                  // c2 = scale * log2 e
    const float* lse;                 // [BH, N] natural log, from the forward pass
    const float* dsum;                // [BH, N] D = rowsum(dO * O) - dLSE
    float* dq_acc;                    // [BH, N, d] fp32, zeroed before the launch
    uint64_t wait_limit_ns;
    int test_stall;                   // test hook: X first waits on a barrier nothing signals
};

// Element-wise add of a shared-memory box into a global tensor (fp32 here),
// performed by the TMA unit; rows outside the tensor are clipped.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// The two values of a packed pair of the element type (bf16, or fp16 with kF16).
template <bool kF16>
__device__ __forceinline__ void unpack2(uint32_t v, float& lo, float& hi) {
    if constexpr (kF16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
        lo = f.x;
        hi = f.y;
    } else {
        lo = bf16_lo(v);
        hi = bf16_hi(v);
    }
}

template <int D>
__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                         const CUtensorMap* tm_do, uint8_t* smem, uint64_t* bars, volatile int* abort_flag,
                         int bh, int j, int i0, int nq, const BwdArgs& a) {
    using C = Cfg<D>;
    const int bb = bh / a.H, hh = bh - bb * a.H;             // batch and head
    mbar_arrive_expect_tx(&bars[kBarKV], 2 * C::kTile);
    for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_4d(smem + C::kOffK + b * 16384, tm_k, &bars[kBarKV], b * 64, j * 128, hh, bb);
        tma_load_4d(smem + C::kOffV + b * 16384, tm_v, &bars[kBarKV], b * 64, j * 128, hh, bb);
    }
    int last_q[2] = {-1, -1}, last_do = -1;
    for (int it = 0; it < nq; ++it) {
        const int s = it & 1;
        // the Q stage's previous block (it - 2) must be released by both issuers
        if (it >= 2 && !wait_or_abort(&bars[kBarQEmpty + s], (uint32_t)(((it >> 1) + 1) & 1), a.wait_limit_ns,
                                      abort_flag))
            break;
        mbar_arrive_expect_tx(&bars[kBarQFull + s], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
            tma_load_4d(smem + C::kOffQ + s * C::kTile + b * 16384, tm_q, &bars[kBarQFull + s], b * 64,
                        (i0 + it) * 128, hh, bb);
        last_q[s] = it;
        if (it >= 1 && !wait_or_abort(&bars[kBarDoEmpty], (uint32_t)((it - 1) & 1), a.wait_limit_ns, abort_flag))
            break;
        mbar_arrive_expect_tx(&bars[kBarDoFull], C::kTile);
        for (int b = 0; b < C::kBoxes; ++b)
            tma_load_4d(smem + C::kOffDO + b * 16384, tm_do, &bars[kBarDoFull], b * 64, (i0 + it) * 128, hh, bb);
        last_do = it;
    }
    // every copy this thread started must land before the CTA may exit
    mbar_wait(&bars[kBarKV], 0, kDrainLimitNs);
    for (int s = 0; s < 2; ++s)
        if (last_q[s] >= 0) mbar_wait(&bars[kBarQFull + s], (uint32_t)((last_q[s] >> 1) & 1), kDrainLimitNs);
    if (last_do >= 0) mbar_wait(&bars[kBarDoFull], (uint32_t)(last_do & 1), kDrainLimitNs);
}

// X: S^T = K Q_i^T, then dV_j += P^T dO_i once P^T is written.
template <int D, bool kF16>
__device__ void mma_x(uint32_t tX, uint8_t* smem, uint64_t* bars, volatile int* abort_flag, int nq,
                      const BwdArgs& a) {
    using C = Cfg<D>;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t sK = smem_u32(smem + C::kOffK);
    // M = 128 keys, N = 128 queries, K = d; both operands K-major
    constexpr uint32_t id_s = idesc_f32acc(128, 128, false, false, kF16);
    // M = 128 keys, N = d, K = 128 queries; A from tensor memory, B (dO) N-major
    constexpr uint32_t id_kv = idesc_f32acc(128, D, false, true, kF16);
    bool ok = !(a.test_stall && !wait_or_abort(&bars[kBarNever], 0, lim, abort_flag)) &&
              wait_or_abort(&bars[kBarKV], 0, lim, abort_flag);
    const uint32_t sDO = smem_u32(smem + C::kOffDO);
    for (int it = 0; ok && it < nq; ++it) {
        const int s = it & 1;
        const uint32_t sQ = smem_u32(smem + C::kOffQ + s * C::kTile);
        if (!wait_or_abort(&bars[kBarQFull + s], (uint32_t)((it >> 1) & 1), lim, abort_flag)) break;
        tc_fence_after();
        // overwrites P^T of the previous block, which that block's dV (issued earlier) reads
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
            mma_ss(tX, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[kBarSFull]);
        mma_commit(&bars[kBarQEmpty + s]);
        if (!wait_or_abort(&bars[kBarPReady], (uint32_t)(it & 1), lim, abort_flag) ||
            !wait_or_abort(&bars[kBarDoFull], (uint32_t)(it & 1), lim, abort_flag))
            break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 queries per step: 8 columns of bf16 pairs, 16 rows of dO
            mma_ts(tX + kAcc, tX + pcol_step(kk), sdesc_sw128(sDO + kk * 2048, 16384, 1024), id_kv,
                   (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarDoEmpty]);
    }
    mma_commit(&bars[kBarDrainX]);
    mbar_wait(&bars[kBarDrainX], 0, kDrainLimitNs);
}

// Y: dP^T = V dO_i^T, then dK_j += dS^T Q_i and dQ_i = dS K_j once dS is written.
template <int D, bool kF16>
__device__ void mma_y(uint32_t tY, uint8_t* smem, uint64_t* bars, volatile int* abort_flag, int nq,
                      const BwdArgs& a) {
    using C = Cfg<D>;
    constexpr bool kDqOverDp = (C::kTdQ == 0);   // dQ reuses the dP^T columns
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
    const uint32_t sDS = smem_u32(smem + C::kOffDS);
    constexpr uint32_t id_s = idesc_f32acc(128, 128, false, false, kF16);
    constexpr uint32_t id_kv = idesc_f32acc(128, D, false, true, kF16);
    // M = 128 queries, N = d, K = 128 keys; A (dS, stored [key][query]) and
    // B (K_j, stored [key][d]) both MN-major
    constexpr uint32_t id_q = idesc_f32acc(128, D, true, true, kF16);
    bool ok = wait_or_abort(&bars[kBarKV], 0, lim, abort_flag);
    const uint32_t sDO = smem_u32(smem + C::kOffDO);
    for (int it = 0; ok && it < nq; ++it) {
        const int s = it & 1;
        const uint32_t sQ = smem_u32(smem + C::kOffQ + s * C::kTile);
        if (!wait_or_abort(&bars[kBarQFull + s], (uint32_t)((it >> 1) & 1), lim, abort_flag) ||
            !wait_or_abort(&bars[kBarDoFull], (uint32_t)(it & 1), lim, abort_flag))
            break;
        if (kDqOverDp && it > 0 && !wait_or_abort(&bars[kBarDqRead], (uint32_t)((it - 1) & 1), lim, abort_flag))
            break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
            mma_ss(tY, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[kBarDpFull]);
        mma_commit(&bars[kBarDoEmpty]);
        // dK over queries 0-63 as soon as their dS^T is written, the rest once all of dS is
        if (!wait_or_abort(&bars[kBarDsHalf], (uint32_t)(it & 1), lim, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tY + kAcc, tY + pcol_step(kk), sdesc_sw128(sQ + kk * 2048, 16384, 1024), id_kv,
                   (it > 0 || kk > 0) ? 1u : 0u);
        if (!wait_or_abort(&bars[kBarDsReady], (uint32_t)(it & 1), lim, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 4; kk < 8; ++kk)
            mma_ts(tY + kAcc, tY + pcol_step(kk), sdesc_sw128(sQ + kk * 2048, 16384, 1024), id_kv, 1u);
        mma_commit(&bars[kBarQEmpty + s]);
        if (!kDqOverDp && it > 0 && !wait_or_abort(&bars[kBarDqRead], (uint32_t)((it - 1) & 1), lim, abort_flag))
            break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 keys per step: 16 rows of dS (two 64-query boxes) and of K_j
            mma_ss(tY + C::kTdQ, sdesc_sw128(sDS + kk * 2048, 16384, 1024),
                   sdesc_sw128(sK + kk * 2048, 16384, 1024), id_q, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarDqReady]);
    }
    mma_commit(&bars[kBarDrainY]);
    mbar_wait(&bars[kBarDrainY], 0, kDrainLimitNs);
}

// P^T of one block's queries 64h..64h+63 into tensor memory (over the S^T
// columns already read) and into registers as bf16 pairs (queries 2e, 2e+1 of
// each 32-query chunk). The second chunk's scores are requested from tensor
// memory before the first chunk's P^T is stored, so that load's latency
// overlaps the store (the columns differ: see pcol).
template <bool kMasked, bool kF16>
__device__ __forceinline__ void p_phase(uint32_t lx, const float* nL, uint64_t c2x2, int r, bool key_ok, bool diag,
                                        int h, uint32_t (&pk)[32]) {
    uint32_t sv[2][32];
    tmem_ld32_nowait(lx + (2 * h) * 32, sv[0]);
    tmem_ld_wait32(sv[0]);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int ch = 2 * h + cc;
        uint32_t t[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int qc = ch * 32 + 2 * e;
            const uint64_t nl = *reinterpret_cast<const uint64_t*>(nL + qc);
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[cc][2 * e]), __uint_as_float(sv[cc][2 * e + 1])), c2x2, nl),
                      x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if (kMasked) {
                if (!key_ok || (diag && qc < r)) p0 = 0.f;
                if (!key_ok || (diag && qc + 1 < r)) p1 = 0.f;
            }
            t[e] = pack2<kF16>(p0, p1);
            pk[cc * 16 + e] = t[e];
        }
        if (cc == 0) tmem_ld32_nowait(lx + (ch + 1) * 32, sv[1]);
        tmem_st16(lx + pcol(ch), t);
        if (cc == 0) tmem_ld_wait32(sv[1]);
    }
}

// Compute warpgroup h (0: queries 0-63 of each block, 1: queries 64-127); the
// two groups share the keys (tensor-memory lanes) and need no exchange: P and
// dS are elementwise in the query. After the loop group 0 writes dV_j and
// group 1 writes dK_j.
template <int D, bool kF16>
__device__ void compute_role(const CUtensorMap* tm_dk, const CUtensorMap* tm_dv, uint32_t tX, uint32_t tY, int w,
                             int h, int lane, uint8_t* smem, uint64_t* bars,
                             volatile int* abort_flag, int bh, int j, int nq, const BwdArgs& a) {
    using C = Cfg<D>;
    const uint64_t lim = a.wait_limit_ns;
    const int r = w * 32 + lane;                              // tensor-memory lane = key within the block
    const uint32_t lx = tX + ((uint32_t)(w * 32) << 16), ly = tY + ((uint32_t)(w * 32) << 16);
    const float* lse_s = reinterpret_cast<const float*>(smem + C::kOffLse);   // [2][128] -LSE log2 e
    const float* dsc_s = lse_s + 2 * 128;                                      // [2][128] -D scale
    // this thread's row of the [key][query] dS buffer: 128 bytes in each of the two
    // 64-query boxes, its 16-byte chunks swizzled with the key (r % 8)
    uint8_t* ds_row = smem + C::kOffDS + r * 128;
    const int ds_swz = r & 7;
    const uint64_t c2x2 = f2_pack(a.c2, a.c2), scale2 = f2_pack(a.scale, a.scale);
    const int key = j * 128 + r;
    const bool key_ok = key < a.N;
    const bool tail_block = j * 128 + 128 > a.N;
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool got = wait_or_abort(bar, parity, lim, abort_flag);
        return __all_sync(0xffffffffu, got);
    };
    for (int it = 0; it < nq; ++it) {
        const uint32_t par = (uint32_t)(it & 1);
        const int lb = it & 1;
        if (!wait_warp(&bars[kBarLseFull + lb], (uint32_t)((it >> 1) & 1)) || !wait_warp(&bars[kBarSFull], par))
            return;
        tc_fence_after();
        const float* L = lse_s + lb * 128;
        const float* Dsc = dsc_s + lb * 128;
        const bool diag = a.causal && it == 0;               // the first query block is block j itself
        uint32_t pk[32];
        if (diag || tail_block)
            p_phase<true, kF16>(lx, L, c2x2, r, key_ok, diag, h, pk);
        else
            p_phase<false, kF16>(lx, L, c2x2, r, key_ok, diag, h, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kBarPReady]);

        if (!wait_warp(&bars[kBarDpFull], par)) return;
        tc_fence_after();
        // the second chunk's dP^T is requested before the first chunk's dS is
        // stored, so that load's latency overlaps the stores (disjoint columns)
        uint32_t dpv[2][32];
        tmem_ld32_nowait(ly + (2 * h) * 32, dpv[0]);
        tmem_ld_wait32(dpv[0]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int ch = 2 * h + cc;
            uint32_t dk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int qc = ch * 32 + 2 * e;
                const uint64_t nd = *reinterpret_cast<const uint64_t*>(Dsc + qc);
                const uint32_t p = pk[cc * 16 + e];
                const uint64_t t2 = f2_fma(f2_pack(__uint_as_float(dpv[cc][2 * e]), __uint_as_float(dpv[cc][2 * e + 1])),
                                           scale2, nd);
                float ds0, ds1, p0, p1;
                unpack2<kF16>(p, p0, p1);
                f2_unpack(f2_mul(f2_pack(p0, p1), t2), ds0, ds1);
                dk[e] = pack2<kF16>(ds0, ds1);
            }
            if (cc == 0) tmem_ld32_nowait(ly + (ch + 1) * 32, dpv[1]);
            tmem_st16(ly + pcol(ch), dk);                     // dS^T over dP^T columns this group has read
            uint8_t* box = ds_row + (ch >> 1) * 16384;       // queries 32ch..32ch+31: chunks 4(ch&1)..+3
#pragma unroll
            for (int c = 0; c < 4; ++c)
                st_shared16(smem_u32(box + ((((ch & 1) * 4 + c) ^ ds_swz) << 4)),
                            make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]));
            if (ch == 1) {                                    // Y's first four dK steps need only these
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[kBarDsHalf]);                // group 0 only
            }
            if (cc == 0) tmem_ld_wait32(dpv[1]);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[kBarDsReady]);
    }
    // dV_j is final once all of X's MMAs are complete, dK_j once all of Y's are.
    // Each warp converts its 32 keys' rows to the element type, writes them
    // 128-byte swizzled into a tile no MMA reads any more (dO's for dV: X's dV
    // products and Y's dP^T, its readers, are complete; V's for dK), and
    // stores them with TMA, which clips rows past N and columns past d.
    // Direct 16-byte stores from the lanes touched 32 rows per instruction.
    const int b_idx = bh / a.H, h_idx = bh % a.H;
    bool drained = true;
#pragma unroll 1
    for (int pass = h; pass < h + 1 && drained; ++pass) {
        if (!wait_warp(&bars[pass == 0 ? kBarDrainX : kBarDrainY], 0)) {
            drained = false;
            break;
        }
        tc_fence_after();
        const uint32_t src = (pass == 0 ? lx : ly) + kAcc;
        uint8_t* stage = smem + (pass == 0 ? C::kOffDO : C::kOffV) + w * 4096;   // this warp's 32 rows
        uint8_t* srow = stage + lane * 128;
#pragma unroll 1
        for (int hb = 0; hb < C::kBoxes; ++hb) {     // 64 columns: one 128-byte row per key
            uint32_t v0[32], v1[32];
            tmem_ld32(src + hb * 64, v0);
            tmem_ld32(src + hb * 64 + 32, v1);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t* vv = (c < 4) ? v0 + c * 8 : v1 + (c - 4) * 8;
                uint4 wv;
                wv.x = pack2<kF16>(__uint_as_float(vv[0]), __uint_as_float(vv[1]));
                wv.y = pack2<kF16>(__uint_as_float(vv[2]), __uint_as_float(vv[3]));
                wv.z = pack2<kF16>(__uint_as_float(vv[4]), __uint_as_float(vv[5]));
                wv.w = pack2<kF16>(__uint_as_float(vv[6]), __uint_as_float(vv[7]));
                st_shared16(smem_u32(srow + hb * 16384 + ((c ^ (lane & 7)) << 4)), wv);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            for (int hb = 0; hb < C::kBoxes; ++hb)
                tma_store_4d(pass == 0 ? tm_dv : tm_dk, stage + hb * 16384, hb * 64, j * 128 + w * 32, h_idx, b_idx);
            bulk_commit();
        }
        __syncwarp();
    }
    // the stores must have read shared memory (and be complete) before the CTA exits
    if (lane == 0) bulk_wait0();
    __syncwarp();
}

// Warps 4-7: stage LSE / D two blocks ahead, read each dQ part out of tensor
// memory (freeing its columns for Y) and add it into the fp32 buffer through
// shared memory and TMA reductions.
template <int D>
__device__ void dq_role(const CUtensorMap* tm_dq, uint32_t tY, int w, int lane, uint8_t* smem, uint64_t* bars,
                        volatile int* abort_flag, int bh, int i0, int nq, const BwdArgs& a) {
    using C = Cfg<D>;
    const uint64_t lim = a.wait_limit_ns;
    const int wq = w & 3;
    const int r = wq * 32 + lane;                             // tensor-memory lane = query within the block
    const uint32_t ly = tY + ((uint32_t)(wq * 32) << 16) + C::kTdQ;
    float* lse_s = reinterpret_cast<float*>(smem + C::kOffLse);
    float* dsc_s = lse_s + 2 * 128;
    // this warp's slot: two boxes of [32 rows][32 fp32], each row one 128-byte
    // line with its 16-byte chunks swizzled by the row (the tensor map's layout)
    uint8_t* slot = smem + C::kOffDQ + wq * 8192;
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        bool got = wait_or_abort(bar, parity, lim, abort_flag);
        return __all_sync(0xffffffffu, got);
    };
    auto fetch = [&](int it) -> float2 {
        const int q = (i0 + it) * 128 + r;
        if (q >= a.N) return make_float2(-INFINITY, 0.f);
        return make_float2(-(a.lse[(int64_t)bh * a.N + q] * kLog2e), -(a.dsum[(int64_t)bh * a.N + q] * a.scale));
    };
    auto stage = [&](int it, float2 val) {
        const int b = it & 1;
        lse_s[b * 128 + r] = val.x;
        dsc_s[b * 128 + r] = val.y;
        mbar_arrive(&bars[kBarLseFull + b]);
    };
    stage(0, fetch(0));
    if (nq > 1) stage(1, fetch(1));
    for (int it = 0; it < nq; ++it) {
        const float2 next_val = (it + 2 < nq) ? fetch(it + 2) : make_float2(0.f, 0.f);
        if (!wait_warp(&bars[kBarDqReady], (uint32_t)(it & 1))) break;
        tc_fence_after();
        uint32_t v[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32_nowait(ly + c * 32, v + c * 32);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld_wait32(v + c * 32);
        tc_fence_before();
        mbar_arrive(&bars[kBarDqRead]);
        // the compute warps finished with this buffer before Y could form this dQ part
        if (it + 2 < nq) stage(it + 2, next_val);
        const int row0 = (i0 + it) * 128 + wq * 32;           // first query row of this warp
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {                    // 64 columns (two boxes) at a time
            if (lane == 0) bulk_wait_read0();                 // the slot's previous reductions have read it
            __syncwarp();
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int e = h * 64 + b * 32 + c * 4;
                    st_shared16(smem_u32(slot + b * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)),
                                make_uint4(v[e], v[e + 1], v[e + 2], v[e + 3]));
                }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < a.N) {
                for (int b = 0; b < 2; ++b)
                    if (h * 64 + b * 32 < a.d) tma_reduce_add_3d(tm_dq, slot + b * 4096, h * 64 + b * 32, row0, bh);
                bulk_commit();
            }
        }
    }
    // the reductions must have read the slot before the CTA exits, and be
    // complete before the kernel's end hands the buffer to the cast
    if (lane == 0) bulk_wait0();
    __syncwarp();
}

}  // namespace bwd

// One CTA per (key block j, batch*head); heavier key blocks (small j under causal masking) first.
// kF16: q, k, v, o, dO and the gradients are fp16 instead of bf16.
template <int D, bool kF16>
__global__ void __launch_bounds__(bwd::kThreads, 1)
attn_bwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                      const __grid_constant__ CUtensorMap tm_dv, const bwd::BwdArgs a) {
    using C = bwd::Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;
    if (C::kPad) {
        smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    } else if (smem_u32(smem_raw) & 1023u) {
        // the swizzled tiles need 1024-byte alignment and there is no room to pad
        if (threadIdx.x == 0) atomicCAS(&g_attn_device_status, 0, (int)ATTN_ERR_LAUNCH);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int j = blockIdx.x / a.BH, bh = blockIdx.x % a.BH;
    const int i0 = a.causal ? j : 0;
    const int nq = a.nkv - i0;

    if (threadIdx.x == 0) {
        mbar_init(&bars[bwd::kBarKV], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[bwd::kBarQFull + s], 1);
            mbar_init(&bars[bwd::kBarQEmpty + s], 2);
            mbar_init(&bars[bwd::kBarLseFull + s], 128);
        }
        mbar_init(&bars[bwd::kBarDoFull], 1);
        mbar_init(&bars[bwd::kBarDoEmpty], 2);
        mbar_init(&bars[bwd::kBarSFull], 1);
        mbar_init(&bars[bwd::kBarPReady], 256);
        mbar_init(&bars[bwd::kBarDpFull], 1);
        mbar_init(&bars[bwd::kBarDsReady], 256);
        mbar_init(&bars[bwd::kBarDqReady], 1);
        mbar_init(&bars[bwd::kBarDqRead], 128);
        mbar_init(&bars[bwd::kBarDrainX], 1);
        mbar_init(&bars[bwd::kBarDrainY], 1);
        mbar_init(&bars[bwd::kBarDsHalf], 128);
        mbar_init(&bars[bwd::kBarNever], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == bwd::kWarpProducer && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_dq);
        prefetch_tmap(&tm_dk);
        prefetch_tmap(&tm_dv);
    }
    if (warp == bwd::kWarpMmaX) {
        tmem_alloc(tmem_slot, bwd::kCols);
        tmem_alloc(tmem_slot + 1, bwd::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tX = tmem_slot[0], tY = tmem_slot[1];

    if (warp < bwd::kWarpDq || (warp >= bwd::kWarpCompute1 && warp < bwd::kWarpProducer)) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(bwd::kRegsCompute));
        bwd::compute_role<D, kF16>(&tm_dk, &tm_dv, tX, tY, warp & 3, warp < bwd::kWarpDq ? 0 : 1, lane, smem, bars,
                                   abort_flag, bh, j, nq, a);
    } else if (warp < bwd::kWarpCompute1) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(bwd::kRegsDq));
        bwd::dq_role<D>(&tm_dq, tY, warp, lane, smem, bars, abort_flag, bh, i0, nq, a);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(bwd::kRegsControl));
        if (warp == bwd::kWarpProducer) {
            if (lane == 0) bwd::producer<D>(&tm_q, &tm_k, &tm_v, &tm_do, smem, bars, abort_flag, bh, j, i0, nq, a);
            __syncwarp();
        } else if (warp == bwd::kWarpMmaX) {
            if (lane == 0) bwd::mma_x<D, kF16>(tX, smem, bars, abort_flag, nq, a);
            __syncwarp();
        } else if (warp == bwd::kWarpMmaY) {
            if (lane == 0) bwd::mma_y<D, kF16>(tY, smem, bars, abort_flag, nq, a);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == bwd::kWarpMmaX) {
        tmem_dealloc(tX, bwd::kCols);
        tmem_dealloc(tY, bwd::kCols);
    }
}

// D = rowsum(dO * O) - dLSE in fp32 per row, and the fp32 dQ buffer zeroed.
// A row is d / 8 lanes (16-byte loads of 8 values), so one warp covers
// 32 / (d / 8) rows at a time (two at d = 128, four at d = 64); grid-stride.
template <bool kF16>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                           const uint16_t* __restrict__ dout,
                                                           const float* __restrict__ dlse,
                                                           float* __restrict__ dsum, float* __restrict__ dq_acc,
                                                           int64_t rows, int d) {
    const int lane = threadIdx.x % 32;
    const int lanes_per_row = d <= 8 ? 1 : d <= 16 ? 2 : d <= 32 ? 4 : d <= 64 ? 8 : 16;
    const int rows_per_warp = 32 / lanes_per_row;
    const int sub = lane / lanes_per_row, c = (lane % lanes_per_row) * 8;
    const int64_t warps = (int64_t)gridDim.x * blockDim.x / 32;
    for (int64_t row0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32 * rows_per_warp; row0 < rows;
         row0 += warps * rows_per_warp) {
        const int64_t row = row0 + sub;
        float s = 0.f;
        if (row < rows && c < d) {
            const uint4 ov = *reinterpret_cast<const uint4*>(o + row * d + c);
            const uint4 gv = *reinterpret_cast<const uint4*>(dout + row * d + c);
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float o0, o1, g0, g1;
                bwd::unpack2<kF16>(ow[e], o0, o1);
                bwd::unpack2<kF16>(gw[e], g0, g1);
                s += o0 * g0 + o1 * g1;
            }
            float4* z = reinterpret_cast<float4*>(dq_acc + row * d + c);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int off = lanes_per_row / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (row < rows && lane % lanes_per_row == 0) dsum[row] = dlse ? s - dlse[row] : s;
    }
}

// dQ: the fp32 accumulation buffer to the element type, eight values per step
// (n % 8 == 0); grid-stride.
template <bool kF16>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const float* __restrict__ dq_acc,
                                                            uint16_t* __restrict__ dq, int64_t n8) {
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n8;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(dq_acc) + 2 * idx);
        const float4 b = __ldcs(reinterpret_cast<const float4*>(dq_acc) + 2 * idx + 1);
        uint4 w;
        w.x = pack2<kF16>(a.x, a.y);
        w.y = pack2<kF16>(a.z, a.w);
        w.z = pack2<kF16>(b.x, b.y);
        w.w = pack2<kF16>(b.z, b.w);
        reinterpret_cast<uint4*>(dq)[idx] = w;
    }
}

// ------------------------------------------------------------------ host side

template <int D, bool kF16>
int launch_bwd_d(const AttnBwdParams& p, cudaStream_t stream, int dev) {
    using C = bwd::Cfg<D>;
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return ATTN_ERR_CUDA;
    const int BH = p.B * p.H;
    CUtensorMap mq, mk, mv, mdo, mdk, mdv;
    long long st[3];                                  // dense [B, H, N, d]
    set_strides(st, (long long)p.H * p.N * p.d, (long long)p.N * p.d, p.d);
    if (!encode_qkv_map(enc, &mq, p.q, p.B, p.H, p.N, p.d, st, 128, kF16) ||
        !encode_qkv_map(enc, &mk, p.k, p.B, p.H, p.N, p.d, st, 128, kF16) ||
        !encode_qkv_map(enc, &mv, p.v, p.B, p.H, p.N, p.d, st, 128, kF16) ||
        !encode_qkv_map(enc, &mdo, p.dout, p.B, p.H, p.N, p.d, st, 128, kF16) ||
        !encode_qkv_map(enc, &mdk, p.dk, p.B, p.H, p.N, p.d, st, 32, kF16) ||   // 32-row boxes: one per warp
        !encode_qkv_map(enc, &mdv, p.dv, p.B, p.H, p.N, p.d, st, 32, kF16))
        return ATTN_ERR_BAD_SHAPE;
    const int64_t rows = (int64_t)BH * p.N;
    float* dq_acc = static_cast<float*>(p.workspace);
    const size_t acc_bytes = ((size_t)rows * p.d * sizeof(float) + 255) & ~(size_t)255;
    float* dsum = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + acc_bytes);
    // the fp32 dQ buffer [BH, N, d] for the TMA reductions: boxes of 32 rows x
    // 32 columns (128 bytes, the 128-byte swizzle span)
    CUtensorMap mdq;
    {
        cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.N, (cuuint64_t)BH};
        cuuint64_t strides[2] = {(cuuint64_t)p.d * 4, (cuuint64_t)p.N * p.d * 4};
        cuuint32_t box[3] = {32, 32, 1};
        cuuint32_t elem[3] = {1, 1, 1};
        if (enc(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dq_acc, dims, strides, box, elem,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return ATTN_ERR_BAD_SHAPE;
    }
    // per-device caches, shared by host threads (the values are idempotent)
    static std::atomic<int> attr_done[64];
    if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(attn_bwd_sm103_kernel<D, kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_LAUNCH;
        }
        if (dev >= 0 && dev < 64) attr_done[dev].store(1, std::memory_order_relaxed);
    }
    static std::atomic<int> sms_cache[64];
    int sms = (dev >= 0 && dev < 64) ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) sms_cache[dev].store(sms, std::memory_order_relaxed);
    }
    // the two element-wise passes: grid-stride, 8 blocks of 256 threads per SM
    const int64_t pre_rows_per_block = 8 * (32 / (p.d <= 8 ? 1 : p.d <= 16 ? 2 : p.d <= 32 ? 4 : p.d <= 64 ? 8 : 16));
    const int64_t pre_need = (rows + pre_rows_per_block - 1) / pre_rows_per_block;
    const int64_t pre_blocks = pre_need < (int64_t)sms * 8 ? pre_need : (int64_t)sms * 8;
    attn_bwd_pre_kernel<kF16><<<(unsigned)pre_blocks, 256, 0, stream>>>(
        static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.dlse, dsum, dq_acc, rows, p.d);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    bwd::BwdArgs a;
    a.BH = BH;
    a.H = p.H;
    a.N = p.N;
    a.d = p.d;
    a.nkv = (p.N + 127) / 128;
    a.causal = p.causal;
    a.scale = p.scale;
    a.c2 = (float)((double)p.scale * 1.4426950408889634);
    a.lse = p.lse;
    a.dsum = dsum;
    a.dq_acc = dq_acc;
    a.wait_limit_ns = g_wait_limit_ns;
    a.test_stall = g_test_stall;
    const int64_t grid = (int64_t)BH * a.nkv;
    attn_bwd_sm103_kernel<D, kF16><<<(unsigned)grid, bwd::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq, mdk, mdv, a);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    const int64_t n8 = rows * p.d / 8;
    const int64_t post_need = (n8 + 255) / 256;
    const int64_t post_blocks = post_need < (int64_t)sms * 8 ? post_need : (int64_t)sms * 8;
    attn_bwd_post_kernel<kF16><<<(unsigned)post_blocks, 256, 0, stream>>>(dq_acc, static_cast<uint16_t*>(p.dq), n8);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

size_t attn_bwd_workspace(int B, int H, int N, int d) {
    const size_t rows = (size_t)B * H * N;
    const size_t acc = (rows * d * sizeof(float) + 255) & ~(size_t)255;
    return acc + ((rows * sizeof(float) + 255) & ~(size_t)255);
}

int launch_attn_bwd(const AttnBwdParams& p, cudaStream_t stream, int dev) {
    if (p.f16) return p.d <= 64 ? launch_bwd_d<64, true>(p, stream, dev) : launch_bwd_d<128, true>(p, stream, dev);
    return p.d <= 64 ? launch_bwd_d<64, false>(p, stream, dev) : launch_bwd_d<128, false>(p, stream, dev);
}

}  // namespace bos
