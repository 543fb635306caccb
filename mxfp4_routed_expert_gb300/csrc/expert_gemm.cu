// Routed experts as a grouped tcgen05 GEMM (prefill and large batches).
//
// The arithmetic is the one of the decode GEMVs (kimi-k3-in-c README, Part II
// section 4, k3_matmul_mxfp4, and section 9, k3_moe step 3): for every
// (token, expert) pair, g = W1_e z, u = W3_e z, h = SiTU(g, u), then
// acc_token += w_pair * W2_e h. The weights are MXFP4 (e2m1 nibbles, low
// nibble = even column, one ue8m0 scale per 32 columns) and are read as
// stored.
//
// Work: the pairs of expert e (contiguous in permutation order) are cut into
// n-tiles of at most 64; a work item is (n-tile, 128-row m-tile of the
// matrix). Weight rows are the MMA's M, pairs its N. Per 128-column k-stage:
//   - one thread issues TMA for the packed weight tiles (128 rows x 64 bytes
//     per matrix, 64-byte swizzle) into a deep ring that the converters
//     release as soon as they have read a stage, and another for the item's
//     pair-ordered fp16 activation rows (the gathered latent z for W1/W3, the
//     h rows for W2; two 64-column halves in the 128-byte swizzled K-major
//     layout, 16-row boxes) into a ring that the MMAs release;
//   - sixteen converter warps (four per TMEM lane quadrant) widen the nibbles
//     with cvt.rn.f16x2.e2m1x2 and multiply each 32-column group by
//     2^(s - smax_row), smax_row being the row's largest scale byte: every
//     factor is a power of two <= 1, so the f16 operand is the exact weight /
//     2^(smax_row - 127) unless a row spans more than 23 binades of scales
//     (0.5 and 1.5 times 2^-24 fall between f16 subnormals).
//     They store it straight into tensor memory (tcgen05.st: row m in lane m,
//     column c = columns 2c, 2c+1), the MMA's A operand, so that shared memory
//     carries only packed weights and activations;
//   - two threads issue tcgen05.mma kind::f16 (A from TMEM, B from shared
//     memory) into fp32 TMEM accumulators, one each. W1/W3: gate and up of
//     the same 128 rows. W2: two adjacent 128-row m-tiles per item when the
//     latent width allows (so each activation tile feeds 256 weight rows), else
//     the two halves of every k-stage, summed in the epilogue. With 64-pair
//     n-tiles two accumulator sets let the next item's MMAs overlap this
//     item's epilogue; the rest of TMEM holds the A ring. An A slot is reused
//     once the activation stage of the k-stage that last held it is
//     released, which both issuers' commits signal;
//   - the epilogue (four dedicated warps with two accumulator sets, else the
//     converter warps between items) reads TMEM, multiply by 2^(smax_row - 127) and the
//     token's activation exponent, then apply SiTU (hardware tanh) and store
//     h (W1/W3), or
//     scale by the pair's routing weight and scatter-add into the token's fp32
//     latent accumulator (W2).
// All waits are bounded (mbar_wait); a role that gives up latches the error
// word and leaves its loop, the producer waits for its own copies still in
// flight, and the CTA frees its TMEM before returning.
#include "k3moe_internal.cuh"
#include "tc_common.cuh"

namespace k3 {

namespace {

constexpr int BM = 128, BK = 128;
constexpr int kMinPairs = 128;                      // smallest batch (token, expert pairs) run here
// warp roles: 0 weight TMA producer, 1 and 2 MMA issuers, 3 activation TMA producer, 4..19 converters,
// 20..23 epilogue (warp % 4 = its TMEM lane quadrant)
constexpr int kConvWarp0 = 4, kConvWarps = 16;
constexpr int kEpiWarp0 = 20, kEpiWarps = 4;
constexpr int kThreads = 24 * 32;
constexpr int kRawRow = BK / 2;                     // packed bytes per row and k-stage
constexpr int kRawBytes = BM * kRawRow;             // one packed weight tile
constexpr int kBoxRows = 16;                        // activation rows per TMA box
constexpr int kSmemBudget = 227 * 1024;
constexpr uint32_t kTmemCols = 512;

// Kernel modes: W1/W3 together (kW13), W2 with the two halves of each k-stage
// on the two issuers (kW2), or W2 with two adjacent 128-row m-tiles per item
// (kW2Pair: the activation tile then feeds twice the weight rows).
enum : int { kW13 = 0, kW2 = 1, kW2Pair = 2 };

// Launch geometry for a mode with n-tiles of BN pairs. TMEM holds
// SETS accumulator sets of two BN-column accumulators (two sets for BN <= 64,
// so that the epilogue overlaps the next item; one for BN = 128), then the
// ring of converted A slots in the remaining columns (256, or 384 for BN = 32). Shared memory holds
// two TMA rings: activation tiles (NB stages, released by the MMAs) and packed
// weight tiles (NR stages, released by the converters as soon as they have
// read them, so that weight loads run far ahead of the tensor cores).
template <int MODE, int BN>
struct Geo {
    static_assert(BN == 32 || BN == 64 || BN == 128, "n-tile of 32, 64 or 128 pairs");
    static constexpr int NM = MODE == kW2 ? 1 : 2;           // weight tiles per k-stage
    static constexpr int SETS = BN <= 64 ? 2 : 1;
    static constexpr uint32_t SET_COLS = 2 * BN;
    static constexpr uint32_t ARING0 = SETS * SET_COLS;     // 128 or 256
    static constexpr int ACOLS = NM * BK / 2;                // TMEM columns per A slot
    static constexpr int NSA = (int)(kTmemCols - ARING0) / ACOLS;
    static constexpr int BSUB = BN * 128;                    // one 64-column half of the activation tile
    static constexpr int BBYTES = 2 * BSUB;                  // one activation stage [half 0 | half 1]
    static constexpr int RBYTES = NM * kRawBytes;            // one weight stage [packed W per matrix]
    static constexpr size_t smem(int nb, int nr)
    {
        return (size_t)nb * BBYTES + (size_t)nr * RBYTES +
               (size_t)(2 * nb + 2 * nr + NSA + 2 * SETS + 2 * tc::ItemQueue::kQ) * 8 + 16 +
               4 * tc::ItemQueue::kQ + 1024;
    }
    // activation stages: deep enough to cover an L2 fetch under load (about
    // 2k cycles for a 32 KB stage) at the tensor-bound stage time
    static constexpr int NB = BBYTES >= 32768 ? 5 : 6;
    static constexpr int ring()                              // weight stages: what is left, at most 16
    {
        int nr = 2;
        while (nr < 16 && smem(NB, nr + 1) <= (size_t)kSmemBudget) nr++;
        return nr;
    }
    static constexpr int NR = ring();
    static constexpr size_t SMEM = smem(NB, NR);
    static_assert(ARING0 <= 256 && NSA >= 2, "accumulators leave room for two A slots");
    static_assert(NB >= NSA, "A slots are released through the activation ring");
    static_assert(SMEM <= (size_t)kSmemBudget && NR >= 4, "shared memory");
};

struct EgArgs {
    const uint8_t *sa, *sb;      // scale rows [E*R, K/32] (W1 and W3, or W2)
    const uint8_t *ma, *mb;      // largest scale byte per row [E*R]
    int K, R, MT;                // input width, rows per expert, items per expert along the rows
    int mstep, mrow;             // rows per item (128, or 256 for kW2Pair); second tile's row offset
    int k, L, I;
    const int *offsets, *perm;
    const int2 *tiles;           // (expert, n-tile index) per n-tile
    const int *n_tiles;
    const float *pair_w;         // [T*k] routing weight per pair slot
    const __half *zp;            // gathered latent [T*k, L + kZPad], exponent in the padding
    __half *h16;                 // [T*k, I]
    float *acc;                  // [T, L]
    float b1, b2, ib1, ib2;      // SiTU bounds and their reciprocals
    const int *wslot;            // expert -> index in the weight arrays (nullptr: the expert)
    int *ticket;                 // items handed out so far (zero at launch)
    int n_ws;                    // experts the weight arrays hold
    int *err;
};

// Index of expert e in the weight arrays: its expert-tier slot, or e itself.
__device__ __forceinline__ int eg_wslot(const EgArgs &g, int e)
{
    if (!g.wslot) return e;
    const int s = g.wslot[e];
    if (s < 0 || s >= g.n_ws) {
        set_err(g.err, kErrBounds, 620);
        return 0;
    }
    return s;
}

// 2^d as an f16x2 bit pattern, d <= 0 (subnormal below 2^-14, zero below 2^-24).
__device__ __forceinline__ uint32_t f16x2_pow2(int d)
{
    uint32_t b;
    if (d >= -14) b = (uint32_t)(d + 15) << 10;
    else if (d >= -24) b = 1u << (d + 24);
    else b = 0u;
    return b | (b << 16);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 2^(s - 127) for a scale byte in [0, 254]; 0 gives the subnormal 2^-127 (255 is
// refused at load).
__device__ __forceinline__ float pow2_e8m0(int s)
{
    return e8m0_to_f32((uint32_t)s);
}


// 16 packed bytes (32 columns, one scale group) -> 16 f16x2 scaled by f.
__device__ __forceinline__ void widen_group(uint4 w, uint32_t f, uint32_t *o)
{
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
        uint32_t h0, h1, h2, h3;
        e2m1x8_to_f16x2x4(words[j], h0, h1, h2, h3);
        o[4 * j + 0] = hmul2(h0, f);
        o[4 * j + 1] = hmul2(h1, f);
        o[4 * j + 2] = hmul2(h2, f);
        o[4 * j + 3] = hmul2(h3, f);
    }
}

// A from tensor memory, B from shared memory.
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
                 "r"(v[15])
                 : "memory");
}

// Epilogue of one item: the calling warp reads its TMEM lane quadrant
// (rows 32 (warp % 4) .. + 31 of the tile) for the pair columns c_first,
// c_first + CSTEP, ... (16 at a time), applies the row and token factors and
// SiTU (W1/W3) or the weighted scatter-add (W2), then releases the
// accumulator set. The per-pair factors are fetched before the wait for the
// accumulators, so their latency overlaps the item's last MMAs.
template <int MODE, int BN, int CSTEP>
__device__ __forceinline__ bool epilogue_item(const EgArgs &g, uint32_t tmem, int item, int local,
                                              uint64_t *tfull, uint64_t *tempty, int c_first)
{
    using GE = Geo<MODE, BN>;
    constexpr bool IS13 = MODE == kW13;
    constexpr int NCH = BN / CSTEP > 0 ? BN / CSTEP : 1;   // chunks of 16 columns per warp (upper bound)
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;   // TMEM lanes 32q..32q+31
    const int erow = q * 32 + lane;         // weight row of the tile
    const int tile = item / g.MT, mt = item - tile * g.MT;
    const int2 td = g.tiles[tile];
    const int cnt = g.offsets[td.x + 1] - g.offsets[td.x];
    const int n_valid = min(BN, cnt - td.y * BN);
    const int pair0 = g.offsets[td.x] + td.y * BN;
    const int row_in_e = mt * g.mstep + erow;
    const size_t grow = (size_t)eg_wslot(g, td.x) * g.R + row_in_e;
    const float rs0 = pow2_e8m0(g.ma[grow]);
    const float rs1 = GE::NM == 2 ? pow2_e8m0(g.mb[grow + g.mrow]) : 0.f;
    // per-pair factors for the columns of each chunk, one lane each (lanes 16..31 repeat 0..15)
    float pf[NCH];       // W1/W3: 2^(token exponent); W2: routing weight
    int pt[NCH];         // W2: token
#pragma unroll
    for (int ci = 0; ci < NCH; ci++) {
        const int c = c_first + ci * CSTEP + (lane & 15);
        pf[ci] = 0.f;
        pt[ci] = 0;
        if (c < n_valid) {
            const int pl = pair0 + c;
            if (IS13) {
                const int ex = *reinterpret_cast<const int *>(g.zp + (size_t)pl * (g.L + kZPad) + g.L);
                pf[ci] = __uint_as_float((uint32_t)(127 + ex) << 23);
            } else {
                pf[ci] = g.pair_w[pl];
                pt[ci] = g.perm[pl] / g.k;
            }
        }
    }
    const int b = local % GE::SETS;
    if (!mbar_wait(&tfull[b], (uint32_t)(local / GE::SETS) & 1u, g.err, 606)) return false;
    tc::fence_after();
    const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * GE::SET_COLS;
#pragma unroll
    for (int ci = 0; ci < NCH; ci++) {
        const int c0 = c_first + ci * CSTEP;
        if (c0 >= n_valid) break;
        float v0[16], v1[16];
        tc::tmem_ld16(tb + (uint32_t)c0, v0);
        tc::tmem_ld16(tb + (uint32_t)(BN + c0), v1);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const float fj = __shfl_sync(0xffffffffu, pf[ci], j);
            const int tj = IS13 ? 0 : __shfl_sync(0xffffffffu, pt[ci], j);
            if (c0 + j < n_valid) {
                const int p = pair0 + c0 + j;
                if (IS13) {
                    g.h16[(size_t)p * g.I + row_in_e] =
                        __float2half_rn(situ_hw(v0[j] * rs0 * fj, v1[j] * rs1 * fj, g.b1, g.b2, g.ib1, g.ib2));
                } else if (MODE == kW2) {
                    atomicAdd(&g.acc[(size_t)tj * g.L + row_in_e], fj * ((v0[j] + v1[j]) * rs0));
                } else {
                    float *ar = g.acc + (size_t)tj * g.L + row_in_e;
                    atomicAdd(ar, fj * (v0[j] * rs0));
                    atomicAdd(ar + g.mrow, fj * (v1[j] * rs1));
                }
            }
        }
    }
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&tempty[b]);
    return true;
}

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_expert_gemm(const __grid_constant__ CUtensorMap ra, const __grid_constant__ CUtensorMap rb,
                  const __grid_constant__ CUtensorMap bx, const __grid_constant__ CUtensorMap bxm,
                  const __grid_constant__ CUtensorMap bxf, EgArgs g)
{
    using GE = Geo<MODE, BN>;
    constexpr bool DUAL = GE::NM == 2;   // two weight tiles per k-stage, one per issuer
    extern __shared__ unsigned char raw_smem[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(raw_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int NB = GE::NB, NR = GE::NR, NSA = GE::NSA, ACOLS = GE::ACOLS;
    constexpr int kSets = GE::SETS, kBSub = GE::BSUB, kBBytes = GE::BBYTES, kRBytes = GE::RBYTES;
    constexpr uint32_t kSetCols = GE::SET_COLS, kARing0 = GE::ARING0;
    unsigned char *bring = sm;                                // [NB] activation stages
    unsigned char *wring = sm + NB * kBBytes;                 // [NR] packed weight stages
    uint64_t *bfull = reinterpret_cast<uint64_t *>(wring + NR * kRBytes);   // activation tile landed
    uint64_t *bfree = bfull + NB;                             // both issuers' MMAs on the stage done
    uint64_t *wfull = bfree + NB;                             // weight tile landed
    uint64_t *wfree = wfull + NR;                             // converters have read it
    uint64_t *aready = wfree + NR;                            // [NSA] A slot written
    uint64_t *tfull = aready + NSA;                           // [kSets] accumulator set complete
    uint64_t *tempty = tfull + kSets;                         // [kSets] epilogue drained it
    tc::ItemQueue iq;                                         // items of this CTA, in order
    iq.full = tempty + kSets;
    iq.empty = iq.full + tc::ItemQueue::kQ;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(iq.empty + tc::ItemQueue::kQ);
    iq.item = reinterpret_cast<int *>(tslot + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NB; i++) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bfree[i], 2);
        }
        for (int i = 0; i < NR; i++) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wfree[i], kConvWarps / 2);   // the warps of one parity read a stage
        }
        for (int i = 0; i < NSA; i++) mbar_init(&aready[i], kConvWarps / 2);
        for (int i = 0; i < kSets; i++) {
            mbar_init(&tfull[i], 2);
            mbar_init(&tempty[i], kSets == 2 ? kEpiWarps : kConvWarps);
        }
        // the weight producer claims the items; the activation producer, the
        // two MMA issuers, the converters and (two sets) the epilogue warps read them
        iq.init(3 + kConvWarps + (kSets == 2 ? kEpiWarps : 0));
        fence_mbar_init();
        tc::prefetch_map(&ra);
        if (DUAL) tc::prefetch_map(&rb);
        tc::prefetch_map(&bx);
        tc::prefetch_map(&bxm);
        tc::prefetch_map(&bxf);
    }
    if (warp == 1) tc::tmem_alloc(tslot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t tmem = *tslot;
    const int n_items = *g.n_tiles * g.MT;
    const int KT = g.K / BK;

    if (warp == 0 || warp == 3) {
        // ---------------- TMA producers: weights (warp 0), activations (warp 3) ----------------
        // Each ring's stages are refilled in k-stage order once their consumers
        // release them; before exiting, a producer waits for its own copies
        // still in flight (a stage holds at most one unconsumed fill).
        if (lane == 0) {
            const bool wts = warp == 0;
            const int depth = wts ? NR : NB;
            uint64_t *fullb = wts ? wfull : bfull;
            uint64_t *freeb = wts ? wfree : bfree;
            int it = 0, slot = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int i = 0; ok; i++) {
                const int item = wts ? iq.claim(g.ticket, n_items, i, g.err, 630) : iq.read_one(i, g.err, 631);
                if (item < 0) break;
                const int tile = item / g.MT, mt = item - tile * g.MT;
                const int2 td = g.tiles[tile];
                const int row0 = eg_wslot(g, td.x) * g.R + mt * g.mstep;   // row in the [slots*R, K/2] view
                const int pair0 = g.offsets[td.x] + td.y * BN;
                const int cnt = g.offsets[td.x + 1] - g.offsets[td.x];
                const int nv = min(BN, cnt - td.y * BN);
                // Activation rows per 64-column half: up to 32 pairs in 16-row
                // boxes, else one box of 64 or BN rows (rows past the tile's
                // pairs are never read by the MMA). A thread issues a TMA copy
                // only every ~100 cycles, so a stage takes at most four.
                const int nb = nv <= 32 ? (nv + kBoxRows - 1) / kBoxRows : 1;
                const int brows = nv <= 32 ? nb * kBoxRows : (nv <= 64 ? 64 : BN);
                const CUtensorMap *bmap = nv <= 32 ? &bx : (nv <= 64 ? &bxm : &bxf);
                const uint32_t tx = wts ? (uint32_t)kRBytes : (uint32_t)(2 * brows * 128);
                for (int kt = 0; kt < KT; kt++, it++) {
                    if (!mbar_wait(&freeb[slot], phase ^ 1u, g.err, wts ? 600 : 608)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&fullb[slot], tx);
                    if (wts) {
                        unsigned char *st = wring + slot * kRBytes;
                        tc::tma_load_2d(st, &ra, kt * kRawRow, row0, &fullb[slot]);
                        if (DUAL) tc::tma_load_2d(st + kRawBytes, &rb, kt * kRawRow, row0 + g.mrow, &fullb[slot]);
                    } else {
                        unsigned char *st = bring + slot * kBBytes;
                        for (int u = 0; u < 2; u++)
                            for (int bx_ = 0; bx_ < nb; bx_++)
                                tc::tma_load_2d(st + u * kBSub + bx_ * kBoxRows * 128, bmap, kt * BK + u * 64,
                                                pair0 + bx_ * kBoxRows, &fullb[slot]);
                    }
                    if (++slot == depth) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int j = 1; j <= depth && j <= it; j++) {
                const int u = it - j;
                mbar_wait(&fullb[u % depth], (uint32_t)(u / depth) & 1u, g.err, 605);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers ----------------
        // W1/W3 and paired W2: issuer q multiplies weight tile q; plain W2:
        // issuer q takes the k-steps 4q..4q+3 of every k-stage. Each writes
        // accumulator q of the set.
        // The whole warp runs the loop, so that its descriptor arithmetic is
        // warp-uniform; all lanes poll the barriers and one elected lane
        // issues (faster than one thread running it alone, most of all at
        // small N where the issue rate bounds the stage).
        const int q = warp - 1;
        {
            int local = 0;
            tc::RingPos<NB> bp;
            tc::RingPos<NSA> ap;
            const uint64_t db0 = tc::desc_sw128(tc::su32(bring));
            const int kk0 = DUAL ? 0 : 4 * q;            // first k-step (of 16 columns)
            constexpr int NK = DUAL ? BK / 16 : BK / 32; // k-steps per k-stage for this issuer
            bool ok = true;
            for (; ok; local++) {
                const int item = iq.read_warp(local, g.err, 632);
                if (item < 0) break;
                const int tile = item / g.MT;
                const int2 td = g.tiles[tile];
                const int cnt = g.offsets[td.x + 1] - g.offsets[td.x];
                const int n = ((min(BN, cnt - td.y * BN) + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t idesc =
                    (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);  // f16 x f16 -> f32
                const int b = local % kSets;
                if (!tc::warp_wait(&tempty[b], ((uint32_t)(local / kSets) & 1u) ^ 1u, g.err, 601)) break;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)b * kSetCols + (uint32_t)q * BN;
                for (int kt = 0; kt < KT; kt++, bp.next(), ap.next()) {
                    if (!tc::warp_wait(&aready[ap.slot], ap.phase, g.err, 603) ||
                        !tc::warp_wait(&bfull[bp.slot], bp.phase, g.err, 609)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t a0 = tmem + kARing0 + (uint32_t)(ap.slot * ACOLS) + (DUAL ? (uint32_t)q * (BK / 2) : 0u);
                    const uint64_t db = db0 + (uint64_t)((bp.slot * kBBytes) >> 4);
                    if (tc::elect_one()) {
#pragma unroll
                        for (int i = 0; i < NK; i++) {
                            const int kk = kk0 + i;
                            // B: half kk / 4 of the activation tile, 32 bytes per k-step inside it
                            const uint64_t bd = db + (uint64_t)(((kk >> 2) * kBSub + (kk & 3) * 32) >> 4);
                            mma_ts(d, a0 + 8 * (uint32_t)kk, bd, idesc, (kt > 0 || i > 0) ? 1u : 0u);
                        }
                        tc::commit(&bfree[bp.slot]);
                    }
                    __syncwarp();
                }
                if (ok && tc::elect_one()) tc::commit(&tfull[b]);
                __syncwarp();
            }
        }
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
        // ---------------- converters: packed e2m1 -> scaled f16 -> TMEM ----------------
        // The warps alternate k-stages (sl & 1 = the parity of the stages a warp
        // takes), so that each warp's fixed per-stage cost (barrier waits and
        // arrivals) spreads over two stage times. Per stage, the eight warps
        // of a parity cover the four lane quadrants twice: one weight tile
        // each (all four scale groups), or for plain W2 two scale groups each.
        const int qd = warp & 3;                      // TMEM lane quadrant
        const int row = qd * 32 + lane;               // weight row of the tile (its TMEM lane)
        const int sl = (warp - kConvWarp0) >> 2;      // 0..3
        const int par = sl & 1;
        const int m = DUAL ? (sl >> 1) : 0;           // weight tile
        const int grp0 = DUAL ? 0 : 2 * (sl >> 1);    // first scale group within the k-stage
        constexpr int NGRP = DUAL ? 4 : 2;
        const uint32_t tlane = (uint32_t)(qd * 32) << 16;
        const int G = g.K / kGroup;
        const int swz = (row >> 1) & 3;              // 64-byte swizzle of the packed tile
        tc::RingPos<NR> wp;           // weight stage of this k-stage
        tc::RingPos<NB> rq;           // activation stage of the k-stage NSA back (its MMAs free the A slot)
        tc::RingPos<NSA> ap;
        int done = 0;             // k-stages of this CTA so far
        int local = 0;            // items of this CTA so far
        bool ok = true;
        // With one accumulator set the issuers stop between items until the
        // accumulators are drained, so the converters run the epilogue
        // themselves (each warp a quarter of the pair columns of its lane
        // quadrant) right after converting their first k-stage of the next
        // item, whose A slot frees up before the previous item's last MMAs end.
        int prev_item = -1;       // the item before this one (its epilogue may still be due)
        for (; ok; local++) {
            const int item = iq.read_warp(local, g.err, 633);
            if (item < 0) break;
            const int tile = item / g.MT, mt = item - tile * g.MT;
            const size_t grow = (size_t)eg_wslot(g, g.tiles[tile].x) * g.R + mt * g.mstep + row + (m ? g.mrow : 0);
            const int smax = m == 0 ? g.ma[grow] : g.mb[grow];
            const uint8_t *sc = (m == 0 ? g.sa : g.sb) + grow * (size_t)G + grp0;   // G % 4 == 0
            bool epi = kSets == 1 && local > 0;      // previous item's epilogue still to run
            for (int kt = 0; kt < KT; kt++, wp.next(), ap.next(), done++) {
                const bool mine = (done & 1) == par;
                if (done >= NSA) {
                    if (mine && !mbar_wait(&bfree[rq.slot], rq.phase, g.err, 607)) {
                        ok = false;
                        break;
                    }
                    rq.next();
                }
                if (!mine) continue;
                uint32_t sv4;
                if (NGRP == 4) sv4 = *reinterpret_cast<const uint32_t *>(sc + 4 * kt);
                else sv4 = *reinterpret_cast<const uint16_t *>(sc + 4 * kt);
                if (!mbar_wait(&wfull[wp.slot], wp.phase, g.err, 604)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const unsigned char *rawp = wring + wp.slot * kRBytes + m * kRawBytes + row * kRawRow;
                const uint32_t acol = kARing0 + (uint32_t)(ap.slot * ACOLS) + (uint32_t)(m * (BK / 2));
                uint4 w[NGRP];
#pragma unroll
                for (int i = 0; i < NGRP; i++)   // 16-byte chunk = scale group of the row
                    w[i] = *reinterpret_cast<const uint4 *>(rawp + (((grp0 + i) ^ swz) << 4));
                __syncwarp();
                if (lane == 0) mbar_arrive(&wfree[wp.slot]);
#pragma unroll
                for (int i = 0; i < NGRP; i++) {
                    uint32_t v[16];
                    // groups above the row's largest scale hold only zeros (the row
                    // maximum skips them): any factor <= 1 leaves them zero
                    widen_group(w[i], f16x2_pow2(min((int)((sv4 >> (8 * i)) & 0xffu) - smax, 0)), v);
                    tmem_st16(tmem + tlane + acol + (uint32_t)(16 * (grp0 + i)), v);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&aready[ap.slot]);
                if (epi) {
                    epi = false;
                    if (!epilogue_item<MODE, BN, 64>(g, tmem, prev_item, local - 1, tfull, tempty, 16 * sl)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (ok && epi &&   // an item with no k-stage of this warp's parity
                !epilogue_item<MODE, BN, 64>(g, tmem, prev_item, local - 1, tfull, tempty, 16 * sl))
                ok = false;
            prev_item = item;
        }
        if (kSets == 1 && ok && local > 0)
            epilogue_item<MODE, BN, 64>(g, tmem, prev_item, local - 1, tfull, tempty, 16 * sl);
    } else if (kSets == 2 && warp >= kEpiWarp0) {
        // ---------------- epilogue (two accumulator sets) ----------------
        for (int local = 0;; local++) {
            const int item = iq.read_warp(local, g.err, 634);
            if (item < 0 || !epilogue_item<MODE, BN, 16>(g, tmem, item, local, tfull, tempty, 0)) break;
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// n-tiles of at most bn pairs: (expert, j) for j < ceil(count_e / bn),
// experts ascending; also zeroes the grouped GEMMs' item counters. One block.
__global__ void __launch_bounds__(1024) k_expert_tiles(const int *counts, int E, int bn, int2 *tiles, int *n_tiles,
                                                      int *ticket)
{
    __shared__ int wsum[32];
    pdl_launch_dependents();
    pdl_wait();
    const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = e < E ? counts[e] : 0;
    const int nt = (c + bn - 1) / bn;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < 32; w++) {
        if (w < warp) base += wsum[w];
        total += wsum[w];
    }
    const int first = base + incl - nt;
    for (int j = 0; j < nt; j++) tiles[first + j] = make_int2(e, j);
    if (threadIdx.x == 0) {
        *n_tiles = total;
        ticket[0] = 0;   // the two grouped GEMM launches that follow hand out items from 0
        ticket[1] = 0;
    }
}

// zp[p] = z16[token of pair p] (L values and the exponent padding); one warp per pair.
__global__ void __launch_bounds__(256) k_gather_latent(const __half *z16, const int *perm, __half *zp,
                                                       int pairs, int k, int L, const int *offsets, int E)
{
    pdl_launch_dependents();
    pdl_wait();
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (p >= pairs || p >= offsets[E]) return;   // offsets[E]: the pairs kept this forward
    const int t = perm[p] / k;
    const int nv = (L + kZPad) / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(z16 + (size_t)t * (L + kZPad));
    uint4 *dst = reinterpret_cast<uint4 *>(zp + (size_t)p * (L + kZPad));
    for (int i = lane; i < nv; i += 32) dst[i] = src[i];
}

// Largest scale byte of every row of an expert matrix stack [rows, G]; load time.
// Only groups with a nonzero nibble count (magnitude bits 0-2 of either
// nibble): a group of zeros contributes nothing whatever its scale, so a large
// scale byte on it must not push the row's real groups below the f16 range.
// One warp per row; a row without any nonzero nibble gets 0. Load time.
__global__ void __launch_bounds__(256) k_row_scale_max(const uint8_t *packed, const uint8_t *s, size_t rows, int G,
                                                       uint8_t *out)
{
    const size_t r = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const uint4 *pr = reinterpret_cast<const uint4 *>(packed + r * (size_t)G * 16);
    const uint8_t *sr = s + r * (size_t)G;
    int m = 0;
    for (int i = lane; i < G; i += 32) {
        const uint4 v = pr[i];
        if (((v.x | v.y | v.z | v.w) & 0x77777777u) != 0u) m = max(m, (int)sr[i]);
    }
    m = (int)__reduce_max_sync(0xffffffffu, (unsigned)m);
    if (lane == 0) out[r] = (uint8_t)m;
}

// Packed weights [rows, cols bytes], boxes of box_cols x box_rows with the
// 64-byte swizzle (16-byte chunk c of row r lands at chunk c ^ ((r >> 1) & 3)).
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                 uint32_t box_rows)
{
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// f16 [rows, cols], row pitch `pitch` elements, 64-column boxes, 128-byte swizzle.
bool make_map_f16_sw128(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint64_t pitch,
                        uint32_t box_rows)
{
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool expert_gemm_ok(const k3moe_config &c)
{
    return c.latent % BK == 0 && c.moe_inter % BK == 0 && c.latent % BM == 0 && c.moe_inter % BM == 0 &&
           (long long)c.max_tokens * c.topk >= kMinPairs;
}

bool expert_mx_ok(const k3moe_config &c)
{
    return c.latent > 0 && c.moe_inter > 0 && c.latent % BK == 0 && c.moe_inter % BK == 0 &&
           c.latent % BM == 0 && c.moe_inter % BM == 0;
}

size_t expert_gemm_max_tiles(const k3moe_config &c)
{
    return (size_t)((long long)c.max_tokens * c.topk / 32 + c.n_experts + 1);   // the narrowest n-tile
}

int expert_gemm_min_pairs() { return kMinPairs; }

template <int MODE, int BN>
cudaError_t set_smem()
{
    return cudaFuncSetAttribute(k_expert_gemm<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Geo<MODE, BN>::SMEM);
}

cudaError_t init_expert_gemm()
{
    cudaError_t e = set_smem<kW13, 32>();
    if (e == cudaSuccess) e = set_smem<kW2, 32>();
    if (e == cudaSuccess) e = set_smem<kW2Pair, 32>();
    if (e == cudaSuccess) e = set_smem<kW13, 64>();
    if (e == cudaSuccess) e = set_smem<kW2, 64>();
    if (e == cudaSuccess) e = set_smem<kW2Pair, 64>();
    if (e == cudaSuccess) e = set_smem<kW13, 128>();
    if (e == cudaSuccess) e = set_smem<kW2, 128>();
    if (e == cudaSuccess) e = set_smem<kW2Pair, 128>();
    return e;
}

// n-tile width of a launch, from the average pairs per expert: 32 when the
// experts see a few tokens each (narrow accumulators leave TMEM for a third A
// slot), 64 below 64 pairs (two accumulator sets), else 128 (every converted
// weight tile then feeds twice the MMA work, with one set).
bool use_expert_split(const k3moe &h, int T)
{
    const long long pairs = (long long)T * h.cfg.topk;
    return h.mx_ok && h.expert_path == K3MOE_EXPERT_MX && pairs < kMinPairs && pairs <= kSplitPairsMax;
}

// Which grouped GEMM a batch that takes the grouped path runs: the
// block-scaled one when asked for, or automatically while the experts see
// fewer than 64 pairs each on average (the weights dominate the bytes each SM
// takes in, and the block-scaled kernel streams them with no conversion);
// above that the f16 one, whose operands take fewer bytes per pair (its
// packed weights are widened in registers, the block-scaled MMA's stay one
// byte per nibble in shared memory).
bool expert_gemm_mx(const k3moe &h, int T)
{
    if (h.expert_path == K3MOE_EXPERT_MX) return true;
    if (h.expert_path != K3MOE_EXPERT_AUTO) return false;
    return (long long)T * h.cfg.topk < 64LL * h.cfg.n_experts;
}

// The block-scaled path (mx) takes 96 in place of 128: the widest tile for
// which two W1/W3 accumulator sets and its scale-factor ring fit in TMEM.
int expert_gemm_bn(const k3moe &h, int T, bool mx)
{
    const long long pairs = (long long)T * h.cfg.topk, E = h.cfg.n_experts;
    return pairs <= 4 * E ? 32 : (pairs < 64 * E ? 64 : (mx ? 96 : 128));
}

cudaError_t launch_expert_tiles(const k3moe &h, int T, cudaStream_t s, bool mx)
{
    return launch_pdl(k_expert_tiles, 1, 1024, 0, s, (const int *)h.ws.counts, h.cfg.n_experts,
                      expert_gemm_bn(h, T, mx), h.ws.tiles, h.ws.n_tiles, h.ws.eg_ticket);
}

cudaError_t launch_gather_latent(const k3moe &h, int T, cudaStream_t s)
{
    const int pairs = T * h.cfg.topk;
    return launch_pdl(k_gather_latent, (pairs + 7) / 8, 256, 0, s, (const __half *)h.ws.z16,
                      (const int *)h.ws.perm, h.ws.zperm, pairs, h.cfg.topk, h.cfg.latent,
                      (const int *)h.ws.offsets, h.cfg.n_experts);
}

// W1/W3 (w13 = true: gathered latent -> h16) or W2 (h16 -> acc).
cudaError_t launch_expert_gemm(const k3moe &h, const LayerDev &w, int T, cudaStream_t s, bool w13)
{
    const k3moe_config &c = h.cfg;
    const int pairs = T * c.topk;
    const int bn = expert_gemm_bn(h, T, false);   // the width the tile list was built for
    if (pairs < kMinPairs) return cudaErrorInvalidValue;
    EgArgs g = {};
    g.k = c.topk;
    g.L = c.latent;
    g.I = c.moe_inter;
    g.offsets = h.ws.offsets;
    g.perm = h.ws.perm;
    g.tiles = h.ws.tiles;
    g.n_tiles = h.ws.n_tiles;
    g.pair_w = h.ws.pair_w;
    g.zp = h.ws.zperm;
    g.h16 = h.ws.h16;
    g.acc = h.ws.acc;
    g.b1 = c.situ_b1;
    g.b2 = c.situ_b2;
    g.ib1 = 1.f / c.situ_b1;
    g.ib2 = 1.f / c.situ_b2;
    g.err = h.ws.err;
    g.ticket = h.ws.eg_ticket + (w13 ? 0 : 1);
    g.wslot = w.wslot;
    g.n_ws = w.n_wslots;
    g.K = w13 ? c.latent : c.moe_inter;
    g.R = w13 ? c.moe_inter : c.latent;
    // W2 takes two adjacent m-tiles per item when its rows allow it
    const int mode = w13 ? kW13 : (c.latent % (2 * BM) == 0 ? kW2Pair : kW2);
    g.mstep = mode == kW2Pair ? 2 * BM : BM;
    g.mrow = mode == kW2Pair ? BM : 0;
    g.MT = g.R / g.mstep;
    CUtensorMap ra, rb, bx, bxm, bxf;
    bool ok;
    const uint64_t rows = (uint64_t)w.n_wslots * g.R;
    if (w13) {
        g.sa = w.w1s;
        g.sb = w.w3s;
        g.ma = w.w1max;
        g.mb = w.w3max;
        ok = make_map_u8(&ra, w.w1p, rows, g.K / 2, kRawRow, BM) &&
             make_map_u8(&rb, w.w3p, rows, g.K / 2, kRawRow, BM) &&
             make_map_f16_sw128(&bx, h.ws.zperm, pairs, c.latent, c.latent + kZPad, kBoxRows) &&
             make_map_f16_sw128(&bxm, h.ws.zperm, pairs, c.latent, c.latent + kZPad, bn < 64 ? bn : 64) &&
             make_map_f16_sw128(&bxf, h.ws.zperm, pairs, c.latent, c.latent + kZPad, bn);
    } else {
        g.sa = g.sb = w.w2s;
        g.ma = g.mb = w.w2max;
        ok = make_map_u8(&ra, w.w2p, rows, g.K / 2, kRawRow, BM) &&
             make_map_f16_sw128(&bx, h.ws.h16, pairs, c.moe_inter, c.moe_inter, kBoxRows) &&
             make_map_f16_sw128(&bxm, h.ws.h16, pairs, c.moe_inter, c.moe_inter, bn < 64 ? bn : 64) &&
             make_map_f16_sw128(&bxf, h.ws.h16, pairs, c.moe_inter, c.moe_inter, bn);
        rb = ra;
    }
    if (!ok) return cudaErrorInvalidValue;
#define K3_EG_LAUNCH(M, N) launch_pdl(k_expert_gemm<M, N>, h.sm_count, kThreads, Geo<M, N>::SMEM, s, ra, rb, bx, bxm, bxf, g)
    if (bn == 128)
        return mode == kW13 ? K3_EG_LAUNCH(kW13, 128) : (mode == kW2 ? K3_EG_LAUNCH(kW2, 128) : K3_EG_LAUNCH(kW2Pair, 128));
    if (bn == 64)
        return mode == kW13 ? K3_EG_LAUNCH(kW13, 64) : (mode == kW2 ? K3_EG_LAUNCH(kW2, 64) : K3_EG_LAUNCH(kW2Pair, 64));
    return mode == kW13 ? K3_EG_LAUNCH(kW13, 32) : (mode == kW2 ? K3_EG_LAUNCH(kW2, 32) : K3_EG_LAUNCH(kW2Pair, 32));
#undef K3_EG_LAUNCH
}

cudaError_t launch_row_scale_max(const uint8_t *packed, const uint8_t *s, size_t rows, int G, uint8_t *out)
{
    k_row_scale_max<<<(unsigned)((rows + 7) / 8), 256>>>(packed, s, rows, G, out);
    return cudaGetLastError();
}

}  // namespace k3
