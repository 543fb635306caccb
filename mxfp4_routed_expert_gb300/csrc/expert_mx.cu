// Routed experts as a grouped block-scaled tcgen05 GEMM (prefill and large
// batches).
//
// The arithmetic is the one of the decode GEMVs (kimi-k3-in-c README, Part II
// section 9, k3_moe step 3): for every (token, expert) pair, g = W1_e z,
// u = W3_e z, h = SiTU(g, u), then acc_token += w_pair * W2_e h. The weights
// are the checkpoint's MXFP4 (section 4: e2m1 nibbles, low nibble = even
// column, one ue8m0 scale per 32 columns), read as stored and never
// re-encoded.
//
// tcgen05.mma.kind::mxf8f6f4.block_scale multiplies them directly with 8-bit
// activations: A = 128 weight rows (TMA with the 16U4_ALIGN16B unpacking
// lands the nibbles in the K-major, 128-byte swizzled layout the MMA reads),
// B = activation rows of the item's pairs in e4m3, both operands' ue8m0 scale
// factors from tensor memory, fp32 accumulators in tensor memory. The tensor
// core applies every scale exactly (byte 0 = 2^-127 and the largest bytes
// included), so no row is rebased or flushed whatever its scale range.
//
// Activations are two-term MXFP8: v = hi 2^eh + lo 2^el per 32-value group
// (hi, lo e4m3), about 8 significant bits more than one e4m3 term, so the
// layer stays within its tolerance. Each k-step runs two MMAs into the same
// accumulator (B = hi tile, then lo tile with its own scales): the MMA time
// of the f16 path, with no operand conversion on the SM.
//
// Work: the pairs of expert e (contiguous in permutation order) form n-tiles
// of BN pairs; an item is (n-tile, 128-row m-tile of the matrix). One
// persistent CTA per SM walks the items. Per 128-column k-stage:
//   - warp 0 (one lane) loads the weight tiles (W1 and W3, or W2; 8 KB packed
//     each, 16 KB in shared memory) into a ring of weight stages, warp 3 (one
//     lane) the hi and lo activation tiles of the item's pairs (128 bytes per
//     row) into a ring of activation stages;
//   - warps 4..7 and 16..19 (even and odd stages), one per TMEM lane
//     quadrant in each group, write the stage's scale factors
//     into a slot of a ring in tensor memory: per weight tile four columns of
//     row scale words (row r in lane r % 32, column r / 32), per activation
//     term BN / 32 columns of pair scale words (pair c in lane c % 32, column
//     c / 32), the same words in every quadrant; byte j of a word scales the
//     k-stage's 32-column group j;
//   - warp 1 (one elected lane) issues the MMAs of K = 32 (the instruction
//     descriptor's scale-factor ids pick byte j) and commits the stages'
//     release;
//   - warps 8..15 (two per lane quadrant, half the pair columns each) drain an
//     accumulator set: W1/W3: SiTU (hardware tanh) and h in two-term MXFP8;
//     W2: times the pair's routing weight, scatter-added into the token's
//     fp32 latent accumulator. Two sets (when tensor memory holds them) let
//     the next item's MMAs overlap this item's epilogue.
// Every wait is bounded (mbar_wait); a role that gives up latches the error
// word and leaves its loop, the producers wait for their own copies still in
// flight, and the CTA frees its tensor memory before returning.
#include "k3moe_internal.cuh"
#include "tc_common.cuh"

namespace k3 {

namespace {

constexpr int BM = 128, BK = 128;
constexpr int kThreads = 20 * 32;
// warp roles: 0 weight TMA, 1 MMA issuer, 2 tensor-memory allocation, 3
// activation TMA, 4..7 scale writers of even stages, 8..15 epilogue, 16..19
// scale writers of odd stages (warp % 4 = the TMEM lane quadrant it may access)
constexpr int kWriterWarp0 = 4, kEpiWarp0 = 8, kWriter2Warp0 = 16;
constexpr int kBoxRows = 16;                    // activation rows per TMA box for small tiles
constexpr int kSmemBudget = 227 * 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCols = 16;                // per scale slot: 2 x 4 weight columns, 2 x 4 pair columns
constexpr int kSfSlots = 8;

// W1/W3 together (kW13), W2 one 128-row m-tile per item (kW2), or W2 with two
// adjacent 128-row m-tiles per item (kW2Pair: the activation tile then feeds
// twice the weight rows; when the latent width is a multiple of 256).
enum : int { kW13 = 0, kW2 = 1, kW2Pair = 2 };

template <int MODE, int BN>
struct MxGeo {
    static_assert(BN == 32 || BN == 64 || BN == 96, "n-tile of 32, 64 or 96 pairs");
    static constexpr int NA = MODE == kW2 ? 1 : 2;            // weight tiles (and accumulators) per stage
    static constexpr int ABYTES = NA * BM * 128;              // weight stage (unpacked nibbles)
    static constexpr int BHALF = BN * 128;                    // one activation term's tile
    static constexpr int BBYTES = 2 * BHALF;                  // activation stage: hi tile, lo tile
    static constexpr uint32_t SET_COLS = NA * BN;
    static constexpr int SETS = 2;                            // accumulator sets
    static constexpr uint32_t SF0 = SETS * SET_COLS;          // scale ring after the accumulators
    // activation stages (from L2): W2 keeps more of them (its weight tile is
    // half the size and its k-stage half the MMA time)
    static constexpr int NBS = MODE != kW2 ? (BBYTES >= 24576 ? 3 : 4) : (BBYTES >= 24576 ? 5 : 6);
    // W1/W3 epilogue staging: per epilogue warp 16 pairs x 32 rows of each e4m3 term
    static constexpr int ESTAGE = MODE == kW13 ? 8 * 1024 : 0;
    static constexpr size_t fixed() { return 1024 + 512 + ESTAGE; }   // alignment pad, barriers, staging
    static constexpr int ring()                               // weight stages (from HBM): what is left
    {
        int n = 2;
        while (n < 12 && (size_t)(n + 1) * ABYTES + (size_t)NBS * BBYTES + fixed() <= (size_t)kSmemBudget) n++;
        return n;
    }
    static constexpr int NAS = ring();
    static constexpr int D = NAS > kSfSlots ? (NAS > NBS ? NAS : NBS) : (kSfSlots > NBS ? kSfSlots : NBS);
    static constexpr size_t SMEM = (size_t)NAS * ABYTES + (size_t)NBS * BBYTES + fixed();
    static_assert(SF0 + kSfSlots * kSfCols <= kTmemCols, "tensor memory");
    static_assert(SMEM <= (size_t)kSmemBudget && NAS >= 3, "shared memory");
    static_assert(D >= NBS, "stage barriers cover every ring");
    static_assert((2 * D + 4 + 2 * tc::ItemQueue::kQ) * 8 + 16 + 4 * tc::ItemQueue::kQ <= 512, "barriers");
};

struct MxArgs {
    const uint8_t *sa, *sb;      // weight scale rows [slots*R, K/32] (W1 and W3, or W2 twice)
    const uint8_t *bs;           // activation scale rows [2*P, K/32] (plane 0 hi, plane 1 lo)
    int P;                       // rows of one activation plane (max tokens x k)
    int K, R, MT;                // input width, rows per expert, items per expert along the rows
    int mstep, mrow;             // rows per item (128, or 256 for kW2Pair); second tile's row offset
    int k, L, I;
    const int *offsets, *perm;
    const int2 *tiles;           // (expert, n-tile index) per n-tile
    const int *n_tiles;
    const float *pair_w;         // [T*k] routing weight per pair slot
    uint8_t *h8, *h8s;           // W1/W3 output: [2*P, I] e4m3, [2*P, I/32] scales
    float *acc;                  // W2 output: [T, L]
    float b1, b2, ib1, ib2;      // SiTU bounds and their reciprocals
    const int *wslot;            // expert -> index in the weight arrays (nullptr: the expert)
    int n_ws;
    int *ticket;                 // items handed out so far (zero at launch)
    // K split over KS items (small batches): an item is (n-tile, m-tile, K
    // range). W2 items add their partial products into acc like whole ones;
    // W1/W3 items add their partial gate and up sums into gu, and the last of
    // the 8 * KS epilogue warps of an (n-tile, m-tile) applies SiTU
    int KS;
    float *gu;                   // [pairs][2][I] partial W1 and W3 sums (zero between launches)
    int *gu_cnt;                 // [n-tiles * MT] epilogue warps arrived (zero between launches)
    int *err;
};

__device__ __forceinline__ int mx_wslot(const MxArgs &g, int e)
{
    if (!g.wslot) return e;
    const int s = g.wslot[e];
    if (s < 0 || s >= g.n_ws) {
        set_err(g.err, kErrBounds, 720);
        return 0;
    }
    return s;
}

// Item geometry: weight row of the tile's first row, first pair, valid pairs.
struct MxItem {
    int row0, pair0, nv, mt;
};

// Items of expert e (nt n-tiles, tile list entries first .. first + nt - 1)
// are MT * first .. MT * (first + nt) - 1, ordered m-tile outer, n-tile inner:
// the nt items that read the same weight tile follow one another, so CTAs
// that take them at about the same time share its bytes through L2 instead
// of each streaming the expert's weights from memory again.
template <int BN>
__device__ __forceinline__ MxItem mx_item(const MxArgs &g, int item)
{
    MxItem it;
    const int2 td = g.tiles[item / g.MT];                    // a tile of the item's expert
    const int e = td.x;
    const int first = item / g.MT - td.y;                    // the expert's first tile
    const int cnt = g.offsets[e + 1] - g.offsets[e];
    const int nt = (cnt + BN - 1) / BN;
    const int local = item - g.MT * first;
    it.mt = local / nt;
    const int j = local - it.mt * nt;
    it.row0 = mx_wslot(g, e) * g.R + it.mt * g.mstep;
    it.pair0 = g.offsets[e] + j * BN;
    it.nv = min(BN, cnt - j * BN);
    return it;
}

// Block-scaled MMA: A and B from shared memory, their scale factors from
// tensor memory. KEEP = 1: A stays in the collector buffer for the next MMA
// (fill); KEEP = 2: this MMA reuses it and lets it go (lastuse). The hi and
// lo MMAs of a weight tile share A, which halves the weight reads from shared
// memory (8-bit operands at M = N = 128 read about as many bytes per clock as
// shared memory delivers).
template <int KEEP>
__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate)
{
    if (KEEP == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X.collector::a::fill [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X.collector::a::lastuse [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A e2m1, B
// e4m3, both K-major, fp32 accumulate, ue8m0 scale factors, M = 128, N = n;
// the scale-factor ids (byte of the scale words) of A and B both j.
__device__ __forceinline__ uint32_t idesc_mx(int n, int j)
{
    return ((uint32_t)j << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24) | ((uint32_t)j << 29);
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_word(const uint8_t *p)
{
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

// Epilogue of one item by one warp: its TMEM lane quadrant (rows 32q .. 32q+31
// of the tile) for the pair columns [c_lo, c_hi), 16 at a time.
// W1/W3: the SiTU output of 16 pairs x the warp's 32 rows (one scale group
// per pair) goes through `stage` (1 KB of shared memory per warp: hi bytes,
// then lo bytes, [pair][row]) so that each lane writes 16 consecutive bytes of
// one pair's h row, instead of one byte per pair.
template <int MODE, int BN>
__device__ __forceinline__ void mx_epilogue(const MxArgs &g, const MxItem &m, uint32_t tacc, int q, int c_lo,
                                            int c_hi, uint8_t *stage)
{
    const int lane = threadIdx.x & 31;
    const int row = m.mt * g.mstep + q * 32 + lane;  // output row of this lane (within the expert)
    for (int c0 = c_lo; c0 < c_hi && c0 < m.nv; c0 += 16) {
        float v0[16];
        tc::tmem_ld16(tacc + (uint32_t)c0, v0);
        if (MODE == kW13) {
            float v1[16];
            tc::tmem_ld16(tacc + (uint32_t)(BN + c0), v1);
            uint32_t sh = 0, sl = 0;                 // scale bytes of pair c0 + lane (lanes 0..15)
#pragma unroll
            for (int j = 0; j < 16; j++) {
                // h in two-term MXFP8: the warp's 32 rows are one scale group of the
                // pair's h row (every lane takes part; a column's validity is uniform)
                const float hv = situ_hw(v0[j], v1[j], g.b1, g.b2, g.ib1, g.ib2);
                uint32_t qh, ql;
                int eh, el;
                mx8_hilo(hv, qh, ql, eh, el);
                stage[j * 32 + lane] = (uint8_t)qh;
                stage[512 + j * 32 + lane] = (uint8_t)ql;
                if (lane == j) {
                    sh = (uint32_t)(eh + 127);
                    sl = (uint32_t)(el + 127);
                }
            }
            __syncwarp();
            // lane L: pair c0 + L / 2, rows 16 (L % 2) .. +15 of the warp's 32
            const int cl = lane >> 1, hr = (lane & 1) * 16;
            if (c0 + cl < m.nv) {
                const size_t off = (size_t)(m.pair0 + c0 + cl) * g.I + (size_t)(row - lane + hr);
                *reinterpret_cast<uint4 *>(g.h8 + off) = *reinterpret_cast<const uint4 *>(stage + cl * 32 + hr);
                *reinterpret_cast<uint4 *>(g.h8 + (size_t)g.P * g.I + off) =
                    *reinterpret_cast<const uint4 *>(stage + 512 + cl * 32 + hr);
            }
            if (lane < 16 && c0 + lane < m.nv) {
                const size_t gs = (size_t)g.I / kGroup;
                const size_t sp = (size_t)(m.pair0 + c0 + lane) * gs + (size_t)((row - lane) / kGroup);
                g.h8s[sp] = (uint8_t)sh;
                g.h8s[(size_t)g.P * gs + sp] = (uint8_t)sl;
            }
            __syncwarp();
        } else {
            const int c = c0 + (lane & 15);
            float pw = 0.f;
            int pt = 0;
            if (c < m.nv) {
                pw = g.pair_w[m.pair0 + c];
                pt = g.perm[m.pair0 + c] / g.k;
            }
            float v1[16];
            if (MODE == kW2Pair) tc::tmem_ld16(tacc + (uint32_t)(BN + c0), v1);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const float wj = __shfl_sync(0xffffffffu, pw, j);
                const int tj = __shfl_sync(0xffffffffu, pt, j);
                if (c0 + j < m.nv) {
                    float *ar = g.acc + (size_t)tj * g.L + row;
                    atomicAdd(ar, wj * v0[j]);
                    if (MODE == kW2Pair) atomicAdd(ar + g.mrow, wj * v1[j]);
                }
            }
        }
    }
}

// W1/W3 epilogue of one warp of an item whose K range is a part of the
// whole: its lane quadrant's rows x the pair columns [c_lo, c_hi) of the
// partial gate and up sums are added into g.gu. The warp that completes the
// (n-tile, m-tile)'s 8 * KS arrivals then finishes the whole tile from g.gu:
// SiTU, h in two-term MXFP8 (one scale group = 32 rows of one pair, one warp
// at a time), g.gu and the counter left zeroed for the next launch.
template <int BN>
__device__ __forceinline__ void mx_epilogue_split(const MxArgs &g, const MxItem &m, int base, uint32_t tacc, int q,
                                                  int c_lo, int c_hi)
{
    const int lane = threadIdx.x & 31;
    const int row = m.mt * g.mstep + q * 32 + lane;
    for (int c0 = c_lo; c0 < c_hi && c0 < m.nv; c0 += 16) {
        float v0[16], v1[16];
        tc::tmem_ld16(tacc + (uint32_t)c0, v0);
        tc::tmem_ld16(tacc + (uint32_t)(BN + c0), v1);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            if (c0 + j < m.nv) {
                float *gp = g.gu + (size_t)(m.pair0 + c0 + j) * 2 * g.I + row;
                atomicAdd(gp, v0[j]);
                atomicAdd(gp + g.I, v1[j]);
            }
        }
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&g.gu_cnt[base], 1) == 8 * g.KS - 1;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    const size_t gs = (size_t)g.I / kGroup;
    for (int c = 0; c < m.nv; c++) {
        const int p = m.pair0 + c;
        float gv[4], uv[4];
#pragma unroll
        for (int grp = 0; grp < 4; grp++) {          // the tile's 128 rows: four scale groups
            const float *gp = g.gu + (size_t)p * 2 * g.I + m.mt * g.mstep + grp * 32 + lane;
            gv[grp] = __ldcg(gp);
            uv[grp] = __ldcg(gp + g.I);
        }
#pragma unroll
        for (int grp = 0; grp < 4; grp++) {
            const int r = m.mt * g.mstep + grp * 32 + lane;
            float *gp = g.gu + (size_t)p * 2 * g.I + r;
            gp[0] = 0.f;
            gp[g.I] = 0.f;
            uint32_t qh, ql;
            int eh, el;
            mx8_hilo(situ_hw(gv[grp], uv[grp], g.b1, g.b2, g.ib1, g.ib2), qh, ql, eh, el);
            g.h8[(size_t)p * g.I + r] = (uint8_t)qh;
            g.h8[((size_t)g.P + p) * g.I + r] = (uint8_t)ql;
            if (lane == 0) {
                g.h8s[(size_t)p * gs + r / kGroup] = (uint8_t)(eh + 127);
                g.h8s[((size_t)g.P + p) * gs + r / kGroup] = (uint8_t)(el + 127);
            }
        }
    }
    if (lane == 0) g.gu_cnt[base] = 0;
}

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_expert_mx(const __grid_constant__ CUtensorMap ra, const __grid_constant__ CUtensorMap rb,
                const __grid_constant__ CUtensorMap b16, const __grid_constant__ CUtensorMap b64,
                const __grid_constant__ CUtensorMap bfull_map, MxArgs g)
{
    using GE = MxGeo<MODE, BN>;
    constexpr int NA = GE::NA, NAS = GE::NAS, NBS = GE::NBS, SETS = GE::SETS, D = GE::D;
    extern __shared__ unsigned char raw_smem[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(raw_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *aring = sm;                                   // [NAS] weight stages
    unsigned char *bring = sm + NAS * GE::ABYTES;                // [NBS] activation stages
    // Stage s (the CTA's k-stages in order) uses weight slot s % NAS, activation
    // slot s % NBS and scale slot s % kSfSlots. ready[s % D] completes when its
    // two tiles have landed and its scales are written (the two producers
    // arrive with their byte counts, the four writers plainly); done[s % D]
    // when its MMAs have finished, which frees all three slots. A role waits
    // for stage s - depth to be done before refilling its slot; since D is at
    // least every depth, no barrier is reused before its waiters have seen it.
    uint8_t *estage = bring + NBS * GE::BBYTES;                // W1/W3 epilogue staging, 1 KB per warp
    uint64_t *ready = reinterpret_cast<uint64_t *>(estage + GE::ESTAGE);
    uint64_t *done = ready + D;
    uint64_t *tfull = done + D;                                  // [2] accumulator set complete
    uint64_t *tempty = tfull + 2;                                // [2] epilogue drained it
    tc::ItemQueue iq;                                            // items of this CTA, in order
    iq.full = tempty + 2;
    iq.empty = iq.full + tc::ItemQueue::kQ;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(iq.empty + tc::ItemQueue::kQ);
    iq.item = reinterpret_cast<int *>(tslot + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < D; i++) {
            mbar_init(&ready[i], 6);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        // the weight producer claims the items; the activation producer, the
        // MMA warp, the eight scale writers and the eight epilogue warps read them
        iq.init(18);
        fence_mbar_init();
        tc::prefetch_map(&ra);
        if (NA == 2) tc::prefetch_map(&rb);
        tc::prefetch_map(&b16);
        tc::prefetch_map(&b64);
        tc::prefetch_map(&bfull_map);
    }
    if (warp == 2) tc::tmem_alloc(tslot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t tmem = *tslot;
    const int n_items = *g.n_tiles * g.MT * g.KS;
    const int KT = g.K / BK;
    const int G = g.K / kGroup;

    if (warp == 0 || warp == 3) {
        // ---------------- TMA producers: weights (warp 0), activations (warp 3) ----------------
        if (lane == 0) {
            const bool wts = warp == 0;
            const int depth = wts ? NAS : NBS;
            int st = 0;
            bool ok = true;
            for (int i = 0; ok; i++) {
                const int item = wts ? iq.claim(g.ticket, n_items, i, g.err, 730) : iq.read_one(i, g.err, 731);
                if (item < 0) break;
                const int base = item / g.KS, ks = item - base * g.KS;   // (n-tile, m-tile), K part
                const MxItem m = mx_item<BN>(g, base);
                const int kt0 = KT * ks / g.KS, kt1 = KT * (ks + 1) / g.KS;
                // activation rows: up to 32 pairs in 16-row boxes, else one box of
                // 64 or BN rows (rows past the tile's pairs are never used)
                const int nb = m.nv <= 32 ? (m.nv + kBoxRows - 1) / kBoxRows : 1;
                const int brows = m.nv <= 32 ? nb * kBoxRows : (m.nv <= 64 ? 64 : BN);
                const CUtensorMap *bmap = m.nv <= 32 ? &b16 : (m.nv <= 64 ? &b64 : &bfull_map);
                // a 4-bit tile counts its packed bytes
                const uint32_t tx = wts ? (uint32_t)(NA * BM * 64) : (uint32_t)(2 * brows * 128);
                for (int kt = kt0; kt < kt1; kt++, st++) {
                    if (st >= depth && !mbar_wait(&done[(st - depth) % D], (uint32_t)((st - depth) / D) & 1u, g.err,
                                                  wts ? 700 : 701)) {
                        ok = false;
                        break;
                    }
                    uint64_t *bar = &ready[st % D];
                    mbar_expect_tx(bar, tx);
                    if (wts) {
                        unsigned char *dst = aring + (st % NAS) * GE::ABYTES;
                        tc::tma_load_2d(dst, &ra, kt * BK, m.row0, bar);
                        if (NA == 2) tc::tma_load_2d(dst + BM * 128, &rb, kt * BK, m.row0 + g.mrow, bar);
                    } else {
                        unsigned char *dst = bring + (st % NBS) * GE::BBYTES;
                        for (int t = 0; t < 2; t++)         // hi plane, lo plane
                            for (int b = 0; b < nb; b++)
                                tc::tma_load_2d(dst + t * GE::BHALF + b * kBoxRows * 128, bmap, kt * BK,
                                                t * g.P + m.pair0 + b * kBoxRows, bar);
                    }
                }
            }
            // before exiting, wait until the last stages' tiles have landed (the
            // MMAs of every stage this CTA runs end before its teardown anyway)
            for (int j = 1; j <= depth && j <= st; j++) {
                const int u = st - j;
                mbar_wait(&done[u % D], (uint32_t)(u / D) & 1u, g.err, 702);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        int local = 0, st = 0;
        bool ok = true;
        const uint64_t da0 = tc::desc_sw128(tc::su32(aring));
        const uint64_t db0 = tc::desc_sw128(tc::su32(bring));
        for (; ok; local++) {
            const int item = iq.read_warp(local, g.err, 732);
            if (item < 0) break;
            const int base = item / g.KS, ks = item - base * g.KS;   // (n-tile, m-tile), K part
            const MxItem m = mx_item<BN>(g, base);
            const int kt0 = KT * ks / g.KS, kt1 = KT * (ks + 1) / g.KS;
            const int n = ((m.nv + 15) / 16) * 16;
            const int b = local % SETS;
            if (!tc::warp_wait(&tempty[b], ((uint32_t)(local / SETS) & 1u) ^ 1u, g.err, 703)) break;
            tc::fence_after();
            const uint32_t d = tmem + (uint32_t)b * GE::SET_COLS;
            for (int kt = kt0; kt < kt1; kt++, st++) {
                if (!tc::warp_wait(&ready[st % D], (uint32_t)(st / D) & 1u, g.err, 704)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint64_t da = da0 + (uint64_t)(((st % NAS) * GE::ABYTES) >> 4);
                const uint64_t db = db0 + (uint64_t)(((st % NBS) * GE::BBYTES) >> 4);
                const uint32_t sf = tmem + GE::SF0 + (uint32_t)(st % kSfSlots) * kSfCols;
                if (tc::elect_one()) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {        // 32 columns (32 bytes of every tile) per MMA
                        const uint32_t id = idesc_mx(n, j);
#pragma unroll
                        for (int a = 0; a < NA; a++) {   // hi term (A kept), then lo term
                            const uint32_t da_ = d + (uint32_t)(a * BN);
                            const uint64_t aa = da + (uint64_t)((a * BM * 128) >> 4) + 2 * j;
                            mma_mx<1>(da_, aa, db + 2 * j, id, sf + 4 * a, sf + 8, (kt > kt0 || j > 0) ? 1u : 0u);
                            mma_mx<2>(da_, aa, db + (uint64_t)(GE::BHALF >> 4) + 2 * j, id, sf + 4 * a, sf + 12, 1u);
                        }
                    }
                    tc::commit(&done[st % D]);
                }
                __syncwarp();
            }
            if (ok && tc::elect_one()) tc::commit(&tfull[b]);
            __syncwarp();
        }
    } else if ((warp >= kWriterWarp0 && warp < kWriterWarp0 + 4) || warp >= kWriter2Warp0) {
        // ---------------- scale-factor writers ----------------
        // Lane i of the warp for lane quadrant q writes TMEM lane 32q + i: the
        // scale words of weight rows i, 32 + i, 64 + i, 96 + i of each weight tile
        // and of pairs i, 32 + i, ... of each activation term (the MMA reads the
        // copy of its own quadrant). Two groups of four warps take alternate
        // stages, so that each has two stage times for the load latency of its
        // words; the words of a stage are loaded before its slot is free, so
        // that their latency also overlaps the wait.
        const uint32_t tl = (uint32_t)((warp & 3) * 32) << 16;
        const int par = warp >= kWriter2Warp0 ? 1 : 0;
        int st = 0;
        bool ok = true;
        for (int i = 0; ok; i++) {
            const int item = iq.read_warp(i, g.err, 733);
            if (item < 0) break;
            const int base = item / g.KS, ks = item - base * g.KS;   // (n-tile, m-tile), K part
            const MxItem m = mx_item<BN>(g, base);
            const int kt0 = KT * ks / g.KS, kt1 = KT * (ks + 1) / g.KS;
            const uint8_t *arow0 = g.sa + (size_t)(m.row0 + lane) * G;
            const uint8_t *arow1 = g.sb + (size_t)(m.row0 + g.mrow + lane) * G;
            for (int kt = kt0; kt < kt1; kt++, st++) {
                if ((st & 1) != par) continue;
                uint32_t wa[2][4], hb[2][4];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    wa[0][c] = ld_word(arow0 + (size_t)(32 * c) * G + 4 * kt);
                    wa[1][c] = NA == 2 ? ld_word(arow1 + (size_t)(32 * c) * G + 4 * kt) : 0u;
                }
#pragma unroll
                for (int t = 0; t < 2; t++)
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int pc = 32 * c + lane;
                        hb[t][c] = (c < (BN + 31) / 32 && pc < m.nv)
                                       ? ld_word(g.bs + ((size_t)t * g.P + m.pair0 + pc) * G + 4 * kt)
                                       : 0u;
                    }
                if (st >= kSfSlots &&
                    !tc::warp_wait(&done[(st - kSfSlots) % D], (uint32_t)((st - kSfSlots) / D) & 1u, g.err, 707)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t col = tmem + tl + GE::SF0 + (uint32_t)(st % kSfSlots) * kSfCols;
                tmem_st4(col, wa[0][0], wa[0][1], wa[0][2], wa[0][3]);
                if (NA == 2) tmem_st4(col + 4, wa[1][0], wa[1][1], wa[1][2], wa[1][3]);
                tmem_st4(col + 8, hb[0][0], hb[0][1], hb[0][2], hb[0][3]);
                tmem_st4(col + 12, hb[1][0], hb[1][1], hb[1][2], hb[1][3]);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ready[st % D]);
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 8) {
        // ---------------- epilogue: two warps per lane quadrant ----------------
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2;
        const uint32_t tl = (uint32_t)(q * 32) << 16;
        constexpr int CH = ((BN / 2 + 15) / 16) * 16;   // pair columns per half, whole chunks of 16
        int local = 0;
        for (;; local++) {
            const int item = iq.read_warp(local, g.err, 734);
            if (item < 0) break;
            const int base = item / g.KS;                            // (n-tile, m-tile)
            const MxItem m = mx_item<BN>(g, base);
            const int b = local % SETS;
            if (!mbar_wait(&tfull[b], (uint32_t)(local / SETS) & 1u, g.err, 708)) break;
            tc::fence_after();
            if (MODE == kW13 && g.KS > 1)
                mx_epilogue_split<BN>(g, m, base, tmem + tl + (uint32_t)b * GE::SET_COLS, q, half * CH,
                                      min(BN, (half + 1) * CH));
            else
                mx_epilogue<MODE, BN>(g, m, tmem + tl + (uint32_t)b * GE::SET_COLS, q, half * CH,
                                      min(BN, (half + 1) * CH), estage + (warp - kEpiWarp0) * 1024);
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// zp[plane][p] = zq[plane][token of pair p] (L bytes) and the same for the
// scale rows (L / 32 bytes); one warp per pair.
__global__ void __launch_bounds__(256) k_gather_zq(const uint8_t *zq, const uint8_t *zqs, uint8_t *zp,
                                                   uint8_t *zps, const int *perm, int pairs, int k, int L,
                                                   int Tm, int P, const int *offsets, int E)
{
    pdl_launch_dependents();
    pdl_wait();
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (p >= pairs || p >= offsets[E]) return;   // offsets[E]: the pairs kept this forward
    const int t = perm[p] / k;
    const int G = L / kGroup;
#pragma unroll
    for (int pl = 0; pl < 2; pl++) {
        const uint4 *src = reinterpret_cast<const uint4 *>(zq + ((size_t)pl * Tm + t) * L);
        uint4 *dst = reinterpret_cast<uint4 *>(zp + ((size_t)pl * P + p) * L);
        for (int i = lane; i < L / 16; i += 32) dst[i] = src[i];
        const uint32_t *ss = reinterpret_cast<const uint32_t *>(zqs + ((size_t)pl * Tm + t) * G);
        uint32_t *sd = reinterpret_cast<uint32_t *>(zps + ((size_t)pl * P + p) * G);
        for (int i = lane; i < G / 4; i += 32) sd[i] = ss[i];
    }
}

// e2m1 weights [rows, K] (K/2 packed bytes per row), boxes of 128 elements x
// 128 rows, unpacked by the copy to one byte per nibble position (the
// 16U4_ALIGN16B form the f8f6f4 MMA kinds read) with the 128-byte swizzle.
bool make_map_e2m1(CUtensorMap *m, const void *base, uint64_t rows, uint64_t K)
{
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K / 2};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 activations [rows, K] bytes, boxes of 128 bytes x box_rows, 128-byte swizzle.
bool make_map_e4m3(CUtensorMap *m, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows)
{
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BN>
cudaError_t set_smem_mx()
{
    return cudaFuncSetAttribute(k_expert_mx<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)MxGeo<MODE, BN>::SMEM);
}

}  // namespace

cudaError_t init_expert_mx()
{
    cudaError_t e = set_smem_mx<kW13, 32>();
    if (e == cudaSuccess) e = set_smem_mx<kW13, 64>();
    if (e == cudaSuccess) e = set_smem_mx<kW13, 96>();
    if (e == cudaSuccess) e = set_smem_mx<kW2, 32>();
    if (e == cudaSuccess) e = set_smem_mx<kW2, 64>();
    if (e == cudaSuccess) e = set_smem_mx<kW2, 96>();
    if (e == cudaSuccess) e = set_smem_mx<kW2Pair, 32>();
    if (e == cudaSuccess) e = set_smem_mx<kW2Pair, 64>();
    if (e == cudaSuccess) e = set_smem_mx<kW2Pair, 96>();
    return e;
}

cudaError_t launch_gather_zq(const k3moe &h, int T, cudaStream_t s)
{
    const k3moe_config &c = h.cfg;
    const int pairs = T * c.topk;
    return launch_pdl(k_gather_zq, (pairs + 7) / 8, 256, 0, s, (const uint8_t *)h.ws.zq,
                      (const uint8_t *)h.ws.zqs, h.ws.zp8, h.ws.zps, (const int *)h.ws.perm, pairs, c.topk,
                      c.latent, c.max_tokens, c.max_tokens * c.topk, (const int *)h.ws.offsets, c.n_experts);
}

// W1/W3 (w13 = true: pair-ordered latent -> h) or W2 (h -> acc).
cudaError_t launch_expert_mx(const k3moe &h, const LayerDev &w, int T, cudaStream_t s, bool w13)
{
    const k3moe_config &c = h.cfg;
    const int pairs = T * c.topk;
    const int bn = expert_gemm_bn(h, T, true);   // the width the tile list was built for
    const bool split = pairs < expert_gemm_min_pairs();
    if (split && (pairs > kSplitPairsMax || !use_expert_split(h, T))) return cudaErrorInvalidValue;
    MxArgs g = {};
    g.P = c.max_tokens * c.topk;
    g.k = c.topk;
    g.L = c.latent;
    g.I = c.moe_inter;
    g.offsets = h.ws.offsets;
    g.perm = h.ws.perm;
    g.tiles = h.ws.tiles;
    g.n_tiles = h.ws.n_tiles;
    g.pair_w = h.ws.pair_w;
    g.h8 = h.ws.h8;
    g.h8s = h.ws.h8s;
    g.acc = h.ws.acc;
    g.b1 = c.situ_b1;
    g.b2 = c.situ_b2;
    g.ib1 = 1.f / c.situ_b1;
    g.ib2 = 1.f / c.situ_b2;
    g.wslot = w.wslot;
    g.n_ws = w.n_wslots;
    g.err = h.ws.err;
    g.ticket = h.ws.eg_ticket + (w13 ? 0 : 1);
    g.K = w13 ? c.latent : c.moe_inter;
    g.R = w13 ? c.moe_inter : c.latent;
    // W2 takes two adjacent m-tiles per item when its rows allow it
    const int mode = w13 ? kW13 : (c.latent % (2 * BM) == 0 ? kW2Pair : kW2);
    g.mstep = mode == kW2Pair ? 2 * BM : BM;
    g.mrow = mode == kW2Pair ? BM : 0;
    g.MT = g.R / g.mstep;
    // K split for small batches: about two items per SM, counting one n-tile
    // per pair (the most a batch of few pairs per expert has). Measured at K3
    // T = 1 (16 pairs): W1/W3 55 / 61 / 70 us with 1 / 2 / 4 parts per item,
    // W2 31 / 29 / 33 us with 1 / 2 / 6 parts; every item part carries a
    // fixed cost (its scale words, its accumulator hand-off, the partial sums)
    g.KS = 1;
    if (split) {
        const long long whole = (long long)pairs * g.MT;
        const long long want = (2LL * h.sm_count + whole - 1) / whole;
        g.KS = (int)std::max<long long>(1, std::min<long long>(want, g.K / BK));
    }
    g.gu = h.ws.gu;
    g.gu_cnt = h.ws.gu_cnt;
    const uint64_t rows = (uint64_t)w.n_wslots * g.R;
    const uint8_t *act = w13 ? h.ws.zp8 : h.ws.h8;
    g.bs = w13 ? h.ws.zps : h.ws.h8s;
    g.sa = w13 ? w.w1s : w.w2s;
    g.sb = w13 ? w.w3s : w.w2s;
    CUtensorMap ra, rb, b16, b64, bfl;
    bool ok = make_map_e2m1(&ra, w13 ? w.w1p : w.w2p, rows, g.K) &&
              make_map_e2m1(&rb, w13 ? w.w3p : w.w2p, rows, g.K) &&
              make_map_e4m3(&b16, act, 2 * (uint64_t)g.P, g.K, kBoxRows) &&
              make_map_e4m3(&b64, act, 2 * (uint64_t)g.P, g.K, bn < 64 ? bn : 64) &&
              make_map_e4m3(&bfl, act, 2 * (uint64_t)g.P, g.K, bn);
    if (!ok) return cudaErrorInvalidValue;
#define K3_MX_LAUNCH(M, N) \
    launch_pdl(k_expert_mx<M, N>, h.sm_count, kThreads, MxGeo<M, N>::SMEM, s, ra, rb, b16, b64, bfl, g)
    if (bn == 96)
        return mode == kW13 ? K3_MX_LAUNCH(kW13, 96) : (mode == kW2 ? K3_MX_LAUNCH(kW2, 96) : K3_MX_LAUNCH(kW2Pair, 96));
    if (bn == 64)
        return mode == kW13 ? K3_MX_LAUNCH(kW13, 64) : (mode == kW2 ? K3_MX_LAUNCH(kW2, 64) : K3_MX_LAUNCH(kW2Pair, 64));
    return mode == kW13 ? K3_MX_LAUNCH(kW13, 32) : (mode == kW2 ? K3_MX_LAUNCH(kW2, 32) : K3_MX_LAUNCH(kW2Pair, 32));
#undef K3_MX_LAUNCH
}

}  // namespace k3
