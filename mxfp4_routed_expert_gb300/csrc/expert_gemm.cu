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
// n-tiles of at most 128; a work item is (n-tile, 128-row m-tile of the
// matrix). Weight rows are the MMA's M, pairs its N, and both operands are
// K-major rows: packed weights, and the pair-ordered fp16 activations (the
// gathered latent z for W1/W3, the h rows for W2). Per 64-column k-tile:
//   - one thread issues TMA for the raw packed tile (128 rows x 32 bytes per
//     matrix) and the item's activation rows (16-row boxes of 128 bytes per
//     row, 128-byte swizzle) into a deep ring;
//   - eight converter warps widen the nibbles with cvt.rn.f16x2.e2m1x2 and
//     multiply each 32-column group by 2^(s - smax_row), smax_row being the
//     row's largest scale byte: every factor is a power of two <= 1, so the
//     f16 operand is the exact weight / 2^(smax_row - 127) unless a row spans
//     more than 24 binades of scales. They write the tile, in the swizzled
//     K-major layout the tensor core reads, into a two-slot ring of its own
//     (so the TMA ring stays deep enough to cover HBM latency);
//   - one thread issues tcgen05.mma kind::f16 into fp32 TMEM accumulators
//     (gate and up side by side for W1/W3), two accumulator sets so that the
//     next item's MMAs overlap this item's epilogue;
//   - four epilogue warps read TMEM, multiply by 2^(smax_row - 127) and the
//     token's activation exponent, then apply SiTU and store h (W1/W3), or
//     scale by the pair's routing weight and scatter-add into the token's fp32
//     latent accumulator (W2).
// All waits are bounded (mbar_wait); a role that gives up latches the error
// word and leaves its loop, the producer waits for its own copies still in
// flight, and the CTA frees its TMEM before returning.
#include "k3moe_internal.cuh"
#include "tc_common.cuh"

namespace k3 {

namespace {

constexpr int BM = 128, BK = 64, BN = 128;
// warp roles: 0 TMA producer, 1 and 2 MMA issuers, 3 idle, 4..11 converters,
// 12..15 epilogue (warp % 4 = its TMEM lane quadrant)
constexpr int kConvWarp0 = 4, kConvWarps = 8;       // two converter threads per weight row
constexpr int kEpiWarp0 = 12, kEpiWarps = 4;
constexpr int kThreads = 16 * 32;
constexpr int kRawRow = BK / 2;                     // packed bytes per row and k-tile
#ifndef K3_EG_ASTAGES
#define K3_EG_ASTAGES 2
#endif
constexpr int kAStages = K3_EG_ASTAGES;             // converted-tile ring
constexpr int kBoxRows = 16;                        // activation rows per TMA box
constexpr int kSmemBudget = 227 * 1024;

constexpr size_t smem_bytes(bool dual, int ns)
{
    return (size_t)kAStages * (dual ? 2 : 1) * BM * BK * 2 +
           (size_t)ns * (BN * BK * 2 + (dual ? 2 : 1) * BM * kRawRow) +
           (size_t)(2 * ns + kAStages + 4) * 8 + 16 + 1024;
}

// TMA ring depth: as many stages as the shared-memory budget holds (at most 12).
constexpr int ring_stages(bool dual)
{
    int ns = 2;
    while (ns < 12 && smem_bytes(dual, ns + 1) <= (size_t)kSmemBudget - 1024) ns++;
    return ns;
}

// Position in a ring of N slots: slot index and the parity of its current use.
template <int N>
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next()
    {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

struct EgArgs {
    const uint8_t *sa, *sb;      // scale rows [E*R, K/32] (W1 and W3, or W2)
    const uint8_t *ma, *mb;      // largest scale byte per row [E*R]
    int K, R, MT;                // input width, rows per expert, m-tiles per expert
    int k, L, I;
    const int *offsets, *perm;
    const int2 *tiles;           // (expert, n-tile index) per n-tile
    const int *n_tiles;
    const float *pair_w;         // [T*k] routing weight per pair slot
    const __half *zp;            // gathered latent [T*k, L + kZPad], exponent in the padding
    __half *h16;                 // [T*k, I]
    float *acc;                  // [T, L]
    float b1, b2;
    int *err;
};

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

// 2^(s - 127) for a scale byte in [1, 254] (0 and 255 clamp; 255 is refused at load).
__device__ __forceinline__ float pow2_e8m0(int s)
{
    return __uint_as_float((uint32_t)min(max(s, 1), 254) << 23);
}

template <bool DUAL>
__global__ void __launch_bounds__(kThreads, 1)
    k_expert_gemm(const __grid_constant__ CUtensorMap ra, const __grid_constant__ CUtensorMap rb,
                  const __grid_constant__ CUtensorMap bx, EgArgs g)
{
    extern __shared__ unsigned char raw_smem[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(raw_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int NM = DUAL ? 2 : 1;
    constexpr int A_BYTES = BM * BK * 2;     // one converted f16 weight tile
    constexpr int A_STAGE = NM * A_BYTES;
    constexpr int B_BYTES = BN * BK * 2;     // activation tile (up to 128 pair rows)
    constexpr int RAW_BYTES = BM * kRawRow;  // one packed weight tile
    constexpr int R_STAGE = B_BYTES + NM * RAW_BYTES;
    // TMEM: two accumulator sets of two 128-column accumulators. W1/W3: gate
    // and up; W2: the two halves of each k-tile (summed in the epilogue), so
    // that each MMA issuer owns one accumulator.
    constexpr uint32_t SET_COLS = 2 * BN;
    constexpr int NSR = ring_stages(DUAL);   // TMA ring depth
    static_assert(NSR > kAStages, "converted slots are released through the TMA ring");
    unsigned char *aring = sm;                               // [kAStages][A_STAGE]
    unsigned char *rring = sm + kAStages * A_STAGE;          // [NSR][R_STAGE]: B, then raw
    uint64_t *full = reinterpret_cast<uint64_t *>(rring + NSR * R_STAGE);   // TMA landed
    uint64_t *rfree = full + NSR;                            // both issuers' MMAs on the stage done
    uint64_t *aready = rfree + NSR;                          // [kAStages] converted tile written
    uint64_t *tfull = aready + kAStages;                     // [2] accumulator set complete
    uint64_t *tempty = tfull + 2;                            // [2] epilogue drained it
    uint32_t *tslot = reinterpret_cast<uint32_t *>(tempty + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSR; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&rfree[i], 2);
        }
        for (int i = 0; i < kAStages; i++) mbar_init(&aready[i], kConvWarps);
        for (int i = 0; i < 2; i++) {
            mbar_init(&tfull[i], 2);
            mbar_init(&tempty[i], kEpiWarps);
        }
        fence_mbar_init();
        tc::prefetch_map(&ra);
        if (DUAL) tc::prefetch_map(&rb);
        tc::prefetch_map(&bx);
    }
    if (warp == 1) tc::tmem_alloc(tslot, 2 * SET_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t tmem = *tslot;
    const int n_items = *g.n_tiles * g.MT;
    const int KT = g.K / BK;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0;
            RingPos<NSR> rp;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                const int tile = item / g.MT, mt = item - tile * g.MT;
                const int2 td = g.tiles[tile];
                const int row0 = td.x * g.R + mt * BM;          // row in the [E*R, K/2] view
                const int pair0 = g.offsets[td.x] + td.y * BN;
                const int cnt = g.offsets[td.x + 1] - g.offsets[td.x];
                const int nb = (min(BN, cnt - td.y * BN) + kBoxRows - 1) / kBoxRows;   // 16-row boxes
                const uint32_t tx = (uint32_t)(nb * kBoxRows * BK * 2 + NM * RAW_BYTES);
                for (int kt = 0; kt < KT; kt++, it++, rp.next()) {
                    const int s = rp.slot;
                    if (!mbar_wait(&rfree[s], rp.phase ^ 1u, g.err, 600)) {
                        ok = false;
                        break;
                    }
                    unsigned char *st = rring + s * R_STAGE;
                    mbar_expect_tx(&full[s], tx);
                    for (int b = 0; b < nb; b++)
                        tc::tma_load_2d(st + b * kBoxRows * 128, &bx, kt * BK, pair0 + b * kBoxRows, &full[s]);
                    tc::tma_load_2d(st + B_BYTES, &ra, kt * kRawRow, row0, &full[s]);
                    if (DUAL) tc::tma_load_2d(st + B_BYTES + RAW_BYTES, &rb, kt * kRawRow, row0, &full[s]);
                }
            }
            // copies still in flight land before the CTA exits (each stage holds at
            // most one unconsumed fill: a refill waits for the previous one's MMAs)
            for (int j = 1; j <= NSR && j <= it; j++) {
                const int u = it - j;
                mbar_wait(&full[u % NSR], (uint32_t)(u / NSR) & 1u, g.err, 605);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers ----------------
        // W1/W3: issuer q multiplies matrix q; W2: issuer q takes the k-steps
        // 2q, 2q+1 of every k-tile. Each writes accumulator q of the set.
        const int q = warp - 1;
        if (lane == 0) {
            int local = 0;
            RingPos<NSR> rp;
            RingPos<kAStages> ap;
            // shared-memory descriptors of slot 0; a byte offset o adds o >> 4
            const uint64_t da0 = tc::desc_sw128(tc::su32(aring)) + (uint64_t)(DUAL ? (q * A_BYTES) >> 4 : 0);
            const uint64_t db0 = tc::desc_sw128(tc::su32(rring));
            const int kk0 = DUAL ? 0 : 2 * q;            // first k-step (of 16 columns)
            constexpr int NK = DUAL ? BK / 16 : BK / 32; // k-steps per k-tile for this issuer
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, local++) {
                const int tile = item / g.MT;
                const int2 td = g.tiles[tile];
                const int cnt = g.offsets[td.x + 1] - g.offsets[td.x];
                const int n = ((min(BN, cnt - td.y * BN) + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t idesc =
                    (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);  // f16 x f16 -> f32
                const int b = local & 1;
                if (!mbar_wait(&tempty[b], ((uint32_t)(local >> 1) & 1u) ^ 1u, g.err, 601)) break;
                tc::fence_after();
                const uint32_t d = tmem + (uint32_t)b * SET_COLS + (uint32_t)q * BN;
                for (int kt = 0; kt < KT; kt++, rp.next(), ap.next()) {
                    // The converters arrive on aready only after their wait on the
                    // TMA barrier of this stage, so aready also orders the
                    // activation tile's arrival before these MMAs.
                    if (!mbar_wait(&aready[ap.slot], ap.phase, g.err, 603)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    // K = 16 per MMA: 32 bytes along the swizzled rows
                    const uint64_t da = da0 + (uint64_t)((ap.slot * A_STAGE) >> 4) + 2 * kk0;
                    const uint64_t db = db0 + (uint64_t)((rp.slot * R_STAGE) >> 4) + 2 * kk0;
                    tc::mma_bf16(d, da, db, idesc, kt > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < NK; kk++) tc::mma_bf16(d, da + 2 * kk, db + 2 * kk, idesc, 1u);
                    tc::commit(&rfree[rp.slot]);
                }
                if (ok) tc::commit(&tfull[b]);
            }
        }
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
        // ---------------- converters: packed e2m1 -> scaled f16, swizzled ----------------
        const int ct = threadIdx.x - kConvWarp0 * 32;   // 0..255
        const int row = ct >> 1, half = ct & 1;       // weight row of the tile, 32-column group of the k-tile
        const int G = g.K / kGroup;
        RingPos<NSR> rp;          // TMA stage of this k-tile
        RingPos<NSR> rq;          // TMA stage of the k-tile kAStages back (its MMAs free the slot)
        RingPos<kAStages> ap;
        int done = 0;             // k-tiles converted so far
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            const int tile = item / g.MT, mt = item - tile * g.MT;
            const size_t grow = (size_t)g.tiles[tile].x * g.R + mt * BM + row;
            const int smax0 = g.ma[grow];
            const int smax1 = DUAL ? g.mb[grow] : 0;
            const uint8_t *sc0 = g.sa + grow * (size_t)G + half;
            const uint8_t *sc1 = DUAL ? g.sb + grow * (size_t)G + half : nullptr;
            int s0 = sc0[0], s1 = DUAL ? sc1[0] : 0;
            for (int kt = 0; kt < KT; kt++, rp.next(), ap.next(), done++) {
                // next k-tile's scale bytes load while this one converts
                const int nx = kt + 1 < KT ? 2 * (kt + 1) : 2 * kt;
                const int s0n = sc0[nx];
                const int s1n = DUAL ? sc1[nx] : 0;
                if (!mbar_wait(&full[rp.slot], rp.phase, g.err, 604)) {
                    ok = false;
                    break;
                }
                if (done >= kAStages) {
                    if (!mbar_wait(&rfree[rq.slot], rq.phase, g.err, 607)) {
                        ok = false;
                        break;
                    }
                    rq.next();
                }
                const unsigned char *rawp = rring + rp.slot * R_STAGE + B_BYTES;
                unsigned char *ast = aring + ap.slot * A_STAGE;
#pragma unroll
                for (int m = 0; m < NM; m++) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(rawp + m * RAW_BYTES + row * kRawRow + half * 16);
                    const uint32_t f = f16x2_pow2((m == 0 ? s0 : s1) - (m == 0 ? smax0 : smax1));
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                    unsigned char *arow = ast + m * A_BYTES + row * 128;
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        // packed word j = columns 8j..8j+7 of the group = 16-byte chunk 4*half + j
                        uint32_t h0, h1, h2, h3;
                        e2m1x8_to_f16x2x4(words[j], h0, h1, h2, h3);
                        uint4 o;
                        o.x = hmul2(h0, f);
                        o.y = hmul2(h1, f);
                        o.z = hmul2(h2, f);
                        o.w = hmul2(h3, f);
                        const int c = 4 * half + j;
                        *reinterpret_cast<uint4 *>(arow + ((c ^ (row & 7)) << 4)) = o;
                    }
                }
                // make the generic-proxy stores visible to the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&aready[ap.slot]);
                s0 = s0n;
                s1 = s1n;
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;                 // TMEM lanes 32q..32q+31
        const int erow = q * 32 + lane;         // weight row of the tile
        int local = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, local++) {
            const int tile = item / g.MT, mt = item - tile * g.MT;
            const int2 td = g.tiles[tile];
            const int cnt = g.offsets[td.x + 1] - g.offsets[td.x];
            const int n_valid = min(BN, cnt - td.y * BN);
            const int pair0 = g.offsets[td.x] + td.y * BN;
            const int row_in_e = mt * BM + erow;
            const size_t grow = (size_t)td.x * g.R + row_in_e;
            const float rs0 = pow2_e8m0(g.ma[grow]);
            const float rs1 = DUAL ? pow2_e8m0(g.mb[grow]) : 0.f;
            const int b = local & 1;
            if (!mbar_wait(&tfull[b], (uint32_t)(local >> 1) & 1u, g.err, 606)) break;
            tc::fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * SET_COLS;
            for (int c0 = 0; c0 < n_valid; c0 += 16) {
                // per-pair factors for columns c0..c0+15, one lane each, then broadcast
                const int pl = pair0 + c0 + (lane & 15);
                const bool lv = c0 + (lane & 15) < n_valid;
                float pf = 0.f;      // W1/W3: 2^(token exponent); W2: routing weight
                int pt = 0;          // W2: token
                if (lv) {
                    if (DUAL) {
                        const int ex = *reinterpret_cast<const int *>(g.zp + (size_t)pl * (g.L + kZPad) + g.L);
                        pf = __uint_as_float((uint32_t)(127 + ex) << 23);
                    } else {
                        pf = g.pair_w[pl];
                        pt = g.perm[pl] / g.k;
                    }
                }
                float v0[16], v1[16];
                tc::tmem_ld16(tb + (uint32_t)c0, v0);
                tc::tmem_ld16(tb + (uint32_t)(BN + c0), v1);
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const float fj = __shfl_sync(0xffffffffu, pf, j);
                    const int tj = DUAL ? 0 : __shfl_sync(0xffffffffu, pt, j);
                    if (c0 + j < n_valid) {
                        const int p = pair0 + c0 + j;
                        if (DUAL)
                            g.h16[(size_t)p * g.I + row_in_e] =
                                __float2half_rn(situ_f(v0[j] * rs0 * fj, v1[j] * rs1 * fj, g.b1, g.b2));
                        else
                            atomicAdd(&g.acc[(size_t)tj * g.L + row_in_e], fj * ((v0[j] + v1[j]) * rs0));
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 2 * SET_COLS);
    }
}

// n-tiles: (expert, j) for j < ceil(count_e / 128), experts ascending. One block.
__global__ void __launch_bounds__(1024) k_expert_tiles(const int *counts, int E, int2 *tiles, int *n_tiles)
{
    __shared__ int wsum[32];
    pdl_launch_dependents();
    pdl_wait();
    const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nt = e < E ? (counts[e] + BN - 1) / BN : 0;
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
    if (threadIdx.x == 0) *n_tiles = total;
}

// zp[p] = z16[token of pair p] (L values and the exponent padding); one warp per pair.
__global__ void __launch_bounds__(256) k_gather_latent(const __half *z16, const int *perm, __half *zp,
                                                       int pairs, int k, int L)
{
    pdl_launch_dependents();
    pdl_wait();
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (p >= pairs) return;
    const int t = perm[p] / k;
    const int nv = (L + kZPad) / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(z16 + (size_t)t * (L + kZPad));
    uint4 *dst = reinterpret_cast<uint4 *>(zp + (size_t)p * (L + kZPad));
    for (int i = lane; i < nv; i += 32) dst[i] = src[i];
}

// Largest scale byte of every row of an expert matrix stack [rows, G]; load time.
__global__ void k_row_scale_max(const uint8_t *s, size_t rows, int G, uint8_t *out)
{
    const size_t r = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const uint8_t *p = s + r * (size_t)G;
    int m = 0;
    for (int i = 0; i < G; i++) m = max(m, (int)p[i]);
    out[r] = (uint8_t)m;
}

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
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
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
    return c.latent % BM == 0 && c.moe_inter % BM == 0 && (long long)c.max_tokens * c.topk >= BN;
}

size_t expert_gemm_max_tiles(const k3moe_config &c)
{
    return (size_t)((long long)c.max_tokens * c.topk / BN + c.n_experts + 1);
}

int expert_gemm_min_pairs() { return BN; }

cudaError_t init_expert_gemm()
{
    cudaError_t e = cudaFuncSetAttribute(k_expert_gemm<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes(true, ring_stages(true)));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_expert_gemm<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes(false, ring_stages(false)));
}

cudaError_t launch_expert_tiles(const k3moe &h, cudaStream_t s)
{
    return launch_pdl(k_expert_tiles, 1, 1024, 0, s, (const int *)h.ws.counts, h.cfg.n_experts,
                      h.ws.tiles, h.ws.n_tiles);
}

cudaError_t launch_gather_latent(const k3moe &h, int T, cudaStream_t s)
{
    const int pairs = T * h.cfg.topk;
    return launch_pdl(k_gather_latent, (pairs + 7) / 8, 256, 0, s, (const __half *)h.ws.z16,
                      (const int *)h.ws.perm, h.ws.zperm, pairs, h.cfg.topk, h.cfg.latent);
}

// W1/W3 (w13 = true: gathered latent -> h16) or W2 (h16 -> acc).
cudaError_t launch_expert_gemm(const k3moe &h, const LayerDev &w, int T, cudaStream_t s, bool w13)
{
    const k3moe_config &c = h.cfg;
    const int pairs = T * c.topk;
    if (pairs < BN) return cudaErrorInvalidValue;
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
    g.err = h.ws.err;
    g.K = w13 ? c.latent : c.moe_inter;
    g.R = w13 ? c.moe_inter : c.latent;
    g.MT = g.R / BM;
    CUtensorMap ra, rb, bx;
    bool ok;
    const uint64_t rows = (uint64_t)c.n_experts * g.R;
    if (w13) {
        g.sa = w.w1s;
        g.sb = w.w3s;
        g.ma = w.w1max;
        g.mb = w.w3max;
        ok = make_map_u8(&ra, w.w1p, rows, g.K / 2, kRawRow, BM) &&
             make_map_u8(&rb, w.w3p, rows, g.K / 2, kRawRow, BM) &&
             make_map_f16_sw128(&bx, h.ws.zperm, pairs, c.latent, c.latent + kZPad, kBoxRows);
    } else {
        g.sa = w.w2s;
        g.ma = w.w2max;
        ok = make_map_u8(&ra, w.w2p, rows, g.K / 2, kRawRow, BM) &&
             make_map_f16_sw128(&bx, h.ws.h16, pairs, c.moe_inter, c.moe_inter, kBoxRows);
        rb = ra;
    }
    if (!ok) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes(w13, ring_stages(w13));
    return w13 ? launch_pdl(k_expert_gemm<true>, h.sm_count, kThreads, smem, s, ra, rb, bx, g)
               : launch_pdl(k_expert_gemm<false>, h.sm_count, kThreads, smem, s, ra, rb, bx, g);
}

cudaError_t launch_row_scale_max(const uint8_t *s, size_t rows, int G, uint8_t *out)
{
    k_row_scale_max<<<(unsigned)((rows + 255) / 256), 256>>>(s, rows, G, out);
    return cudaGetLastError();
}

}  // namespace k3
