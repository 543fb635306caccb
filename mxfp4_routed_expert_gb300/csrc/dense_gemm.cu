// Dense projections of the layer as tcgen05 tensor-core GEMMs (prefill and
// batched decode, T >= 16).
//
// The steps (kimi-k3-in-c README, Part II section 9, k3_moe steps 1, 2, 5, 6):
//   RD: router logits x . Wr (E rows) and latent down projection x . Wd (L rows);
//   SH: the fused shared experts' gate/up pair with SiTU-GLU in the epilogue;
//   UP: y = Wu . n + Ws2 . s over the concatenated K = L + S.
//
// Orientation: the weight rows are the MMA's M (A operand, 128-row tiles) and
// the tokens its N (B operand, 16..256 per tile), so small token counts waste
// no tensor work on padding rows. A and B are K-major bf16 tiles of 64 columns
// (128 bytes, 128-byte swizzle) loaded by TMA into a ring of shared-memory
// stages; one warp issues tcgen05.mma (kind::f16, fp32 accumulators in
// TMEM) and commits each stage back to the producer; after the last k-tile all
// eight warps read the accumulators with tcgen05.ld (two warps per TMEM lane
// quadrant, alternate 16-column groups) and run the epilogue. When
// the (M, N) tile grid is too small to occupy the GPU, K is split across CTAs
// whose fp32 partials meet in global memory by atomic addition; the last CTA
// of a tile (counted in global memory) applies the epilogue.
#include <algorithm>

#include "k3moe_internal.cuh"
#include "tc_common.cuh"

namespace k3 {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int kThreads = 256;   // warps 0 and 1 also produce and issue; all eight run the epilogue
constexpr int kSmemBudget = 227 * 1024;

enum Mode : int { RD = 0, SH = 1, UP = 2 };

struct GemmArgs {
    int mode;
    int T;           // tokens (N extent)
    int BN;          // N tile (multiple of 16, <= 256)
    int KT;          // k-tiles in total
    int KTA;         // UP: k-tiles taken from map a0 (the rest from a1); RD: m-tiles of map a0
    int splits;      // split-K factor
    int ns;          // pipeline stages
    int E, L, S, H;
    float *logits, *z;          // RD outputs (fp32 [T,E], [T,L])
    float *cat;                 // SH: fp32 copy of the shared SiTU at cat[:, L:] (pitch L+S)
    __nv_bfloat16 *act;         // SH: bf16 shared SiTU at act[:, L:] (pitch L+S)
    __nv_bfloat16 *y;           // UP output [T, H]
    float b1, b2, ib1, ib2;     // SiTU bounds and their reciprocals
    float *part;                // split-K partials [T, 2*R] fp32 (zeroed), R = rows of the mode
    int *tile_count;            // split-K arrival counters per (m-tile, n-tile), left at 0
    int *err;
};

// One output run of an m-tile: for token n, nrows consecutive elements of
// esz bytes at base + (n * pitch + r0) * esz (vec: every run starts on 16 bytes).
struct OutRun {
    unsigned char *base;
    int pitch, r0, nrows, esz;
    bool vec;
};

__device__ __forceinline__ OutRun out_run(unsigned char *base, int pitch, int r0, int rows, int esz)
{
    OutRun o;
    o.base = base;
    o.pitch = pitch;
    o.r0 = r0;
    o.nrows = rows - r0 < BM ? rows - r0 : BM;
    o.esz = esz;
    o.vec = ((reinterpret_cast<uintptr_t>(base) + (uintptr_t)r0 * esz) % 16 == 0) &&
            ((size_t)pitch * esz) % 16 == 0;
    return o;
}

// The output runs of slab k of this CTA's tile: the m-tile mt + k (router+down
// and up+shared-down), or for the shared gate/up the fp32 and bf16 copies of
// the SiTU of its one m-tile.
__device__ __forceinline__ OutRun tile_run(const GemmArgs &g, int mt, int k)
{
    if (g.mode == SH) {
        return k == 0 ? out_run(reinterpret_cast<unsigned char *>(g.cat + g.L), g.L + g.S, mt * BM, g.S, 4)
                      : out_run(reinterpret_cast<unsigned char *>(g.act + g.L), g.L + g.S, mt * BM, g.S, 2);
    }
    const int m = mt + k;
    if (g.mode == RD) {
        return m < g.KTA ? out_run(reinterpret_cast<unsigned char *>(g.logits), g.E, m * BM, g.E, 4)
                         : out_run(reinterpret_cast<unsigned char *>(g.z), g.L, (m - g.KTA) * BM, g.L, 4);
    }
    return out_run(reinterpret_cast<unsigned char *>(g.y), g.H, m * BM, g.H, 2);
}

// Epilogue of an unsplit tile, staged through shared memory (the operand ring
// is idle once the MMAs are done): each round, the eight warps write
// kStageTokens tokens' values of their rows (TMEM lane = row) into slabs laid out
// [token][128 rows], then all threads copy every token's row run to global
// memory in 16-byte pieces. Element-wise stores (one 2- or 4-byte element per
// lane, 32 rows of one token per warp instruction) ran the epilogue at about
// 45 us per 256-token tile; staged, a warp instruction writes whole runs.
constexpr int kStageTokens = 32;
constexpr int kSlabBytes = kStageTokens * BM * 4;
constexpr int kStageBytes = 2 * kSlabBytes;

template <bool MPAIR>
__device__ __forceinline__ void epilogue_staged(const GemmArgs &g, unsigned char *stage, uint32_t tbase,
                                                bool dual, int mt, int n0, int rit, int half)
{
    const int nslab = (g.mode == SH || MPAIR) ? 2 : 1;
    OutRun run[2];
    run[0] = tile_run(g, mt, 0);
    run[1] = tile_run(g, mt, nslab > 1 ? 1 : 0);
    float *f0 = reinterpret_cast<float *>(stage);
    float *f1 = reinterpret_cast<float *>(stage + kSlabBytes);
    __nv_bfloat16 *b0 = reinterpret_cast<__nv_bfloat16 *>(stage);
    __nv_bfloat16 *b1 = reinterpret_cast<__nv_bfloat16 *>(stage + kSlabBytes);
    for (int c0 = 0; c0 < g.BN; c0 += kStageTokens) {
        const int cw = g.BN - c0 < kStageTokens ? g.BN - c0 : kStageTokens;   // a multiple of 16
        for (int c = 16 * half; c < cw; c += 32) {
            float v0[16], v1[16];
            tc::tmem_ld16(tbase + (uint32_t)(c0 + c), v0);
            if (dual) tc::tmem_ld16(tbase + (uint32_t)(g.BN + c0 + c), v1);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int at = (c + j) * BM + rit;
                if (g.mode == SH) {
                    const float sv = situ_exp(v0[j], v1[j], g.b1, g.b2, g.ib1, g.ib2);
                    f0[at] = sv;
                    b1[at] = __float2bfloat16_rn(sv);
                } else if (g.mode == RD) {
                    f0[at] = v0[j];
                    if (MPAIR) f1[at] = v1[j];
                } else {
                    b0[at] = __float2bfloat16_rn(v0[j]);
                    if (MPAIR) b1[at] = __float2bfloat16_rn(v1[j]);
                }
            }
        }
        __syncthreads();
        for (int k = 0; k < nslab; k++) {
            const OutRun o = run[k];
            if (o.nrows <= 0) continue;   // a second m-tile past the matrix
            const int epp = 16 / o.esz;   // elements per 16-byte piece
            const int ppr = BM / epp;     // pieces per token
            const unsigned char *slab = stage + k * kSlabBytes;
            for (int i = threadIdx.x; i < cw * ppr; i += kThreads) {
                const int tk = i / ppr, e0 = (i - tk * ppr) * epp;
                const int n = n0 + c0 + tk;
                if (n >= g.T || e0 >= o.nrows) continue;
                unsigned char *dst = o.base + ((size_t)n * o.pitch + o.r0 + e0) * o.esz;
                const unsigned char *src = slab + (size_t)(tk * BM + e0) * o.esz;
                if (o.vec && e0 + epp <= o.nrows) {
                    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
                } else if (o.esz == 4) {
                    for (int e = 0; e < epp && e0 + e < o.nrows; e++)
                        reinterpret_cast<uint32_t *>(dst)[e] = reinterpret_cast<const uint32_t *>(src)[e];
                } else {
                    for (int e = 0; e < epp && e0 + e < o.nrows; e++)
                        reinterpret_cast<uint16_t *>(dst)[e] = reinterpret_cast<const uint16_t *>(src)[e];
                }
            }
        }
        __syncthreads();
    }
}

__device__ __forceinline__ void epilogue_store(const GemmArgs &g, int row, int n, float v0, float v1)
{
    if (g.mode == RD) {
        if (row < g.E) g.logits[(size_t)n * g.E + row] = v0;
        else g.z[(size_t)n * g.L + (row - g.E)] = v0;
    } else if (g.mode == SH) {
        const float s = situ_exp(v0, v1, g.b1, g.b2, g.ib1, g.ib2);
        g.cat[(size_t)n * (g.L + g.S) + g.L + row] = s;
        g.act[(size_t)n * (g.L + g.S) + g.L + row] = __float2bfloat16_rn(s);
    } else {
        g.y[(size_t)n * g.H + row] = __float2bfloat16_rn(v0);
    }
}

// MPAIR: RD/UP with two m-tiles per CTA (its own instantiation, so that the
// one-tile kernel compiles as if the pairing did not exist). WIDE: the
// producer and the MMA issuer are whole warps (below 512 tokens), else lone
// threads (see the roles below).
template <bool MPAIR, bool WIDE>
__global__ void __launch_bounds__(kThreads, 1)
    k_dense_gemm(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                 const __grid_constant__ CUtensorMap b, GemmArgs g)
{
    extern __shared__ unsigned char raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // two accumulators: gate and up (SH), or two m-tiles (RD/UP with mpair)
    const bool dual = g.mode == SH || MPAIR;
    const int a_bytes = BM * BK * 2, b_bytes = g.BN * BK * 2;
    const int stage_bytes = (dual ? 2 : 1) * a_bytes + b_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + g.ns * stage_bytes);
    uint64_t *empty = full + g.ns;
    uint64_t *done = empty + g.ns;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    __shared__ int last_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = blockIdx.x, mt = MPAIR ? 2 * (int)blockIdx.y : (int)blockIdx.y, ks = blockIdx.z;
    const uint32_t tcols = dual ? 2u * (uint32_t)g.BN : (uint32_t)g.BN;
    uint32_t alloc_cols = 32;
    while (alloc_cols < tcols) alloc_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < g.ns; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
        tc::prefetch_map(&a0);
        tc::prefetch_map(&a1);
        tc::prefetch_map(&b);
    }
    if (warp == 2) tc::tmem_alloc(tslot, alloc_cols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t tmem = *tslot;

    // k-tile range of this split
    const int kt0 = (int)((long long)g.KT * ks / g.splits);
    const int kt1 = (int)((long long)g.KT * (ks + 1) / g.splits);
    const int n0 = nt * g.BN;
    // RD: m-tiles [0, KTA) come from the router map, the rest from the down map
    const CUtensorMap *amap = &a0;
    int arow = mt * BM;
    if (g.mode == RD && mt >= g.KTA) {
        amap = &a1;
        arow = (mt - g.KTA) * BM;
    }
    // the second m-tile of an mpair CTA (rows past the matrix load as zeros
    // and are never stored)
    const CUtensorMap *amap2 = &a0;
    int arow2 = (mt + 1) * BM;
    if (g.mode == RD && mt + 1 >= g.KTA) {
        amap2 = &a1;
        arow2 = (mt + 1 - g.KTA) * BM;
    }

    // Roles. With few tokens per tile (WIDE) the producer and the MMA issuer
    // are whole warps: every lane runs the loop, so that the descriptors and
    // coordinates are warp-uniform, lane 0 polls the barrier and one elected
    // lane issues; a lone issuing thread spent about 250 cycles per
    // tcgen05.mma there whatever its N. With 256-token tiles the MMAs bound
    // the stage and lone threads measured faster (dense gate/up at 4096
    // tokens 2.27 against 2.46 ms).
    if (warp == 0 && (WIDE || lane == 0)) {
        // ---------------- TMA producer ----------------
        for (int kt = kt0; kt < kt1; kt++) {
            const int i = kt - kt0, s = i % g.ns;
            const uint32_t ph = (uint32_t)(i / g.ns) & 1u;
            if (WIDE ? !tc::lane0_wait(&empty[s], ph ^ 1u, g.err, 500) : !mbar_wait(&empty[s], ph ^ 1u, g.err, 500))
                break;
            if (!WIDE || tc::elect_one()) {
                unsigned char *st = sm + s * stage_bytes;
                mbar_expect_tx(&full[s], (uint32_t)stage_bytes);
                if (g.mode == UP) {
                    const bool first = kt < g.KTA;
                    const CUtensorMap *m = first ? &a0 : &a1;
                    const int kc = (first ? kt : kt - g.KTA) * BK;
                    tc::tma_load_2d(st, m, kc, arow, &full[s]);
                    if (MPAIR) tc::tma_load_2d(st + a_bytes, m, kc, arow + BM, &full[s]);
                } else {
                    tc::tma_load_2d(st, amap, kt * BK, arow, &full[s]);
                    if (MPAIR) tc::tma_load_2d(st + a_bytes, amap2, kt * BK, arow2, &full[s]);
                    else if (dual) tc::tma_load_2d(st + a_bytes, &a1, kt * BK, arow, &full[s]);
                }
                tc::tma_load_2d(st + (dual ? 2 : 1) * a_bytes, &b, kt * BK, n0, &full[s]);
            }
            if (WIDE) __syncwarp();
        }
    } else if (warp == 1 && (WIDE || lane == 0)) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = tc::idesc_bf16(BM, g.BN);
        for (int kt = kt0; kt < kt1; kt++) {
            const int i = kt - kt0, s = i % g.ns;
            const uint32_t ph = (uint32_t)(i / g.ns) & 1u;
            if (WIDE ? !tc::lane0_wait(&full[s], ph, g.err, 501) : !mbar_wait(&full[s], ph, g.err, 501)) break;
            tc::fence_after();
            const uint32_t sa = tc::su32(sm + s * stage_bytes);
            const uint32_t sb = sa + (dual ? 2 : 1) * a_bytes;
            if (!WIDE || tc::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    tc::mma_bf16(tmem, tc::desc_sw128(sa + kk * 32), tc::desc_sw128(sb + kk * 32), idesc, acc);
                    if (dual)
                        tc::mma_bf16(tmem + (uint32_t)g.BN, tc::desc_sw128(sa + a_bytes + kk * 32),
                                     tc::desc_sw128(sb + kk * 32), idesc, acc);
                }
                tc::commit(&empty[s]);
            }
            if (WIDE) __syncwarp();
        }
        if (!WIDE || tc::elect_one()) tc::commit(done);
    }
    __syncwarp();

    // ---------------- epilogue: all eight warps ----------------
    const bool have_acc = kt1 > kt0;
    if (have_acc) mbar_wait(done, 0, g.err, 502);
    tc::fence_after();
    // warp w reads TMEM lanes 32 (w % 4) .. + 31; the two halves of the CTA
    // take alternate 16-column groups
    const int quad = warp & 3, half = warp >> 2;
    const int row_in_tile = quad * 32 + lane;
    // rows of this tile in the mode's row numbering
    int row;
    bool row_ok;
    auto tile_row = [&](int m, int &r, bool &ok) {
        if (g.mode == RD) {
            r = m < g.KTA ? m * BM + row_in_tile : g.E + (m - g.KTA) * BM + row_in_tile;
            ok = m < g.KTA ? r < g.E : (r - g.E) < g.L;
        } else {
            r = m * BM + row_in_tile;
            ok = r < (g.mode == SH ? g.S : g.H);
        }
    };
    tile_row(mt, row, row_ok);
    const int R = g.mode == RD ? g.E + g.L : (g.mode == SH ? g.S : g.H);
    const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16);

    if (g.splits == 1) {
        // every MMA has completed (done), so the ring's shared memory is free
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epilogue_staged<MPAIR>(g, sm, tbase, dual, mt, n0, row_in_tile, half);
    } else {
        // partial sums meet in g.part; the last CTA of the tile finishes it
        if (have_acc) {
            for (int c = 16 * half; c < g.BN; c += 32) {
                float v0[16], v1[16];
                tc::tmem_ld16(tbase + (uint32_t)c, v0);
                if (dual) tc::tmem_ld16(tbase + (uint32_t)(g.BN + c), v1);
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int n = n0 + c + j;
                    if (row_ok && n < g.T) {
                        atomicAdd(&g.part[(size_t)n * 2 * R + row], v0[j]);
                        if (dual) atomicAdd(&g.part[(size_t)n * 2 * R + R + row], v1[j]);
                    }
                }
            }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            int *cnt = &g.tile_count[mt * gridDim.x + nt];
            const int prev = atomicAdd(cnt, 1);
            last_flag = prev == g.splits - 1;
            if (last_flag) *cnt = 0;   // leave the counter ready for the next launch
        }
        __syncthreads();
        if (last_flag) {
            __threadfence();
            // 16 columns at a time: all their loads in flight before any use,
            // so that the tile costs BN / 16 L2 round trips, not BN
            for (int c = 16 * half; c < g.BN; c += 32) {
                float v0[16], v1[16];
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int n = n0 + c + j;
                    v0[j] = 0.f;
                    v1[j] = 0.f;
                    if (row_ok && n < g.T) {
                        const float *pp = &g.part[(size_t)n * 2 * R];
                        v0[j] = __ldcg(&pp[row]);
                        if (dual) v1[j] = __ldcg(&pp[R + row]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int n = n0 + c + j;
                    if (row_ok && n < g.T) {
                        float *pp = &g.part[(size_t)n * 2 * R];
                        pp[row] = 0.f;          // leave the partials zeroed for the next launch
                        if (dual) pp[R + row] = 0.f;
                        epilogue_store(g, row, n, v0[j], v1[j]);
                    }
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, alloc_cols);
    }
}

// N tile: a multiple of 16 no larger than T, at most 256. When the tile grid
// spans several waves of the GPU, the width that minimises waves x (N + a
// per-tile overhead worth 32 columns) is taken, so that the last wave is not
// nearly empty (tiles past T read zero rows and store nothing).
int pick_bn(int T, int mtiles, int sms)
{
    int bn = (T / 16) * 16;
    if (bn > 256) bn = 256;
    if (T < 512) {
        // past the split-K range: narrower tiles while the grid would leave
        // half the SMs idle (the other n-tiles read the weights from L2)
        if (T > kSplitTokensMax)
            while (bn > 64 && (long long)mtiles * ((T + bn - 1) / bn) * 2 <= sms) bn = ((bn / 2 + 15) / 16) * 16;
        return bn;
    }
    long long best = -1;
    int pick = bn;
    for (int c = bn; c >= 128; c -= 16) {
        const long long tiles = (long long)mtiles * ((T + c - 1) / c);
        const long long cost = ((tiles + sms - 1) / sms) * (c + 32);
        if (best < 0 || cost < best) {
            best = cost;
            pick = c;
        }
    }
    return pick;
}

int stages_for(bool dual, int BN)
{
    const int stage = (dual ? 2 : 1) * BM * BK * 2 + BN * BK * 2;
    int ns = (kSmemBudget - 2048) / stage;
    return ns > 8 ? 8 : ns;
}

}  // namespace

cudaError_t init_dense_gemm()
{
    for (auto *k : {k_dense_gemm<true, false>, k_dense_gemm<false, false>, k_dense_gemm<false, true>}) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget - 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t dense_gemm_part_floats(const k3moe_config &c)
{
    const int R = std::max(std::max(c.n_experts + c.latent, c.shared_inter), c.hidden);
    return (size_t)kSplitTokensMax * 2 * (size_t)R;
}

size_t dense_gemm_tile_counters(const k3moe_config &c)
{
    const int R = std::max(std::max(c.n_experts + c.latent, c.shared_inter), c.hidden);
    return (size_t)((R + BM - 1) / BM + 8) * (size_t)((kSplitTokensMax + 15) / 16);
}

// part: 0 = router + down, 1 = shared gate/up, 2 = up + shared down (needs the
// normed latent in act[:, :L] and the shared SiTU in act[:, L:]).
cudaError_t launch_dense_gemm(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x,
                              __nv_bfloat16 *y, int T, cudaStream_t s, int part)
{
    const k3moe_config &c = h.cfg;
    GemmArgs g = {};
    g.mode = part;
    g.T = T;

    g.E = c.n_experts;
    g.L = c.latent;
    g.S = c.shared_inter;
    g.H = c.hidden;
    g.logits = h.ws.logits;
    g.z = h.ws.z;
    g.cat = h.ws.cat;
    g.act = h.ws.act;
    g.y = y;
    g.b1 = c.situ_b1;
    g.b2 = c.situ_b2;
    g.ib1 = 1.0f / c.situ_b1;
    g.ib2 = 1.0f / c.situ_b2;
    g.part = h.ws.gemm_part;
    g.tile_count = h.ws.gemm_tiles;
    g.err = h.ws.err;
    CUtensorMap a0, a1, b;
    int mtiles;
    bool ok = true;
    // From 512 tokens the single-matrix projections (router+down, up+shared
    // down) take two adjacent m-tiles per CTA, so that one activation tile
    // feeds 256 weight rows as the shared gate/up's does: the operand bytes
    // each SM takes in per MMA are what bounds these GEMMs at large T.
    const bool mpair = part != 1 && T >= 512;
    auto grid_m = [&](int mt) { return mpair ? (mt + 1) / 2 : mt; };
    if (part == 0) {
        const int mta = (c.n_experts + BM - 1) / BM;
        mtiles = mta + (c.latent + BM - 1) / BM;
        g.BN = pick_bn(T, grid_m(mtiles), h.sm_count);
        g.KTA = mta;
        g.KT = c.hidden / BK;
        ok = tc::make_map_bf16_sw128(&a0, w.router_w, c.n_experts, c.hidden, c.hidden, BM) &&
             tc::make_map_bf16_sw128(&a1, w.down_w, c.latent, c.hidden, c.hidden, BM) &&
             tc::make_map_bf16_sw128(&b, x, T, c.hidden, c.hidden, g.BN);
    } else if (part == 1) {
        mtiles = (c.shared_inter + BM - 1) / BM;
        g.BN = pick_bn(T, mtiles, h.sm_count);
        g.KT = c.hidden / BK;
        ok = tc::make_map_bf16_sw128(&a0, w.sh_w1, c.shared_inter, c.hidden, c.hidden, BM) &&
             tc::make_map_bf16_sw128(&a1, w.sh_w3, c.shared_inter, c.hidden, c.hidden, BM) &&
             tc::make_map_bf16_sw128(&b, x, T, c.hidden, c.hidden, g.BN);
    } else {
        mtiles = (c.hidden + BM - 1) / BM;
        g.BN = pick_bn(T, grid_m(mtiles), h.sm_count);
        g.KTA = c.latent / BK;
        g.KT = (c.latent + c.shared_inter) / BK;
        // a dense feed-forward layer has no latent columns: KTA = 0, a0 unused
        ok = (is_dense(c) || tc::make_map_bf16_sw128(&a0, w.up_w, c.hidden, c.latent, c.latent, BM)) &&
             tc::make_map_bf16_sw128(&a1, w.sh_w2, c.hidden, c.shared_inter, c.shared_inter, BM) &&
             tc::make_map_bf16_sw128(&b, h.ws.act, T, c.latent + c.shared_inter,
                                     c.latent + c.shared_inter, g.BN);
    }
    if (!ok) return cudaErrorInvalidValue;
    if (part == 2 && is_dense(c)) a0 = a1;
    const int ntiles = (T + g.BN - 1) / g.BN;
    int splits = 1;
    if (T <= kSplitTokensMax) {
        while (splits < 8 && mtiles * ntiles * splits * 2 <= h.sm_count && g.KT / (splits * 2) >= 4)
            splits *= 2;
    }
    g.splits = splits;
    const bool dual = part == 1 || mpair;
    g.ns = stages_for(dual, g.BN);
    const size_t ring = (size_t)g.ns * ((dual ? 2 : 1) * BM * BK * 2 + g.BN * BK * 2);
    if (ring < (size_t)kStageBytes) return cudaErrorInvalidValue;   // the epilogue stages in the ring
    const size_t smem = ring + 1024 + 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ntiles, (unsigned)grid_m(mtiles), (unsigned)splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the paired tiles run from 512 tokens, where the roles are lone threads
    if (mpair) return cudaLaunchKernelEx(&cfg, k_dense_gemm<true, false>, a0, a1, b, g);
    if (T >= 512) return cudaLaunchKernelEx(&cfg, k_dense_gemm<false, false>, a0, a1, b, g);
    return cudaLaunchKernelEx(&cfg, k_dense_gemm<false, true>, a0, a1, b, g);
}

// act[t, 0:L] = bf16(acc[t] / sqrt(mean(acc[t]^2) + eps) * gain): the latent
// norm of the aggregate for the tensor-core up projection.
__global__ void __launch_bounds__(256) k_norm_act(const float *acc, const __nv_bfloat16 *gain,
                                                  __nv_bfloat16 *act, int L, int ld, float eps)
{
    __shared__ float red[8];
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x;
    const float *a = acc + (size_t)t * L;
    float ss = 0.f;
    for (int i = threadIdx.x; i < L; i += blockDim.x) ss = fmaf(a[i], a[i], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) tot += red[i];
    const float inv = gain ? 1.0f / sqrtf(tot / (float)L + eps) : 1.f;
    for (int i = threadIdx.x; i < L; i += blockDim.x)
        act[(size_t)t * ld + i] = __float2bfloat16_rn(gain ? a[i] * inv * __bfloat162float(gain[i]) : a[i]);
}

cudaError_t launch_norm_act(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    const k3moe_config &c = h.cfg;
    return launch_pdl(k_norm_act, T, 256, 0, s, (const float *)h.ws.acc,
                      (const __nv_bfloat16 *)(c.latent_norm ? w.gain : nullptr), h.ws.act, c.latent,
                      c.latent + c.shared_inter, c.rms_eps);
}

}  // namespace k3
