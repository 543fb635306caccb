// bf16 weight-streaming GEMVs for one or two tokens (decode), TMA-fed.
//
// The three dense steps of the layer (kimi-k3-in-c README, Part II section 9,
// k3_moe steps 1, 2, 5 and 6; bf16 widening is a 16-bit shift, section 5):
//   RD: router logits x . Wr (E rows) and the latent down projection x . Wd
//       (L rows), both fp32 outputs;
//   SH: the fused shared experts' gate/up pair, SiTU-GLU applied per row pair;
//   UP: y = Wu . n + Ws2 . s with n = RMSNorm(acc) * gain (the norm of the
//       aggregate, section 9 step 4) and s the shared SiTU output, bf16 output.
//
// Persistent, one CTA per SM: a producer thread streams weight-row stages
// through a shared-memory ring with 3D tensor TMA copies: a matrix viewed as
// (64 columns, column blocks, rows) lands 16 rows x 1024 columns of a stage in
// one copy (4- and 1-row boxes take the rows of a partial group), since a
// thread issues a TMA copy only every ~150 cycles;
// sixteen consumer warps each own one row (RD, UP) or one gate/up row pair
// (SH) of a stage. The activations of the TB tokens sit in shared memory as
// bf16 for the whole kernel. The producer starts streaming weights before the
// programmatic-launch wait on the previous kernel (weights do not depend on
// it) while the consumers wait and then stage the activations. Router+down,
// a layer's first kernel, is launched in plain stream order; the shared
// gate/up, which reads only the layer input, waits only before it exits (so
// that its completion implies its predecessors'). A unit is one
// row (or pair) per consumer warp over the whole K; units are split evenly and
// contiguously over the CTAs.
#include <algorithm>
#include <cstring>

#include "decode_common.cuh"
#include "tc_common.cuh"

namespace k3 {

namespace {

constexpr int kCW = 16;                 // consumer warps
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kPieceBytes = 2048;       // bytes of one row piece (1024 bf16 columns)
constexpr int kPieceCols = kPieceBytes / 2;
constexpr int kMaxChunksPerLane = kPieceBytes / 16 / 32;   // 4
constexpr int kSmemBudget = 227 * 1024;

enum Mode : int { RD = 0, SH = 1, UP = 2 };

struct DenseTArgs {
    int mode, T, K;                     // K: input width (H for RD/SH, L+S for UP)
    const __nv_bfloat16 *x;            // RD/SH: [T, H]
    const float *acc;                  // UP: [T, L]
    const float *cat;                  // UP: shared part at cat[:, L:], pitch L+S
    const __nv_bfloat16 *gain;         // UP: [L] or null
    float eps;
    int L, S, E, H;
    const __nv_bfloat16 *wa, *wb;      // RD: router, down; SH: w1, w3; UP: up, shared w2
    float *out_a, *out_b;              // RD: logits [T,E], z [T,L]; SH: cat (+L), pitch L+S
    __nv_bfloat16 *y;                  // UP: [T, H]
    float b1, b2;
    int units;                         // rows (RD: E+L, UP: H) or gate/up row pairs (SH: S)
    int wait;                          // consumers wait for the previous kernel (0: they read only x)
    int ns;                            // pipeline stages
    // RD/SH from the residual: x = bf16(RMSNorm(hin) * pgain) made in the
    // kernel (x unused); the first CTA of RD also stores it to xout
    const float *hin;                  // [T, H] fp32
    const __nv_bfloat16 *pgain;        // [H]
    __nv_bfloat16 *xout;               // [T, H] or null
    int *err;
};

__device__ __forceinline__ int pieces_of(int cols) { return (cols + kPieceCols - 1) / kPieceCols; }

// Row tensor maps of one weight matrix (boxes of 16, 4 and 1 rows, 1024 columns).
struct RowMaps {
    CUtensorMap m16, m4, m1;
};
struct DenseMaps {
    RowMaps a, b;   // the mode's two matrices (RD: router, down; SH: w1, w3; UP: up, shared w2)
};
constexpr int kPieceBlocks = kPieceCols / 64;

// Rows [r, r + n) of a matrix, column blocks from y0, into consecutive
// kPieceBytes rows at dst: 16-row boxes, then 4-row, then single rows.
__device__ __forceinline__ void load_rows(const RowMaps &m, unsigned char *dst, int r, int n, int y0,
                                          uint64_t *bar, uint64_t pol)
{
    int i = 0;
    for (; n - i >= 16; i += 16) tc::tma_load_3d(dst + i * kPieceBytes, &m.m16, 0, y0, r + i, bar, pol);
    for (; n - i >= 4; i += 4) tc::tma_load_3d(dst + i * kPieceBytes, &m.m4, 0, y0, r + i, bar, pol);
    for (; i < n; i++) tc::tma_load_3d(dst + i * kPieceBytes, &m.m1, 0, y0, r + i, bar, pol);
}

// Piece p of a row: which matrix (0: wa, 1: wb), its first column inside that
// matrix, its width, and where its activations start in the staged vector.
// RD/SH rows are one matrix of H columns; UP rows are [Wu (L) | Ws2 (S)].
struct Piece {
    int mat, col0, ncol, xoff;
};

__device__ __forceinline__ Piece piece_info(const DenseTArgs &a, int p)
{
    Piece q;
    if (a.mode != UP) {
        q.mat = 0;
        q.col0 = p * kPieceCols;
        q.ncol = min(kPieceCols, a.H - q.col0);
        q.xoff = q.col0;
    } else {
        const int pl = pieces_of(a.L);
        q.mat = p < pl ? 0 : 1;
        q.col0 = (p < pl ? p : p - pl) * kPieceCols;
        q.ncol = min(kPieceCols, (p < pl ? a.L : a.S) - q.col0);
        q.xoff = (p < pl ? 0 : a.L) + q.col0;
    }
    return q;
}

__device__ __forceinline__ int npieces_of(const DenseTArgs &a)
{
    return a.mode != UP ? pieces_of(a.H) : pieces_of(a.L) + pieces_of(a.S);
}

template <int TB>
__global__ void __launch_bounds__(kThreads, 1) k_dense_tma(const __grid_constant__ DenseMaps mp, DenseTArgs a)
{
    extern __shared__ __align__(128) unsigned char sm[];
    const bool sh = a.mode == SH;
    // a stage holds one piece of every row of a group: 16 rows (RD, UP) or the
    // gate and up rows of 16 pairs (SH)
    const int rows_per_stage = sh ? 2 * kCW : kCW;
    const int stage_bytes = rows_per_stage * kPieceBytes;
    const int NS = a.ns;
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(sm + NS * stage_bytes);   // [TB][K]
    uint64_t *full = reinterpret_cast<uint64_t *>(xs + TB * a.K);
    uint64_t *empty = full + NS;
    __shared__ float red[TB][kCW];
    __shared__ double dred[TB][kCW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int npieces = npieces_of(a);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCW);
        }
        fence_mbar_init();
    }
    if (threadIdx.x == kCW * 32) {
        tc::prefetch_map(&mp.a.m16);
        tc::prefetch_map(&mp.b.m16);
    }
    __syncthreads();
    pdl_launch_dependents();
    // The producer reads weights only, which no earlier kernel writes: it
    // starts filling the ring at once, while the kernel this one depends on
    // drains. The consumers wait for it before they read activations.
    if (warp != kCW && a.wait) pdl_wait();

    // balanced contiguous range of rows (or pairs) of this CTA
    const int r0 = (int)((long long)a.units * blockIdx.x / gridDim.x);
    const int r1 = (int)((long long)a.units * (blockIdx.x + 1) / gridDim.x);

    if (warp == kCW) {
        // ---------------- producer thread: weight pieces only ----------------
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int slot = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int g0 = r0; g0 < r1 && ok; g0 += kCW) {
                const int ng = min(kCW, r1 - g0);
                for (int p = 0; p < npieces; p++) {
                    if (!mbar_wait(&empty[slot], phase ^ 1u, a.err, 400 + slot)) {
                        ok = false;
                        break;
                    }
                    const Piece q = piece_info(a, p);
                    unsigned char *st = sm + slot * stage_bytes;
                    // whole boxes land: a piece's columns past the matrix read as zeros
                    mbar_expect_tx(&full[slot], (uint32_t)((sh ? 2 : 1) * ng * kPieceBytes));
                    const int y0 = (q.col0 / kPieceCols) * kPieceBlocks;
                    if (a.mode == RD) {
                        const int nr = max(0, min(ng, a.E - g0));   // router rows, then down rows
                        if (nr > 0) load_rows(mp.a, st, g0, nr, y0, &full[slot], pol);
                        if (ng > nr) load_rows(mp.b, st + nr * kPieceBytes, g0 + nr - a.E, ng - nr, y0, &full[slot], pol);
                    } else if (sh) {
                        load_rows(mp.a, st, g0, ng, y0, &full[slot], pol);
                        load_rows(mp.b, st + kCW * kPieceBytes, g0, ng, y0, &full[slot], pol);
                    } else {
                        load_rows(q.mat == 0 ? mp.a : mp.b, st, g0, ng, y0, &full[slot], pol);
                    }
                    issued++;
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            const int n = issued < NS ? issued : NS;
            for (int j = issued - n; j < issued; j++)
                mbar_wait(&full[j % NS], (uint32_t)(j / NS) & 1u, a.err, 401);
        }
        return;
    }

    // ---------------- consumers: stage the activations as bf16 ----------------
    const int nct = kCW * 32;
    if (a.mode != UP && a.hin) {
        // RMSNorm in front of the MoE (k3_rmsnorm sums the squares in double and
        // forms inv = (float)(1 / sqrt(mean + eps)) in double; x = h * inv *
        // gain in float). Each thread sums its squares in fp32 and the partial
        // sums meet in double: this part's fp64 rate is too low for a double
        // per element.
#pragma unroll
        for (int t = 0; t < TB; t++) {
            const float sf = t < a.T ? residual_sumsq<8>(a.hin + (size_t)t * a.H, a.H / 4, threadIdx.x, nct) : 0.f;
            const double sd = warp_sum_d((double)sf);
            if (lane == 0) dred[t][warp] = sd;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nct));
        if (threadIdx.x == 0) {   // one thread: the double divide and root are slow here
#pragma unroll
            for (int t = 0; t < TB; t++) {
                double tot = 0.0;
#pragma unroll
                for (int w = 0; w < kCW; w++) tot += dred[t][w];
                red[t][0] = (float)(1.0 / sqrt(tot / (double)a.H + (double)a.eps));
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nct));
#pragma unroll
        for (int t = 0; t < TB; t++) {
            if (t < a.T) {
                const float inv = red[t][0];
                __nv_bfloat16 *o2 = (a.xout && blockIdx.x == 0) ? a.xout + (size_t)t * a.H : nullptr;
                residual_write<4>(a.hin + (size_t)t * a.H, a.pgain, inv, xs + t * a.K, o2, a.H / 4,
                                  threadIdx.x, nct);
            } else {
                for (int i = threadIdx.x; i < a.H / 8; i += nct)
                    reinterpret_cast<uint4 *>(xs + t * a.K)[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nct));
    } else if (a.mode != UP) {
        const int nv = TB * a.H / 8;
        for (int i = threadIdx.x; i < nv; i += nct) {
            const int t = (8 * i) / a.H;
            reinterpret_cast<uint4 *>(xs)[i] =
                t < a.T ? reinterpret_cast<const uint4 *>(a.x)[i] : make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nct));
    } else {
        // [RMSNorm(acc) * gain | shared SiTU], rounded to bf16
        float ss[TB];
#pragma unroll
        for (int t = 0; t < TB; t++) {
            ss[t] = 0.f;
            for (int i = threadIdx.x; i < a.L / 4; i += nct) {
                if (t < a.T) {
                    const float4 v = reinterpret_cast<const float4 *>(a.acc + (size_t)t * a.L)[i];
                    ss[t] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
            }
            ss[t] = warp_sum(ss[t]);
            if (lane == 0) red[t][warp] = ss[t];
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nct));
#pragma unroll
        for (int t = 0; t < TB; t++) {
            float inv = 1.f;
            if (a.gain) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < kCW; w++) tot += red[t][w];
                inv = 1.0f / sqrtf(tot / (float)a.L + a.eps);
            }
            for (int i = threadIdx.x; i < a.K / 2; i += nct) {
                float2 v = make_float2(0.f, 0.f);
                if (t < a.T) {
                    if (2 * i < a.L) {
                        v = reinterpret_cast<const float2 *>(a.acc + (size_t)t * a.L)[i];
                        if (a.gain) {
                            v.x *= inv * __bfloat162float(a.gain[2 * i]);
                            v.y *= inv * __bfloat162float(a.gain[2 * i + 1]);
                        }
                    } else {
                        v = reinterpret_cast<const float2 *>(a.cat + (size_t)t * a.K)[i];
                    }
                }
                reinterpret_cast<__nv_bfloat162 *>(xs + t * a.K)[i] = __floats2bfloat162_rn(v.x, v.y);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nct));
    }

    // ---------------- consumers: stream ----------------
    // warp w takes unit w of every group: row g0 + w (RD, UP) or the gate and
    // up rows of pair g0 + w (SH)
    int slot = 0;
    uint32_t phase = 0;
    for (int g0 = r0; g0 < r1; g0 += kCW) {
        const int ng = min(kCW, r1 - g0);
        const bool have = warp < ng;
        float a0[TB], a1[TB], b0[TB], b1[TB];
#pragma unroll
        for (int t = 0; t < TB; t++) a0[t] = a1[t] = b0[t] = b1[t] = 0.f;
        for (int p = 0; p < npieces; p++) {
            if (!mbar_wait(&full[slot], phase, a.err, 410 + slot)) return;
            if (have) {
                const unsigned char *st = sm + slot * stage_bytes;
                const Piece pc = piece_info(a, p);
                const int nch = pc.ncol / 8;
                const unsigned char *ra = st + warp * kPieceBytes;
                const unsigned char *rb = st + (kCW + warp) * kPieceBytes;
#pragma unroll
                for (int q = 0; q < kMaxChunksPerLane; q++) {
                    const int c = lane + 32 * q;
                    if (c < nch) {
                        const uint4 wa = *reinterpret_cast<const uint4 *>(ra + 16 * c);
                        uint4 wb = make_uint4(0u, 0u, 0u, 0u);
                        if (sh) wb = *reinterpret_cast<const uint4 *>(rb + 16 * c);
#pragma unroll
                        for (int t = 0; t < TB; t++) {
                            const uint4 xv = *reinterpret_cast<const uint4 *>(xs + t * a.K + pc.xoff + 8 * c);
                            dot8_bf16(wa, xv, a0[t], a1[t]);
                            if (sh) dot8_bf16(wb, xv, b0[t], b1[t]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == NS) {
                slot = 0;
                phase ^= 1u;
            }
        }
        float va[TB], vb[TB];
#pragma unroll
        for (int t = 0; t < TB; t++) {
            va[t] = warp_sum(a0[t] + a1[t]);
            vb[t] = sh ? warp_sum(b0[t] + b1[t]) : 0.f;
        }
        if (have && lane < TB && lane < a.T) {
            const int t = lane;
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int q = 0; q < TB; q++)
                if (q == t) {
                    v0 = va[q];
                    v1 = vb[q];
                }
            const int r = g0 + warp;
            if (a.mode == RD) {
                if (r < a.E) a.out_a[(size_t)t * a.E + r] = v0;
                else a.out_b[(size_t)t * a.L + (r - a.E)] = v0;
            } else if (sh) {
                a.out_a[(size_t)t * (a.L + a.S) + a.L + r] = situ_f(v0, v1, a.b1, a.b2);
            } else {
                a.y[(size_t)t * a.H + r] = __float2bfloat16_rn(v0);
            }
        }
    }
    // A kernel that skipped its dependency wait still waits before it exits:
    // the next kernel waits only for this one, and this one's completion must
    // imply that of every earlier kernel of the forward.
    if (!a.wait && threadIdx.x == 0) pdl_wait();
}

// Stages that fit beside the activations, at most 8.
int stages_for(int mode, int K, int TB)
{
    const int stage = (mode == SH ? 2 * kCW : kCW) * kPieceBytes;
    const int avail = kSmemBudget - TB * K * 2 - 2 * 8 * 8 - 1024;
    const int ns = avail / stage;
    return ns > 8 ? 8 : ns;
}

size_t dense_tma_smem(int mode, int K, int TB, int ns)
{
    return (size_t)ns * (mode == SH ? 2 * kCW : kCW) * kPieceBytes + (size_t)TB * K * 2 +
           2 * ns * sizeof(uint64_t);
}

}  // namespace

bool dense_tma_fits(const k3moe_config &c, int TB)
{
    return c.hidden % 64 == 0 && c.latent % 64 == 0 && c.shared_inter % 64 == 0 &&   // row maps
           stages_for(SH, c.hidden, TB) >= 2 && stages_for(RD, c.hidden, TB) >= 2 &&
           stages_for(UP, c.latent + c.shared_inter, TB) >= 2;
}

static bool make_row_maps(RowMaps *m, const void *base, int rows, int cols)
{
    return tc::make_map_bf16_rows(&m->m16, base, rows, cols, kPieceBlocks, 16) &&
           tc::make_map_bf16_rows(&m->m4, base, rows, cols, kPieceBlocks, 4) &&
           tc::make_map_bf16_rows(&m->m1, base, rows, cols, kPieceBlocks, 1);
}

static bool make_dense_maps(const k3moe_config &c, const LayerDev &w, int part, DenseMaps *mp)
{
    if (is_dense(c)) {   // feed-forward layer: gate/up, then the down matrix alone
        if (part == 1)
            return make_row_maps(&mp->a, w.sh_w1, c.shared_inter, c.hidden) &&
                   make_row_maps(&mp->b, w.sh_w3, c.shared_inter, c.hidden);
        if (part == 2 && make_row_maps(&mp->b, w.sh_w2, c.hidden, c.shared_inter)) {
            mp->a = mp->b;   // no latent columns: matrix a is never read
            return true;
        }
        return false;
    }
    if (part == 0)
        return make_row_maps(&mp->a, w.router_w, c.n_experts, c.hidden) &&
               make_row_maps(&mp->b, w.down_w, c.latent, c.hidden);
    if (part == 1)
        return make_row_maps(&mp->a, w.sh_w1, c.shared_inter, c.hidden) &&
               make_row_maps(&mp->b, w.sh_w3, c.shared_inter, c.hidden);
    return make_row_maps(&mp->a, w.up_w, c.hidden, c.latent) &&
           make_row_maps(&mp->b, w.sh_w2, c.hidden, c.shared_inter);
}

static_assert(sizeof(DenseMaps) == 6 * sizeof(CUtensorMap), "six maps per part");

// The maps of a loaded layer depend only on its weight pointers: built once.
bool build_dense_tma_maps(const k3moe_config &c, LayerDev &w)
{
    w.dense_maps_ok = false;
    for (int part = is_dense(c) ? 1 : 0; part < 3; part++) {
        DenseMaps mp;
        if (!make_dense_maps(c, w, part, &mp)) return false;
        memcpy(w.dense_maps[part], &mp, sizeof(mp));
    }
    w.dense_maps_ok = true;
    return true;
}

cudaError_t init_dense_tma(const k3moe_config &c)
{
    (void)c;
    // dynamic shared memory never exceeds the budget minus 1 KB (stages_for),
    // which leaves room for the kernel's static arrays
    cudaError_t e = cudaFuncSetAttribute(k_dense_tma<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget - 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_dense_tma<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBudget - 1024);
}

// part: 0 = router + down, 1 = shared gate/up, 2 = up (with the latent norm)
cudaError_t launch_dense_tma(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x,
                             __nv_bfloat16 *y, int T, cudaStream_t s, int part, const float *hin,
                             int t0, bool ordered, bool wait, bool spare_sm)
{
    const k3moe_config &c = h.cfg;
    DenseTArgs a = {};
    a.T = T;
    a.L = c.latent;
    a.S = c.shared_inter;
    a.E = c.n_experts;
    a.H = c.hidden;
    a.b1 = c.situ_b1;
    a.b2 = c.situ_b2;
    a.eps = c.rms_eps;
    a.err = h.ws.err;
    a.x = x;
    if (hin && part != 2) {
        a.hin = hin;
        a.pgain = w.post_gain;
        a.xout = part == 0 ? h.ws.xn : nullptr;
    }
    if (part == 0) {
        a.mode = RD;
        a.K = c.hidden;
        a.wa = w.router_w;
        a.wb = w.down_w;
        a.out_a = h.ws.logits;
        a.out_b = h.ws.z;
        a.units = c.n_experts + c.latent;
    } else if (part == 1) {
        a.mode = SH;
        a.K = c.hidden;
        a.wa = w.sh_w1;
        a.wb = w.sh_w3;
        a.out_a = h.ws.cat + (size_t)t0 * (c.latent + c.shared_inter);
        a.units = c.shared_inter;
    } else {
        a.mode = UP;
        a.K = c.latent + c.shared_inter;
        a.wa = w.up_w;
        a.wb = w.sh_w2;
        a.acc = h.ws.acc + (size_t)t0 * c.latent;
        a.cat = h.ws.cat + (size_t)t0 * (c.latent + c.shared_inter);
        a.gain = c.latent_norm ? w.gain : nullptr;
        a.y = y;
        a.units = c.hidden;
    }
    DenseMaps mp;
    if (w.dense_maps_ok) memcpy(&mp, w.dense_maps[part], sizeof(mp));
    else if (!make_dense_maps(c, w, part, &mp)) return cudaErrorInvalidValue;
    const int TB = T == 1 ? 1 : 2;
    a.ns = stages_for(a.mode, a.K, TB);
    const int groups = (a.units + kCW - 1) / kCW;
    const int sms = spare_sm && h.sm_count > 1 ? h.sm_count - 1 : h.sm_count;
    const int grid = groups < sms ? groups : sms;
    const size_t smem = dense_tma_smem(a.mode, a.K, TB, a.ns);
    // The shared gate/up reads only the layer input x and writes its own output
    // rows; the layer's first kernel (router+down, launched in stream order)
    // has already waited for everything the input depends on.
    a.wait = a.mode != SH || wait;
    if (a.mode == RD || ordered)
        return TB == 1 ? launch_ordered(k_dense_tma<1>, grid, kThreads, smem, s, mp, a)
                       : launch_ordered(k_dense_tma<2>, grid, kThreads, smem, s, mp, a);
    return TB == 1 ? launch_pdl(k_dense_tma<1>, grid, kThreads, smem, s, mp, a)
                   : launch_pdl(k_dense_tma<2>, grid, kThreads, smem, s, mp, a);
}

}  // namespace k3
