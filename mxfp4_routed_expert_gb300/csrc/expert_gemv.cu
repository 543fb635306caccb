// MXFP4 routed-expert GEMVs for decode (few tokens per expert).
//
// The expert weights are read exactly as stored: e2m1 nibbles two per byte
// (low nibble = even column, bit 3 = sign) with one ue8m0 scale per 32
// columns (kimi-k3-in-c README, Part II section 4 and k3_matmul_mxfp4;
// colibri docs/kimi_k3.md "Weights"). A 16-byte chunk of a row is 32 nibbles,
// i.e. exactly one scale group. Nibbles are widened in registers with
// cvt.rn.f16x2.e2m1x2 (exact), multiplied with fp16 activations by packed
// f16x2 FMAs over the 32 columns of a group, and every group partial is scaled
// by 2^(s-127) and accumulated in fp32.
//
// Both kernels are persistent and warp-specialised (one CTA per SM):
//   - one producer thread streams the weight rows through a ring of shared
//     memory stages with bulk TMA copies (cp.async.bulk + mbarrier); a stage
//     is 8 consecutive rows (of W1 and W3, or of W2) plus their scale bytes,
//     and the first stage of a work unit also carries the unit's activation
//     row;
//   - eight consumer warps each take one row of every stage; lane l owns the
//     column groups l, l+32, l+64, l+96 and keeps their activations in
//     registers for the whole unit; after the unit's 8 stages one
//     transpose-reduction across the warp gives each row's dot product.
// A work unit is (pair, 64 weight rows), where a pair is one (token, expert)
// assignment; units are ordered by (expert, row block, pair) so a second
// token of the same expert re-reads rows the L2 has just seen.
//
// k_w13_tma: gate row of W1 and up row of W3 against the fp16 latent z of
//   the pair's token; SiTU-GLU in the epilogue; h written per pair
//   (README section 9, k3_moe step 3 and k3_situ_glu).
// k_w2_tma: h . W2 rows, times the pair's routing weight, scatter-added into
//   the token's fp32 latent accumulator.
#include "k3moe_internal.cuh"

namespace k3 {

constexpr int kCW = 8;                  // consumer warps
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kRowsPerWarp = 2;          // rows of one stage each consumer warp takes
constexpr int kStageRows = kCW * kRowsPerWarp;          // 16
constexpr int kUnitStages = 4;
constexpr int kUnitRows = kStageRows * kUnitStages;     // 64
constexpr int kUnitVals = kRowsPerWarp * kUnitStages;   // dot products per warp and unit
constexpr int kMaxQ = 4;                 // column groups per lane (K <= 4096)
constexpr int kW13Stages = 3;
constexpr int kW2Stages = 6;

struct StageMeta {
    int p;      // pair slot (perm order)
    int t;      // token
    int rb;     // row block
    float f;    // w13: 2^zexp[t] (undoes the fp16 scaling of z); w2: routing weight
};

struct ExpTArgs {
    const uint8_t *pa, *sa, *pb, *sb;   // W1/W3 (w13) or W2 (w2): packed rows, scale rows
    int K;          // input width (L for w13, I for w2)
    int R;          // rows per expert (I for w13, L for w2)
    int L, k, E, T;
    const int *offsets, *perm;
    const __half *z16;     // w13 input [T, L]
    const int *zexp;       // [T]
    __half *h16;           // w13 output / w2 input [T*k, I]
    const float *wts;      // [T, k]
    float *acc;            // [T, L]
    float b1, b2;
    long long units;       // T*k*(R/64)
    int *err;
};

__host__ __device__ constexpr int al128(int n) { return (n + 127) & ~127; }

// Byte offsets inside one stage.
struct StageLayout {
    int kb, g;            // bytes per packed row, scale bytes per row
    int off_b, off_sa, off_sb, off_x, bytes;
    __host__ __device__ StageLayout(int K, bool two)
    {
        kb = K / 2;
        g = K / kGroup;
        off_b = kStageRows * kb;                         // second matrix (w13 only)
        off_sa = two ? 2 * kStageRows * kb : kStageRows * kb;
        off_sb = off_sa + kStageRows * g;
        off_x = al128(off_sb + (two ? kStageRows * g : 0));
        bytes = al128(off_x + 2 * K);
    }
};

__device__ __forceinline__ int find_expert(const int *offsets, int E, long long u, int RB)
{
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)offsets[mid] * RB <= u) lo = mid; else hi = mid;
    }
    return lo;
}

// 32 nibbles (one 16-byte chunk) against 32 fp16 activations held as 16 f16x2;
// two partial accumulators for instruction-level parallelism.
__device__ __forceinline__ float chunk_dot(const uint4 w, const uint32_t (&x)[16])
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t h0 = 0u, h1 = 0u;
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint32_t a0, a1, a2, a3;
        e2m1x8_to_f16x2x4(ww[q], a0, a1, a2, a3);
        h0 = hfma2(a0, x[4 * q], h0);
        h1 = hfma2(a1, x[4 * q + 1], h1);
        h0 = hfma2(a2, x[4 * q + 2], h0);
        h1 = hfma2(a3, x[4 * q + 3], h1);
    }
    return f16x2_sum(h0) + f16x2_sum(h1);
}

// Warp sum of each of v[0..N) (N a power of two, 2..32). Each halving step
// exchanges half of the remaining values with the partner lane, so after
// log2(N) steps one value is left per lane; plain butterflies over the lower
// lane bits finish the sum. Lane l ends with the total of v[(l >> s) & (N-1)],
// s = 5 - log2(N): for N = 16 lane l holds v[l/2], for N = 8 it holds v[l/4].
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane)
{
#pragma unroll
    for (int step = 0; (N >> step) > 1; step++) {
        const int off = 16 >> step, n = N >> step;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; i++) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = 16 / N; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

template <bool W13>
__global__ void __launch_bounds__(kThreads, 1) k_expert_tma(ExpTArgs a)
{
    extern __shared__ __align__(128) unsigned char sm[];
    constexpr int NS = W13 ? kW13Stages : kW2Stages;
    const StageLayout lay(a.K, W13);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + NS * lay.bytes);
    uint64_t *empty = full + NS;
    StageMeta *meta = reinterpret_cast<StageMeta *>(empty + NS);
    int *offs = reinterpret_cast<int *>(meta + NS);   // expert offsets [E+1]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = a.R / kUnitRows;
    const int G = a.K / kGroup;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCW);
        }
        fence_mbar_init();
    }
    pdl_launch_dependents();
    pdl_wait();   // routing tables and activations come from the previous kernels
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) offs[i] = a.offsets[i];
    __syncthreads();

    // balanced contiguous unit range of this CTA
    const long long u0 = a.units * blockIdx.x / gridDim.x;
    const long long u1 = a.units * (blockIdx.x + 1) / gridDim.x;
    const size_t eb = (size_t)a.R * lay.kb, es = (size_t)a.R * lay.g;

    if (warp == kCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();
            const uint64_t pol_keep = l2_policy_evict_last();
            int slot = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (long long u = u0; u < u1 && ok; u++) {
                const int e = find_expert(offs, a.E, u, RB);
                const int off = offs[e], cnt = offs[e + 1] - off;
                const long long local = u - (long long)off * RB;
                if (cnt <= 0 || local < 0 || local >= (long long)cnt * RB ||
                    off + cnt > a.T * a.k) {
                    set_err(a.err, kErrBounds, (int)u);
                    break;
                }
                const int rb = (int)(local / cnt), i = (int)(local % cnt);
                const int p = off + i;
                const int pf = a.perm[p];
                const int t = pf / a.k;
                if (t < 0 || t >= a.T) {
                    set_err(a.err, kErrBounds, (int)u);
                    break;
                }
                const float f = W13 ? __uint_as_float((uint32_t)(127 + a.zexp[t]) << 23) : a.wts[pf];
                const uint64_t pol = (cnt == 1) ? pol_stream : pol_keep;
                const uint8_t *PA = a.pa + (size_t)e * eb, *SA = a.sa + (size_t)e * es;
                const uint8_t *PB = W13 ? a.pb + (size_t)e * eb : nullptr;
                const uint8_t *SB = W13 ? a.sb + (size_t)e * es : nullptr;
                for (int s = 0; s < kUnitStages; s++) {
                    if (!mbar_wait(&empty[slot], phase ^ 1u, a.err, 100 + slot)) {
                        ok = false;
                        break;
                    }
                    meta[slot] = StageMeta{p, t, rb, f};
                    unsigned char *st = sm + slot * lay.bytes;
                    const int row0 = rb * kUnitRows + s * kStageRows;
                    uint32_t bytes = (uint32_t)(kStageRows * (lay.kb + lay.g)) * (W13 ? 2u : 1u);
                    if (s == 0) bytes += 2u * a.K;
                    mbar_expect_tx(&full[slot], bytes);
                    bulk_g2s(st, PA + (size_t)row0 * lay.kb, kStageRows * lay.kb, &full[slot], pol);
                    bulk_g2s(st + lay.off_sa, SA + (size_t)row0 * lay.g, kStageRows * lay.g,
                             &full[slot], pol);
                    if (W13) {
                        bulk_g2s(st + lay.off_b, PB + (size_t)row0 * lay.kb, kStageRows * lay.kb,
                                 &full[slot], pol);
                        bulk_g2s(st + lay.off_sb, SB + (size_t)row0 * lay.g, kStageRows * lay.g,
                                 &full[slot], pol);
                    }
                    if (s == 0) {
                        const __half *xsrc = W13 ? a.z16 + (size_t)t * a.K : a.h16 + (size_t)p * a.K;
                        bulk_g2s(st + lay.off_x, xsrc, 2u * a.K, &full[slot], pol_keep);
                    }
                    issued++;
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            // drain: no bulk copy may still target shared memory when the CTA exits
            const int n = issued < NS ? issued : NS;
            for (int j = issued - n; j < issued; j++)
                mbar_wait(&full[j % NS], (uint32_t)(j / NS) & 1u, a.err, 200);
        }
        return;
    }

    // ---------------- consumers ----------------
    int slot = 0;
    uint32_t phase = 0;
    uint32_t xr[kMaxQ][16];
    for (long long u = u0; u < u1; u++) {
        float va[kUnitVals], vb[kUnitVals];
        int p = 0, t = 0, rb = 0;
        float f = 0.f;
        bool ok = true;
#pragma unroll
        for (int s = 0; s < kUnitStages; s++) {
            if (!mbar_wait(&full[slot], phase, a.err, 300 + slot)) {
                ok = false;
                break;
            }
            const unsigned char *st = sm + slot * lay.bytes;
            if (s == 0) {
                const StageMeta m = meta[slot];
                p = m.p;
                t = m.t;
                rb = m.rb;
                f = m.f;
#pragma unroll
                for (int q = 0; q < kMaxQ; q++) {
                    const int g = lane + 32 * q;
                    if (g < G) {
                        const uint4 *xp = reinterpret_cast<const uint4 *>(st + lay.off_x + g * 64);
#pragma unroll
                        for (int c = 0; c < 4; c++) {
                            const uint4 v = xp[c];
                            xr[q][4 * c] = v.x;
                            xr[q][4 * c + 1] = v.y;
                            xr[q][4 * c + 2] = v.z;
                            xr[q][4 * c + 3] = v.w;
                        }
                    }
                }
            }
#pragma unroll
            for (int hr = 0; hr < kRowsPerWarp; hr++) {
                const int r = warp + kCW * hr;   // row inside the stage
                const unsigned char *ra = st + r * lay.kb;
                const unsigned char *ca = st + lay.off_sa + r * lay.g;
                const unsigned char *rbp = st + lay.off_b + r * lay.kb;
                const unsigned char *cbp = st + lay.off_sb + r * lay.g;
                float aa = 0.f, ab = 0.f;
#pragma unroll
                for (int q = 0; q < kMaxQ; q++) {
                    const int g = lane + 32 * q;
                    if (g < G) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(ra + g * 16);
                        aa += chunk_dot(w, xr[q]) * e8m0_to_f32(ca[g]);
                        if (W13) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(rbp + g * 16);
                            ab += chunk_dot(v, xr[q]) * e8m0_to_f32(cbp[g]);
                        }
                    }
                }
                va[kRowsPerWarp * s + hr] = aa;
                vb[kRowsPerWarp * s + hr] = ab;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == NS) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (!ok) return;
        // value i = 2*s + hr belongs to row rb*64 + s*16 + hr*8 + warp
        if (W13) {
            float v[2 * kUnitVals];
#pragma unroll
            for (int i = 0; i < kUnitVals; i++) {
                v[i] = va[i];
                v[kUnitVals + i] = vb[i];
            }
            // lane l ends with v[l >> 1]: the gate of value l/2 for l < 16, its up at l + 16
            const float r = transpose_reduce<2 * kUnitVals>(v, lane);
            const float up = __shfl_down_sync(0xffffffffu, r, 16);
            if (lane < 16 && (lane & 1) == 0) {
                const int i = lane >> 1;
                const int row = rb * kUnitRows + (i >> 1) * kStageRows + (i & 1) * kCW + warp;
                a.h16[(size_t)p * a.R + row] = __float2half_rn(situ_f(r * f, up * f, a.b1, a.b2));
            }
        } else {
            // lane l ends with va[l >> 2]
            const float r = transpose_reduce<kUnitVals>(va, lane);
            if ((lane & 3) == 0) {
                const int i = lane >> 2;
                const int row = rb * kUnitRows + (i >> 1) * kStageRows + (i & 1) * kCW + warp;
                atomicAdd(&a.acc[(size_t)t * a.L + row], f * r);
            }
        }
    }
}

static size_t exp_smem(int K, bool w13, int E)
{
    const StageLayout lay(K, w13);
    const int NS = w13 ? kW13Stages : kW2Stages;
    return (size_t)NS * lay.bytes + 2 * NS * sizeof(uint64_t) + NS * sizeof(StageMeta) +
           (size_t)(E + 1) * sizeof(int);
}

cudaError_t init_expert_kernels(const k3moe_config &c)
{
    cudaError_t e = cudaFuncSetAttribute(k_expert_tma<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)exp_smem(c.latent, true, c.n_experts));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_expert_tma<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)exp_smem(c.moe_inter, false, c.n_experts));
}

bool expert_smem_fits(const k3moe_config &c)
{
    return exp_smem(c.latent, true, c.n_experts) <= 227 * 1024 &&
           exp_smem(c.moe_inter, false, c.n_experts) <= 227 * 1024;
}

static ExpTArgs base_args(const k3moe &h, int T)
{
    const k3moe_config &c = h.cfg;
    ExpTArgs a;
    a.L = c.latent;
    a.k = c.topk;
    a.E = c.n_experts;
    a.T = T;
    a.offsets = h.ws.offsets;
    a.perm = h.ws.perm;
    a.z16 = h.ws.z16;
    a.zexp = h.ws.zexp;
    a.h16 = h.ws.h16;
    a.wts = h.ws.wts;
    a.acc = h.ws.acc;
    a.b1 = c.situ_b1;
    a.b2 = c.situ_b2;
    a.err = h.ws.err;
    return a;
}

cudaError_t launch_expert_w13(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    ExpTArgs a = base_args(h, T);
    a.pa = w.w1p;
    a.sa = w.w1s;
    a.pb = w.w3p;
    a.sb = w.w3s;
    a.K = h.cfg.latent;
    a.R = h.cfg.moe_inter;
    a.units = (long long)T * h.cfg.topk * (a.R / kUnitRows);
    const int grid = (int)(a.units < h.sm_count ? a.units : h.sm_count);
    return launch_pdl(k_expert_tma<true>, grid, kThreads, exp_smem(a.K, true, a.E), s, a);
}

cudaError_t launch_expert_w2(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    ExpTArgs a = base_args(h, T);
    a.pa = w.w2p;
    a.sa = w.w2s;
    a.pb = nullptr;
    a.sb = nullptr;
    a.K = h.cfg.moe_inter;
    a.R = h.cfg.latent;
    a.units = (long long)T * h.cfg.topk * (a.R / kUnitRows);
    const int grid = (int)(a.units < h.sm_count ? a.units : h.sm_count);
    return launch_pdl(k_expert_tma<false>, grid, kThreads, exp_smem(a.K, false, a.E), s, a);
}

}  // namespace k3
