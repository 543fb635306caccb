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
//     is 16 consecutive rows (of W1 and W3, or of W2) plus their scale bytes,
//     and a stage that starts a new (token, expert) pair also carries that
//     pair's activation row;
//   - sixteen consumer warps each take one row of every stage; lane l owns the
//     column groups l, l+32, l+64, l+96 and keeps their activations in
//     registers for the unit; a warp reduction gives each row's dot product.
// A work unit is (pair, 16 or 64 weight rows), where a pair is one (token, expert)
// assignment; units are ordered by (expert, row block, pair) so a second
// token of the same expert re-reads rows the L2 has just seen.
//
// k_w13_tma: gate row of W1 and up row of W3 against the fp16 latent z of
//   the pair's token; SiTU-GLU in the epilogue (hardware tanh, as in the
//   grouped GEMM); h written per pair
//   (README section 9, k3_moe step 3 and k3_situ_glu).
// k_w2_tma: h . W2 rows, times the pair's routing weight, scatter-added into
//   the token's fp32 latent accumulator.
#include "decode_common.cuh"

namespace k3 {

constexpr int kCW = 16;                 // consumer warps
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kRowsPerWarp = 1;          // rows of one stage each consumer warp takes
constexpr int kStageRows = kCW * kRowsPerWarp;          // 16
// Stages per work unit: w13 units are one stage (fine-grained balance across
// CTAs); w2 stages are smaller, so its units span four stages to amortise the
// per-unit bookkeeping.
template <bool W13> struct UnitShape {
    static constexpr int stages = W13 ? 1 : 4;
    static constexpr int rows = kStageRows * stages;
    static constexpr int vals = kRowsPerWarp * stages;   // dot products per warp and unit
};
constexpr int kMaxQ = 4;                 // column groups per lane (K <= 4096)
constexpr int kW13Stages = 3;
constexpr int kW2Stages = 6;

struct StageMeta {
    int p;      // pair slot (perm order)
    int t;      // token
    int rb;     // row block
    float f;    // w2: routing weight of the pair (w13 reads its factor from the z row)
    int fresh;  // 1: the stage carries a new activation row (the pair changed)
};

struct ExpTArgs {
    const uint8_t *pa, *sa, *pb, *sb;   // W1/W3 (w13) or W2 (w2): packed rows, scale rows
    int K;          // input width (L for w13, I for w2)
    int R;          // rows per expert (I for w13, L for w2)
    int L, k, E, T;
    const int *offsets, *perm;
    const __half *z16;     // w13 input [T, L + kZPad] (exponent in the padding)
    __half *h16;           // w13 output / w2 input [T*k, I]
    const float *pair_w;   // [T*k] routing weight per pair slot
    float *acc;            // [T, L]
    float b1, b2, ib1, ib2;   // SiTU bounds and their reciprocals
    long long units;       // T*k*(R/64)
    const int *wslot;      // expert -> index in the weight arrays (nullptr: the expert itself)
    int n_ws;              // experts the weight arrays hold
    int *err;
};

__host__ __device__ constexpr int al128(int n) { return (n + 127) & ~127; }
__host__ __device__ constexpr int ilog2c(int n) { return n <= 1 ? 0 : 1 + ilog2c(n / 2); }

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
        bytes = al128(off_x + 2 * (K + kZPad));
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
    constexpr int kUnitStages = UnitShape<W13>::stages;
    constexpr int kUnitRows = UnitShape<W13>::rows;
    constexpr int kUnitVals = UnitShape<W13>::vals;
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

    // balanced contiguous unit range of this CTA, over the pairs this forward
    // kept (offsets[E]; every pair unless the routing dropped a weight tail)
    const long long kept = (long long)offs[a.E] * RB;
    const long long units = kept < a.units ? kept : a.units;
    const long long u0 = units * blockIdx.x / gridDim.x;
    const long long u1 = units * (blockIdx.x + 1) / gridDim.x;
    const size_t eb = (size_t)a.R * lay.kb, es = (size_t)a.R * lay.g;

    if (warp == kCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();
            const uint64_t pol_keep = l2_policy_evict_last();
            int slot = 0, issued = 0, prev_p = -1;
            uint32_t phase = 0;
            bool ok = true;
            // unit decode from the shared-memory offsets; the two global loads a
            // unit needs (token of the pair, its routing weight) are issued one
            // unit ahead so that their latency overlaps the current unit's copies
            struct U {
                int e, cnt, rb, p;
                bool bad;
            };
            auto decode = [&](long long u) {
                U d;
                d.e = find_expert(offs, a.E, u, RB);
                const int off = offs[d.e];
                d.cnt = offs[d.e + 1] - off;
                const long long local = u - (long long)off * RB;
                d.bad = d.cnt <= 0 || local < 0 || local >= (long long)d.cnt * RB ||
                        off + d.cnt > a.T * a.k;
                d.rb = d.bad ? 0 : (int)(local / d.cnt);
                d.p = d.bad ? 0 : off + (int)(local % d.cnt);
                return d;
            };
            U cur = decode(u0 < u1 ? u0 : 0);
            int pf_cur = u0 < u1 ? a.perm[cur.p] : 0;
            float w_cur = (!W13 && u0 < u1) ? a.pair_w[cur.p] : 0.f;
            for (long long u = u0; u < u1 && ok; u++) {
                U nxt = cur;
                int pf_nxt = 0;
                float w_nxt = 0.f;
                if (u + 1 < u1) {
                    nxt = decode(u + 1);
                    pf_nxt = a.perm[nxt.p];
                    if (!W13) w_nxt = a.pair_w[nxt.p];
                }
                const int e = cur.e, rb = cur.rb, p = cur.p, cnt = cur.cnt;
                const int t = pf_cur / a.k;
                if (cur.bad || t < 0 || t >= a.T) {
                    set_err(a.err, kErrBounds, (int)u);
                    break;
                }
                const int we = a.wslot ? a.wslot[e] : e;
                if (we < 0 || we >= a.n_ws) {
                    set_err(a.err, kErrBounds, (int)u);
                    break;
                }
                const float f = w_cur;
                const uint64_t pol = (cnt == 1) ? pol_stream : pol_keep;
                const uint8_t *PA = a.pa + (size_t)we * eb, *SA = a.sa + (size_t)we * es;
                const uint8_t *PB = W13 ? a.pb + (size_t)we * eb : nullptr;
                const uint8_t *SB = W13 ? a.sb + (size_t)we * es : nullptr;
                for (int s = 0; s < kUnitStages; s++) {
                    if (!mbar_wait(&empty[slot], phase ^ 1u, a.err, 100 + slot)) {
                        ok = false;
                        break;
                    }
                    const int fresh = (s == 0 && p != prev_p) ? 1 : 0;
                    if (s == 0) prev_p = p;
                    meta[slot] = StageMeta{p, t, rb, f, fresh};
                    unsigned char *st = sm + slot * lay.bytes;
                    const int row0 = rb * kUnitRows + s * kStageRows;
                    uint32_t bytes = (uint32_t)(kStageRows * (lay.kb + lay.g)) * (W13 ? 2u : 1u);
                    const uint32_t xbytes = W13 ? 2u * (a.K + kZPad) : 2u * a.K;
                    if (fresh) bytes += xbytes;
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
                    if (fresh) {
                        const __half *xsrc = W13 ? a.z16 + (size_t)t * (a.K + kZPad)
                                                 : a.h16 + (size_t)p * a.K;
                        bulk_g2s(st + lay.off_x, xsrc, xbytes, &full[slot], pol_keep);
                    }
                    issued++;
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                cur = nxt;
                pf_cur = pf_nxt;
                w_cur = w_nxt;
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
    float fz = 1.f;
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
                if (!W13) f = m.f;
                // the activation row is reloaded only when the pair changes; w13's
                // output factor 2^e (undoing z's fp16 scaling) rides in its padding
                if (W13 && m.fresh)
                    fz = __uint_as_float((uint32_t)(127 + *reinterpret_cast<const int *>(
                                                              st + lay.off_x + 2 * a.K))
                                         << 23);
                if (m.fresh)
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
        // value i (stage i / kRowsPerWarp, row hr = i % kRowsPerWarp of the warp)
        // belongs to row rb*64 + stage*16 + hr*kCW + warp
        if (W13) {
            constexpr int N = 2 * kUnitVals;
            constexpr int sft = 5 - ilog2c(N);
            float v[N];
#pragma unroll
            for (int i = 0; i < kUnitVals; i++) {
                v[i] = va[i];
                v[kUnitVals + i] = vb[i];
            }
            // lane l ends with v[l >> sft]: gate values first, their up values 16 lanes on
            const float r = transpose_reduce<N>(v, lane);
            const float up = __shfl_down_sync(0xffffffffu, r, 16);
            if (lane < 16 && (lane & ((1 << sft) - 1)) == 0) {
                const int i = lane >> sft;
                const int row = rb * kUnitRows + (i / kRowsPerWarp) * kStageRows +
                                (i % kRowsPerWarp) * kCW + warp;
                a.h16[(size_t)p * a.R + row] =
                    __float2half_rn(situ_hw(r * fz, up * fz, a.b1, a.b2, a.ib1, a.ib2));
            }
        } else {
            constexpr int N = kUnitVals;
            constexpr int sft = 5 - ilog2c(N);
            // lane l ends with va[l >> sft]
            const float r = transpose_reduce<N>(va, lane);
            if ((lane & ((1 << sft) - 1)) == 0) {
                const int i = lane >> sft;
                const int row = rb * kUnitRows + (i / kRowsPerWarp) * kStageRows +
                                (i % kRowsPerWarp) * kCW + warp;
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

static ExpTArgs base_args(const k3moe &h, const LayerDev &w, int T)
{
    const k3moe_config &c = h.cfg;
    ExpTArgs a;
    a.wslot = w.wslot;
    a.n_ws = w.n_wslots;
    a.L = c.latent;
    a.k = c.topk;
    a.E = c.n_experts;
    a.T = T;
    a.offsets = h.ws.offsets;
    a.perm = h.ws.perm;
    a.z16 = h.ws.z16;
    a.h16 = h.ws.h16;
    a.pair_w = h.ws.pair_w;
    a.acc = h.ws.acc;
    a.b1 = c.situ_b1;
    a.b2 = c.situ_b2;
    a.ib1 = 1.f / c.situ_b1;
    a.ib2 = 1.f / c.situ_b2;
    a.err = h.ws.err;
    return a;
}

cudaError_t launch_expert_w13(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    ExpTArgs a = base_args(h, w, T);
    a.pa = w.w1p;
    a.sa = w.w1s;
    a.pb = w.w3p;
    a.sb = w.w3s;
    a.K = h.cfg.latent;
    a.R = h.cfg.moe_inter;
    a.units = (long long)T * h.cfg.topk * (a.R / UnitShape<true>::rows);
    const int grid = (int)(a.units < h.sm_count ? a.units : h.sm_count);
    return launch_pdl(k_expert_tma<true>, grid, kThreads, exp_smem(a.K, true, a.E), s, a);
}

cudaError_t launch_expert_w2(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    ExpTArgs a = base_args(h, w, T);
    a.pa = w.w2p;
    a.sa = w.w2s;
    a.pb = nullptr;
    a.sb = nullptr;
    a.K = h.cfg.moe_inter;
    a.R = h.cfg.latent;
    a.units = (long long)T * h.cfg.topk * (a.R / UnitShape<false>::rows);
    const int grid = (int)(a.units < h.sm_count ? a.units : h.sm_count);
    return launch_pdl(k_expert_tma<false>, grid, kThreads, exp_smem(a.K, false, a.E), s, a);
}

}  // namespace k3
