// MXFP4 routed-expert GEMVs for small per-expert token counts (decode).
//
// The expert weights are read exactly as stored: e2m1 nibbles two per byte
// (low nibble = even column, bit 3 = sign) with one ue8m0 scale per 32
// columns (kimi-k3-in-c README, Part II section 4 and k3_matmul_mxfp4;
// colibri docs/kimi_k3.md "Weights"). One 16-byte load is 32 nibbles, i.e.
// exactly one scale group. The nibbles are widened in registers with
// cvt.rn.f16x2.e2m1x2 (exact), multiplied with fp16 activations by packed
// f16x2 FMAs over the 32 columns of a group, and the group partial is scaled
// by 2^(s-127) and accumulated in fp32.
//
// k_w13: for each (touched expert, block of rows) the gate row of W1 and the
//   up row of W3 are dotted with the fp16 latent of each token routed there;
//   SiTU-GLU is applied in the epilogue and h is written in pair order
//   (README section 9, k3_moe step 3 and k3_situ_glu).
// k_w2: h . W2^T per pair, multiplied by the pair's routing weight and
//   scatter-added into the token's fp32 latent accumulator.
#include "k3moe_internal.cuh"

namespace k3 {

constexpr int kExpWarps = 8;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerItem = kExpWarps * kRowsPerWarp;   // 32
constexpr int kMaxChunks = 8;                            // 16-byte chunks per lane and row

struct ExpArgs {
    const uint8_t *pa, *sa;   // W1 (w13) or W2 (w2): packed, scales
    const uint8_t *pb, *sb;   // W3 (w13 only)
    int K;                    // input width of the matrix (L for w13, I for w2)
    int R;                    // rows of the matrix (I for w13, L for w2)
    int k, E;
    int L, I;
    const int *touched, *n_touched, *counts, *offsets, *perm;
    const __half *z16;        // w13 input [T, L]
    const int *zexp;          // [T]
    __half *h16;              // w13 output / w2 input [T*k, I]
    const float *wts;         // [T, k]
    float *acc;               // w2 output [T, L]
    float b1, b2;
    int T;
    int *err;
};

// Dot of one 32-column group: 16 packed bytes against 32 fp16 activations.
__device__ __forceinline__ float group_dot(const uint4 w, const __half *xg)
{
    const uint4 *xp = reinterpret_cast<const uint4 *>(xg);
    const uint4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
    const uint32_t xw[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                             x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t h = 0u;
#pragma unroll
    for (int q = 0; q < 4; q++)
#pragma unroll
        for (int b = 0; b < 4; b++) h = hfma2(e2m1x2_to_f16x2((ww[q] >> (8 * b)) & 0xFFu),
                                             xw[4 * q + b], h);
    return f16x2_sum(h);
}

// Stage the activations of tokens [g0, g0+tg) of one expert into shared memory.
template <int TG>
__device__ __forceinline__ void stage_rows(const __half *src_base, const int *rows_idx, int tg,
                                           int K, __half *xs)
{
    const int v_per_row = K / 8;
    for (int i = threadIdx.x; i < TG * v_per_row; i += blockDim.x) {
        const int t = i / v_per_row, c = i - t * v_per_row;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < tg) v = reinterpret_cast<const uint4 *>(src_base + (size_t)rows_idx[t] * K)[c];
        reinterpret_cast<uint4 *>(xs)[i] = v;
    }
}

template <int TG>
__global__ void __launch_bounds__(kExpWarps * 32) k_w13(ExpArgs a)
{
    extern __shared__ __align__(16) unsigned char smraw[];
    __half *xs = reinterpret_cast<__half *>(smraw);   // [TG][L]
    __shared__ int tok[TG], slot[TG];
    __shared__ float zsc[TG];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.K / kGroup;          // groups per row
    const int nchunk = 2 * G;            // W1 groups, then W3 groups
    const int rb_per = a.R / kRowsPerItem;
    const int n_items = *a.n_touched * rb_per;
    const size_t prow = (size_t)a.K / 2, srow = (size_t)G;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int si = item / rb_per, rb = item - si * rb_per;
        const int e = a.touched[si];
        if (e < 0 || e >= a.E) {
            if (threadIdx.x == 0) set_err(a.err, kErrBounds, e);
            return;
        }
        const int cnt = a.counts[e], off = a.offsets[e];
        const uint8_t *P1 = a.pa + (size_t)e * a.R * prow, *S1 = a.sa + (size_t)e * a.R * srow;
        const uint8_t *P3 = a.pb + (size_t)e * a.R * prow, *S3 = a.sb + (size_t)e * a.R * srow;
        for (int g0 = 0; g0 < cnt; g0 += TG) {
            const int tg = min(TG, cnt - g0);
            __syncthreads();
            if (threadIdx.x < TG) {
                const int i = threadIdx.x;
                int t = 0, sl = 0;
                if (i < tg) {
                    sl = off + g0 + i;
                    t = a.perm[sl] / a.k;
                    if (t < 0 || t >= a.T) {
                        set_err(a.err, kErrBounds, t);
                        t = 0;
                    }
                }
                tok[i] = t;
                slot[i] = sl;
                zsc[i] = __uint_as_float((uint32_t)(127 + a.zexp[t]) << 23);
            }
            __syncthreads();
            stage_rows<TG>(a.z16, tok, tg, a.K, xs);
            __syncthreads();
#pragma unroll 1
            for (int rr = 0; rr < kRowsPerWarp; rr++) {
                const int row = rb * kRowsPerItem + warp * kRowsPerWarp + rr;
                uint4 wv[kMaxChunks];
                uint32_t sv[kMaxChunks];
#pragma unroll
                for (int q = 0; q < kMaxChunks; q++) {
                    const int c = lane + 32 * q;
                    if (c < nchunk) {
                        const bool b3 = c >= G;
                        const int g = b3 ? c - G : c;
                        wv[q] = ld_stream((b3 ? P3 : P1) + row * prow + (size_t)g * 16);
                        sv[q] = (b3 ? S3 : S1)[row * srow + g];
                    }
                }
                float acc1[TG], acc3[TG];
#pragma unroll
                for (int t = 0; t < TG; t++) acc1[t] = acc3[t] = 0.f;
#pragma unroll
                for (int q = 0; q < kMaxChunks; q++) {
                    const int c = lane + 32 * q;
                    if (c < nchunk) {
                        const bool b3 = c >= G;
                        const int g = b3 ? c - G : c;
                        const float s = e8m0_to_f32(sv[q]);
#pragma unroll
                        for (int t = 0; t < TG; t++) {
                            const float p = group_dot(wv[q], xs + t * a.K + g * kGroup) * s;
                            if (b3) acc3[t] += p; else acc1[t] += p;
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < TG; t++) {
                    acc1[t] = warp_sum(acc1[t]);
                    acc3[t] = warp_sum(acc3[t]);
                }
                if (lane < tg) {
                    // lane t writes token t (values are identical in every lane)
#pragma unroll
                    for (int t = 0; t < TG; t++) {
                        if (t == lane) {
                            const float gg = acc1[t] * zsc[t], uu = acc3[t] * zsc[t];
                            a.h16[(size_t)slot[t] * a.R + row] =
                                __float2half_rn(situ_f(gg, uu, a.b1, a.b2));
                        }
                    }
                }
            }
        }
    }
}

template <int TG>
__global__ void __launch_bounds__(kExpWarps * 32) k_w2(ExpArgs a)
{
    extern __shared__ __align__(16) unsigned char smraw[];
    __half *xs = reinterpret_cast<__half *>(smraw);   // [TG][I]
    __shared__ int tok[TG], slotrow[TG];
    __shared__ float wgt[TG];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.K / kGroup;
    const int rb_per = a.R / kRowsPerItem;
    const int n_items = *a.n_touched * rb_per;
    const size_t prow = (size_t)a.K / 2, srow = (size_t)G;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int si = item / rb_per, rb = item - si * rb_per;
        const int e = a.touched[si];
        if (e < 0 || e >= a.E) {
            if (threadIdx.x == 0) set_err(a.err, kErrBounds, e);
            return;
        }
        const int cnt = a.counts[e], off = a.offsets[e];
        const uint8_t *P = a.pa + (size_t)e * a.R * prow, *S = a.sa + (size_t)e * a.R * srow;
        for (int g0 = 0; g0 < cnt; g0 += TG) {
            const int tg = min(TG, cnt - g0);
            __syncthreads();
            if (threadIdx.x < TG) {
                const int i = threadIdx.x;
                int t = 0, sl = 0;
                float w = 0.f;
                if (i < tg) {
                    sl = off + g0 + i;
                    const int p = a.perm[sl];
                    t = p / a.k;
                    if (t < 0 || t >= a.T) {
                        set_err(a.err, kErrBounds, t);
                        t = 0;
                    } else {
                        w = a.wts[p];
                    }
                }
                tok[i] = t;
                slotrow[i] = sl;
                wgt[i] = w;
            }
            __syncthreads();
            stage_rows<TG>(a.h16, slotrow, tg, a.K, xs);
            __syncthreads();
#pragma unroll 1
            for (int rr = 0; rr < kRowsPerWarp; rr++) {
                const int row = rb * kRowsPerItem + warp * kRowsPerWarp + rr;
                uint4 wv[kMaxChunks];
                uint32_t sv[kMaxChunks];
#pragma unroll
                for (int q = 0; q < kMaxChunks; q++) {
                    const int c = lane + 32 * q;
                    if (c < G) {
                        wv[q] = ld_stream(P + row * prow + (size_t)c * 16);
                        sv[q] = S[row * srow + c];
                    }
                }
                float acc[TG];
#pragma unroll
                for (int t = 0; t < TG; t++) acc[t] = 0.f;
#pragma unroll
                for (int q = 0; q < kMaxChunks; q++) {
                    const int c = lane + 32 * q;
                    if (c < G) {
                        const float s = e8m0_to_f32(sv[q]);
#pragma unroll
                        for (int t = 0; t < TG; t++)
                            acc[t] += group_dot(wv[q], xs + t * a.K + c * kGroup) * s;
                    }
                }
#pragma unroll
                for (int t = 0; t < TG; t++) acc[t] = warp_sum(acc[t]);
#pragma unroll
                for (int t = 0; t < TG; t++)
                    if (t == lane && t < tg)
                        atomicAdd(&a.acc[(size_t)tok[t] * a.L + row], wgt[t] * acc[t]);
            }
        }
    }
}

static ExpArgs base_args(const k3moe &h, int T)
{
    const k3moe_config &c = h.cfg;
    ExpArgs a;
    a.k = c.topk;
    a.E = c.n_experts;
    a.L = c.latent;
    a.I = c.moe_inter;
    a.touched = h.ws.touched;
    a.n_touched = h.ws.n_touched;
    a.counts = h.ws.counts;
    a.offsets = h.ws.offsets;
    a.perm = h.ws.perm;
    a.z16 = h.ws.z16;
    a.zexp = h.ws.zexp;
    a.h16 = h.ws.h16;
    a.wts = h.ws.wts;
    a.acc = h.ws.acc;
    a.b1 = c.situ_b1;
    a.b2 = c.situ_b2;
    a.T = T;
    a.err = h.ws.err;
    return a;
}

template <typename Kern>
static int exp_grid(const k3moe &h, Kern kern, size_t smem, long long items_upper)
{
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kExpWarps * 32, smem);
    if (per_sm < 1) per_sm = 1;
    const long long cap = (long long)h.sm_count * per_sm;
    return (int)(items_upper < cap ? items_upper : cap);
}

cudaError_t launch_expert_w13(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    ExpArgs a = base_args(h, T);
    a.pa = w.w1p;
    a.sa = w.w1s;
    a.pb = w.w3p;
    a.sb = w.w3s;
    a.K = h.cfg.latent;
    a.R = h.cfg.moe_inter;
    const long long pairs = (long long)T * h.cfg.topk;
    const long long slots = pairs < h.cfg.n_experts ? pairs : h.cfg.n_experts;
    const long long items = slots * (a.R / kRowsPerItem);
    if (T == 1) {
        const size_t smem = (size_t)1 * a.K * sizeof(__half);
        cudaFuncSetAttribute(k_w13<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_w13<1><<<exp_grid(h, k_w13<1>, smem, items), kExpWarps * 32, smem, s>>>(a);
    } else {
        const size_t smem = (size_t)4 * a.K * sizeof(__half);
        cudaFuncSetAttribute(k_w13<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_w13<4><<<exp_grid(h, k_w13<4>, smem, items), kExpWarps * 32, smem, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_expert_w2(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    ExpArgs a = base_args(h, T);
    a.pa = w.w2p;
    a.sa = w.w2s;
    a.pb = nullptr;
    a.sb = nullptr;
    a.K = h.cfg.moe_inter;
    a.R = h.cfg.latent;
    const long long pairs = (long long)T * h.cfg.topk;
    const long long slots = pairs < h.cfg.n_experts ? pairs : h.cfg.n_experts;
    const long long items = slots * (a.R / kRowsPerItem);
    if (T == 1) {
        const size_t smem = (size_t)1 * a.K * sizeof(__half);
        cudaFuncSetAttribute(k_w2<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_w2<1><<<exp_grid(h, k_w2<1>, smem, items), kExpWarps * 32, smem, s>>>(a);
    } else {
        const size_t smem = (size_t)4 * a.K * sizeof(__half);
        cudaFuncSetAttribute(k_w2<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k_w2<4><<<exp_grid(h, k_w2<4>, smem, items), kExpWarps * 32, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace k3
