// Router epilogue and token -> expert permutation.
//
// k_route (one block per token): sigmoid of the router logits, the
// score-correction bias added for SELECTION only, a warp-level top-k over up
// to 1024 experts (32 scores per lane, k rounds of a warp arg-max with ties
// going to the lower expert id), and the renormalised UNBIASED weights.
// kimi-k3-in-c README, Part II section 9 (k3_router); colibri
// docs/kimi_k3.md "Stable LatentMoE". The same block prepares the expert GEMV
// input: z scaled by a per-token power of two into fp16, and clears the
// token's fp32 accumulator row.
//
// k_perm (one block): per-expert counts, exclusive offsets, and the pair list
// grouped by expert with tokens in ascending order inside an expert, plus the
// ascending list of experts that received at least one token.
#include <climits>

#include "k3moe_internal.cuh"

namespace k3 {

struct RouteArgs {
    const float *logits;   // [T, E]
    const float *bias;     // [E]
    int T, E, k, renorm;
    float routed_scale;
    int *ids;              // [T, k]
    float *wts;            // [T, k]
    const float *z;        // [T, L]
    __half *z16;           // [T, L]
    int *zexp;             // [T]
    float *acc;            // [T, L]
    int L;
    int *err;
};

constexpr int kPerLane = kMaxExperts / 32;

__global__ void __launch_bounds__(128) k_route(RouteArgs a)
{
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float red[4];
    __shared__ float wsel[kMaxTopk];

    // ---- expert GEMV input: fp16 z with a per-token power-of-two scale ----
    const float *zr = a.z + (size_t)t * a.L;
    float m = 0.f;
    for (int i = threadIdx.x; i < a.L; i += blockDim.x) m = fmaxf(m, fabsf(zr[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    // max * 2^-ex lands in [32, 64): every fp16 product with an e2m1 value
    // (|v| <= 6) and every 16-term partial sum stays far below 65504.
    int ex = 0;
    if (m > 0.f && isfinite(m)) ex = min(max(ilogbf(m) - 5, -100), 100);
    const float sc = __uint_as_float((uint32_t)(127 - ex) << 23);
    for (int i = threadIdx.x; i < a.L; i += blockDim.x) {
        a.z16[(size_t)t * a.L + i] = __float2half_rn(zr[i] * sc);
        a.acc[(size_t)t * a.L + i] = 0.f;
    }
    if (threadIdx.x == 0) a.zexp[t] = ex;

    if (warp != 0) return;
    // ---- router: sigmoid, bias for selection, top-k, weights ----
    const float *lg = a.logits + (size_t)t * a.E;
    float ch[kPerLane], scv[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; i++) {
        const int e = lane + 32 * i;
        if (e < a.E) {
            const float s = sigmoid_f(lg[e]);
            scv[i] = s;
            ch[i] = s + a.bias[e];
        } else {
            scv[i] = 0.f;
            ch[i] = 0.f;
        }
    }
    uint32_t taken = 0;
    for (int j = 0; j < a.k; j++) {
        float bv = 0.f, bs = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < kPerLane; i++) {
            const int e = lane + 32 * i;
            if (e < a.E && !((taken >> i) & 1u)) {
                if (be == INT_MAX || ch[i] > bv) {   // ascending e per lane: '>' keeps the lower id
                    bv = ch[i];
                    be = e;
                    bs = scv[i];
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
                bs = os;
            }
        }
        if (be == INT_MAX) {   // fewer candidates than k: rejected on the host, kept safe here
            if (lane == 0) set_err(a.err, kErrBounds, t);
            return;
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == 0) {
            a.ids[(size_t)t * a.k + j] = be;
            wsel[j] = bs;
        }
    }
    __syncwarp();
    if (lane == 0) {
        float s = 0.f;
        for (int j = 0; j < a.k; j++) s += wsel[j];
        const bool rn = a.renorm && s > 0.f;
        for (int j = 0; j < a.k; j++) {
            const float w = rn ? wsel[j] / s : wsel[j];
            a.wts[(size_t)t * a.k + j] = w * a.routed_scale;
        }
    }
}

cudaError_t launch_route(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    const k3moe_config &c = h.cfg;
    RouteArgs a;
    a.logits = h.ws.logits;
    a.bias = w.bias;
    a.T = T;
    a.E = c.n_experts;
    a.k = c.topk;
    a.renorm = c.renorm;
    a.routed_scale = c.routed_scale;
    a.ids = h.ws.ids;
    a.wts = h.ws.wts;
    a.z = h.ws.z;
    a.z16 = h.ws.z16;
    a.zexp = h.ws.zexp;
    a.acc = h.ws.acc;
    a.L = c.latent;
    a.err = h.ws.err;
    k_route<<<T, 128, 0, s>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------

struct PermArgs {
    const int *ids;   // [T, k]
    int T, k, E;
    int *counts, *offsets, *perm, *touched, *n_touched;
    int *err;
};

// Block-wide exclusive scan of one int per thread (1024 threads).
__device__ __forceinline__ int block_excl_scan(int v, int *wsum, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = wsum[lane];
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += n;
        }
        wsum[lane] = si - s;
        if (lane == 31) *total = si;
    }
    __syncthreads();
    const int r = wsum[warp] + incl - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(1024) k_perm(PermArgs a)
{
    extern __shared__ int sm[];
    int *hist = sm;                       // [32][E]: per-warp counts, then per-warp bases
    int *base = sm + 32 * a.E;            // [E]: expert offsets
    __shared__ int wsum[32];
    __shared__ int total_pairs, total_touched;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 32 * a.E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int tpw = (a.T + 31) / 32;
    const int tb = warp * tpw, te = min(a.T, tb + tpw);
    for (int t = tb; t < te; t++) {
        if (lane < a.k) {
            const int e = a.ids[(size_t)t * a.k + lane];
            if (e >= 0 && e < a.E)
                atomicAdd(&hist[warp * a.E + e], 1);
            else
                set_err(a.err, kErrBounds, t);
        }
    }
    __syncthreads();
    // per expert: counts over warps -> per-warp running bases
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < a.E) {
        for (int w = 0; w < 32; w++) {
            const int c = hist[w * a.E + e];
            hist[w * a.E + e] = cnt;
            cnt += c;
        }
    }
    const int off = block_excl_scan(e < a.E ? cnt : 0, wsum, &total_pairs);
    const int tpos = block_excl_scan((e < a.E && cnt > 0) ? 1 : 0, wsum, &total_touched);
    if (e < a.E) {
        base[e] = off;
        a.counts[e] = cnt;
        a.offsets[e] = off;
        if (cnt > 0) a.touched[tpos] = e;
    }
    if (threadIdx.x == 0) {
        a.offsets[a.E] = total_pairs;
        *a.n_touched = total_touched;
    }
    __syncthreads();
    // placement: each warp walks its tokens in order, so tokens stay ascending
    for (int t = tb; t < te; t++) {
        if (lane < a.k) {
            const int ee = a.ids[(size_t)t * a.k + lane];
            if (ee >= 0 && ee < a.E) {
                const int pos = base[ee] + atomicAdd(&hist[warp * a.E + ee], 1);
                a.perm[pos] = t * a.k + lane;
            }
        }
        __syncwarp();
    }
}

cudaError_t launch_perm(const k3moe &h, int T, cudaStream_t s)
{
    const k3moe_config &c = h.cfg;
    PermArgs a;
    a.ids = h.ws.ids;
    a.T = T;
    a.k = c.topk;
    a.E = c.n_experts;
    a.counts = h.ws.counts;
    a.offsets = h.ws.offsets;
    a.perm = h.ws.perm;
    a.touched = h.ws.touched;
    a.n_touched = h.ws.n_touched;
    a.err = h.ws.err;
    const size_t smem = (size_t)33 * c.n_experts * sizeof(int);
    cudaFuncSetAttribute(k_perm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_perm<<<1, 1024, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace k3
