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
// Permutation (three launches over 32-token chunks, T > 1): per-expert
// counts, exclusive offsets, and the pair list grouped by expert with tokens
// in ascending order inside an expert, plus the ascending list of experts
// that received at least one token. For T == 1 k_route writes these itself.
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
    __half *z16;           // [T, L + kZPad]: scaled fp16 z, then the exponent (int32)
    float *acc;            // [T, L]
    int L;
    int fuse_perm;         // T == 1: also write counts/offsets/perm/touched
    int *counts, *offsets, *perm, *touched, *n_touched;
    float *pair_w;
    int *err;
};

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kZPer = 4096 / kRouteThreads;          // latent <= 4096
constexpr int kEPer = kMaxExperts / kRouteThreads;   // experts per thread (contiguous ids)

// Float -> unsigned key with the same order (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide sum of one int per thread; `buf` holds kRouteWarps ints.
__device__ __forceinline__ int block_sum(int v, int *buf)
{
    v = __reduce_add_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) buf[threadIdx.x >> 5] = v;
    __syncthreads();
    int s = 0;
#pragma unroll
    for (int w = 0; w < kRouteWarps; w++) s += buf[w];
    return s;
}

// Block-wide exclusive prefix sum in thread order; `buf` holds kRouteWarps ints.
__device__ __forceinline__ int block_excl(int v, int *buf)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) buf[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; w++) base += buf[w];
    return base + incl - v;
}

__global__ void __launch_bounds__(kRouteThreads) k_route(RouteArgs a)
{
    const int t = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float red[kRouteWarps];
    __shared__ int cnt[2][kRouteWarps];
    __shared__ int scan_buf[kRouteWarps];
    __shared__ float sel_ch[kMaxTopk], sel_sc[kMaxTopk];
    __shared__ int sel_e[kMaxTopk];
    pdl_launch_dependents();
    // the selection bias is a layer weight: read it before waiting on the router
    float bv[kEPer];
#pragma unroll
    for (int j = 0; j < kEPer; j++) {
        const int e = kEPer * tid + j;
        bv[j] = e < a.E ? a.bias[e] : 0.f;
    }
    pdl_wait();

    // ---- expert GEMV input: fp16 z with a per-token power-of-two scale ----
    const float *zr = a.z + (size_t)t * a.L;
    float zv[kZPer];
    float m = 0.f;
#pragma unroll
    for (int q = 0; q < kZPer; q++) {
        const int i = tid + q * kRouteThreads;
        zv[q] = i < a.L ? zr[i] : 0.f;
        m = fmaxf(m, fabsf(zv[q]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;

    // ---- router scores: thread tid owns experts kEPer*tid ... kEPer*tid + kEPer-1 ----
    const float *lg = a.logits + (size_t)t * a.E;
    float ch[kEPer], scv[kEPer];
    uint32_t key[kEPer];
    bool valid[kEPer];
#pragma unroll
    for (int j = 0; j < kEPer; j++) {
        const int e = kEPer * tid + j;
        valid[j] = e < a.E;
        const float sgm = valid[j] ? sigmoid_f(lg[e]) : 0.f;
        scv[j] = sgm;
        ch[j] = sgm + bv[j];
        key[j] = order_key(ch[j]);
    }
    // k-th largest key by a bitwise search: the largest thr with #(key >= thr) >= k
    uint32_t thr = 0u;
    for (int bit = 31; bit >= 0; bit--) {
        const uint32_t cand = thr | (1u << bit);
        int c = 0;
#pragma unroll
        for (int j = 0; j < kEPer; j++) c += (valid[j] && key[j] >= cand) ? 1 : 0;
        c = __reduce_add_sync(0xffffffffu, c);
        int *buf = cnt[bit & 1];
        if (lane == 0) buf[warp] = c;
        __syncthreads();
        int total = 0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; w++) total += buf[w];
        if (total >= a.k) thr = cand;
    }
    // experts above thr are all picked; ties at thr go to the lower ids
    int gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < kEPer; j++) {
        gt += (valid[j] && key[j] > thr) ? 1 : 0;
        eq += (valid[j] && key[j] == thr) ? 1 : 0;
    }
    const int packed_before = block_excl(gt | (eq << 16), scan_buf);
    __syncthreads();
    const int n_gt = block_sum(gt, scan_buf);
    int gt_before = packed_before & 0xFFFF, eq_before = packed_before >> 16;
    const int need_eq = a.k - n_gt;
#pragma unroll
    for (int j = 0; j < kEPer; j++) {
        if (!valid[j]) continue;
        int pos = -1;
        if (key[j] > thr) {
            pos = gt_before++;
        } else if (key[j] == thr) {
            if (eq_before < need_eq) pos = n_gt + eq_before;
            eq_before++;
        }
        if (pos >= 0 && pos < a.k) {
            sel_ch[pos] = ch[j];
            sel_sc[pos] = scv[j];
            sel_e[pos] = kEPer * tid + j;
        }
    }
    __syncthreads();

    m = red[0];
#pragma unroll
    for (int w = 1; w < kRouteWarps; w++) m = fmaxf(m, red[w]);
    // max * 2^-ex lands in [32, 64): every fp16 product with an e2m1 value
    // (|v| <= 6) and every 16-term partial sum stays far below 65504.
    int ex = 0;
    if (m > 0.f && isfinite(m)) ex = min(max(ilogbf(m) - 5, -100), 100);
    const float zsc = __uint_as_float((uint32_t)(127 - ex) << 23);
#pragma unroll
    for (int q = 0; q < kZPer; q++) {
        const int i = tid + q * kRouteThreads;
        if (i < a.L) {
            a.z16[(size_t)t * (a.L + kZPad) + i] = __float2half_rn(zv[q] * zsc);
            a.acc[(size_t)t * a.L + i] = 0.f;
        }
    }
    if (tid == 0) *reinterpret_cast<int *>(a.z16 + (size_t)t * (a.L + kZPad) + a.L) = ex;

    // ---- warp 0: selection order (ch desc, id asc), weights, and for T == 1
    //      the permutation tables ----
    if (warp == 0) {
        const bool have = lane < a.k;
        const float v = have ? sel_ch[lane] : 0.f;
        const int e = have ? sel_e[lane] : INT_MAX;
        const float sc = have ? sel_sc[lane] : 0.f;
        int rank = 0, id_rank = 0;
        for (int q = 0; q < a.k; q++) {
            const float vq = __shfl_sync(0xffffffffu, v, q);
            const int eq_ = __shfl_sync(0xffffffffu, e, q);
            rank += (vq > v || (vq == v && eq_ < e)) ? 1 : 0;
            id_rank += (eq_ < e) ? 1 : 0;
        }
        float ssum = sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
        if (have) {
            const bool rn = a.renorm && ssum > 0.f;
            const float wv = (rn ? sc / ssum : sc) * a.routed_scale;
            a.ids[(size_t)t * a.k + rank] = e;
            a.wts[(size_t)t * a.k + rank] = wv;
            if (a.fuse_perm) {   // single token: one pair per picked expert, in id order
                a.perm[id_rank] = rank;
                a.pair_w[id_rank] = wv;
                a.touched[id_rank] = e;
            }
        }
        if (a.fuse_perm && lane == 0) *a.n_touched = a.k;
    }
    if (a.fuse_perm) {
        // counts/offsets for every expert: offsets[e] = #picked ids below e
        for (int e = tid; e <= a.E; e += kRouteThreads) {
            int below = 0, here = 0;
            for (int q = 0; q < a.k; q++) {
                below += sel_e[q] < e ? 1 : 0;
                here += sel_e[q] == e ? 1 : 0;
            }
            a.offsets[e] = below;
            if (e < a.E) a.counts[e] = here;
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
    a.acc = h.ws.acc;
    a.L = c.latent;
    a.fuse_perm = T == 1;
    a.counts = h.ws.counts;
    a.offsets = h.ws.offsets;
    a.perm = h.ws.perm;
    a.touched = h.ws.touched;
    a.n_touched = h.ws.n_touched;
    a.pair_w = h.ws.pair_w;
    a.err = h.ws.err;
    return launch_pdl(k_route, T, kRouteThreads, 0, s, a);
}

// ---------------------------------------------------------------------------

struct PermArgs {
    const int *ids;   // [T, k]
    const float *wts; // [T, k]
    int T, k, E;
    int *counts, *offsets, *perm, *touched, *n_touched;
    float *pair_w;    // [T*k] weight of each pair slot
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

// The permutation is a stable counting sort of the (token, slot) pairs by
// expert, in three launches over chunks of kPermChunk tokens:
//   1. per chunk (one warp), the number of its pairs that chose each expert;
//   2. (one block, a thread per expert) each chunk's starting position per
//      expert = the expert's offset + the pairs of earlier chunks, the expert
//      counts, offsets and the list of touched experts;
//   3. per chunk (one warp), its pairs placed in token order. The k experts of
//      one token are distinct, so the lanes of a step never share a counter and
//      tokens stay ascending inside every expert's run.
constexpr int kPermChunk = 32;
constexpr int kPermWarps = 8;            // chunks per block in steps 1 and 3

__global__ void __launch_bounds__(kPermWarps * 32) k_perm_hist(PermArgs a, int *hist)
{
    extern __shared__ int sh[];          // [kPermWarps][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *h = sh + warp * a.E;
    pdl_launch_dependents();
    pdl_wait();
    const int chunk = blockIdx.x * kPermWarps + warp;
    const int t0 = chunk * kPermChunk;
    if (t0 >= a.T) return;
    for (int e = lane; e < a.E; e += 32) h[e] = 0;
    __syncwarp();
    const int t1 = min(a.T, t0 + kPermChunk);
    for (int t = t0; t < t1; t++) {
        if (lane < a.k) {
            const int e = a.ids[(size_t)t * a.k + lane];
            if (e >= 0 && e < a.E) h[e] += 1;      // distinct experts within a token
            else set_err(a.err, kErrBounds, t);
        }
        __syncwarp();
    }
    int *out = hist + (size_t)chunk * a.E;
    for (int e = lane; e < a.E; e += 32) out[e] = h[e];
}

__global__ void __launch_bounds__(1024) k_perm_scan(PermArgs a, int *hist, int n_chunks)
{
    __shared__ int wsum[32];
    __shared__ int total_pairs, total_touched;
    pdl_launch_dependents();
    pdl_wait();
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < a.E) {
        // running sum over chunks, four loads in flight
        int c = 0;
        for (; c + 4 <= n_chunks; c += 4) {
            int *p = hist + (size_t)c * a.E + e;
            const int v0 = p[0], v1 = p[a.E], v2 = p[2 * (size_t)a.E], v3 = p[3 * (size_t)a.E];
            p[0] = cnt;
            p[a.E] = cnt + v0;
            p[2 * (size_t)a.E] = cnt + v0 + v1;
            p[3 * (size_t)a.E] = cnt + v0 + v1 + v2;
            cnt += v0 + v1 + v2 + v3;
        }
        for (; c < n_chunks; c++) {
            int *p = hist + (size_t)c * a.E + e;
            const int v = *p;
            *p = cnt;
            cnt += v;
        }
    }
    const int off = block_excl_scan(e < a.E ? cnt : 0, wsum, &total_pairs);
    const int tpos = block_excl_scan((e < a.E && cnt > 0) ? 1 : 0, wsum, &total_touched);
    if (e < a.E) {
        a.counts[e] = cnt;
        a.offsets[e] = off;
        if (cnt > 0) a.touched[tpos] = e;
    }
    if (threadIdx.x == 0) {
        a.offsets[a.E] = total_pairs;
        *a.n_touched = total_touched;
    }
}

__global__ void __launch_bounds__(kPermWarps * 32) k_perm_place(PermArgs a, const int *hist)
{
    extern __shared__ int sh[];          // [kPermWarps][E]: next position per expert
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *pos = sh + warp * a.E;
    pdl_launch_dependents();
    pdl_wait();
    const int chunk = blockIdx.x * kPermWarps + warp;
    const int t0 = chunk * kPermChunk;
    if (t0 >= a.T) return;
    const int *base = hist + (size_t)chunk * a.E;
    for (int e = lane; e < a.E; e += 32) pos[e] = a.offsets[e] + base[e];
    __syncwarp();
    const int t1 = min(a.T, t0 + kPermChunk);
    for (int t = t0; t < t1; t++) {
        if (lane < a.k) {
            const int e = a.ids[(size_t)t * a.k + lane];
            if (e >= 0 && e < a.E) {
                const int p = pos[e]++;
                a.perm[p] = t * a.k + lane;
                a.pair_w[p] = a.wts[(size_t)t * a.k + lane];
            }
        }
        __syncwarp();
    }
}

int perm_chunks(int T) { return (T + kPermChunk - 1) / kPermChunk; }

// step 0: chunk histograms; 1: chunk bases, counts, offsets, touched list;
// 2: placement.
cudaError_t launch_perm(const k3moe &h, int T, cudaStream_t s, int step)
{
    const k3moe_config &c = h.cfg;
    PermArgs a;
    a.ids = h.ws.ids;
    a.wts = h.ws.wts;
    a.pair_w = h.ws.pair_w;
    a.T = T;
    a.k = c.topk;
    a.E = c.n_experts;
    a.counts = h.ws.counts;
    a.offsets = h.ws.offsets;
    a.perm = h.ws.perm;
    a.touched = h.ws.touched;
    a.n_touched = h.ws.n_touched;
    a.err = h.ws.err;
    const int nch = perm_chunks(T);
    const int blocks = (nch + kPermWarps - 1) / kPermWarps;
    const size_t smem = (size_t)kPermWarps * c.n_experts * sizeof(int);
    if (step == 0) return launch_pdl(k_perm_hist, blocks, kPermWarps * 32, smem, s, a, h.ws.perm_hist);
    if (step == 1) return launch_pdl(k_perm_scan, 1, 1024, 0, s, a, h.ws.perm_hist, nch);
    return launch_pdl(k_perm_place, blocks, kPermWarps * 32, smem, s, a, (const int *)h.ws.perm_hist);
}

cudaError_t init_route_kernels(const k3moe_config &c)
{
    const int smem = (int)((size_t)kPermWarps * c.n_experts * sizeof(int));
    cudaError_t e = cudaFuncSetAttribute(k_perm_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_perm_place, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace k3
