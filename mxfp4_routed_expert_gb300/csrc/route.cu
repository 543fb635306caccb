// Router epilogue and token -> expert permutation.
//
// k_route (one block per token): sigmoid of the router logits, the
// score-correction bias added for SELECTION only, a warp-level top-k over up
// to 1024 experts (32 scores per lane, k rounds of a warp arg-max with ties
// going to the lower expert id), and the renormalised UNBIASED weights.
// kimi-k3-in-c README, Part II section 9 (k3_router); colibri
// docs/kimi_k3.md "Stable LatentMoE". The same block prepares the expert GEMV
// input: z scaled by a per-token power of two into fp16 (and, for the grouped
// block-scaled path, z in two-term MXFP8), and clears the token's fp32
// accumulator row.
//
// Permutation (three launches over 32-token chunks, T > 1): per-expert
// counts, exclusive offsets, and the pair list grouped by expert with tokens
// in ascending order inside an expert, plus the ascending list of experts
// that received at least one token. For T == 1 k_route writes these itself.
#include <climits>

#include "decode_common.cuh"

namespace k3 {

__global__ void __launch_bounds__(kRouteThreads) k_route(RouteArgs a)
{
    __shared__ RouteSmem rs;
    pdl_launch_dependents();
    route_token(a, blockIdx.x, rs, RouteBlockSync{}, [] { pdl_wait(); });
}

// The router epilogue's arguments for a batch of T tokens (T == 1 also writes
// the pair tables).
static RouteArgs route_args(const k3moe &h, const LayerDev &w, int T)
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
    a.topp = h.topp;
    a.ids = h.ws.ids;
    a.wts = h.ws.wts;
    a.z = h.ws.z;
    a.z16 = h.ws.z16;
    // the block-scaled grouped expert path reads z in two-term MXFP8
    const bool mx = (h.egemm_ok && expert_gemm_mx(h, T) && T * c.topk >= expert_gemm_min_pairs()) ||
                    use_expert_split(h, T);
    a.zq = mx ? h.ws.zq : nullptr;
    a.zqs = mx ? h.ws.zqs : nullptr;
    a.zq_rows = c.max_tokens;
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
    return a;
}

cudaError_t launch_route(const k3moe &h, const LayerDev &w, int T, cudaStream_t s)
{
    const RouteArgs a = route_args(h, w, T);
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
// Steps 1 and 3 first copy the chunk's ids (and weights) to shared memory with
// all their loads in flight, so that the serial pass over the chunk's tokens
// waits on no global load.
constexpr int kPermChunk = 32;
constexpr int kPermWarps = 8;            // chunks per block in steps 1 and 3

// shared memory of steps 1 (place = false) and 3: per warp the expert
// counters [E], then the chunk's ids [kPermChunk * k] (and weights)
size_t perm_smem(const k3moe_config &c, bool place)
{
    return (size_t)kPermWarps * ((size_t)c.n_experts + (size_t)kPermChunk * c.topk * (place ? 2 : 1)) * sizeof(int);
}

__global__ void __launch_bounds__(kPermWarps * 32) k_perm_hist(PermArgs a, int *hist)
{
    extern __shared__ int sh[];          // per warp: [E] counters, [kPermChunk * k] ids
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *h = sh + (size_t)warp * (a.E + kPermChunk * a.k);
    int *ids = h + a.E;
    pdl_launch_dependents();
    pdl_wait();
    const int chunk = blockIdx.x * kPermWarps + warp;
    const int t0 = chunk * kPermChunk;
    if (t0 >= a.T) return;
    const int nt = min(a.T, t0 + kPermChunk) - t0;
    for (int i = lane; i < nt * a.k; i += 32) ids[i] = a.ids[(size_t)t0 * a.k + i];
    for (int e = lane; e < a.E; e += 32) h[e] = 0;
    __syncwarp();
    for (int t = 0; t < nt; t++) {
        if (lane < a.k) {
            const int e = ids[t * a.k + lane];
            if (e >= 0 && e < a.E) h[e] += 1;      // distinct experts within a token
            else if (e != -1) set_err(a.err, kErrBounds, t0 + t);   // -1: dropped by the weight cut
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
    extern __shared__ int sh[];          // per warp: [E] next position per expert, the chunk's ids and weights
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *pos = sh + (size_t)warp * (a.E + 2 * kPermChunk * a.k);
    int *ids = pos + a.E;
    float *wv = reinterpret_cast<float *>(ids + kPermChunk * a.k);
    pdl_launch_dependents();
    pdl_wait();
    const int chunk = blockIdx.x * kPermWarps + warp;
    const int t0 = chunk * kPermChunk;
    if (t0 >= a.T) return;
    const int nt = min(a.T, t0 + kPermChunk) - t0;
    for (int i = lane; i < nt * a.k; i += 32) {
        ids[i] = a.ids[(size_t)t0 * a.k + i];
        wv[i] = a.wts[(size_t)t0 * a.k + i];
    }
    const int *base = hist + (size_t)chunk * a.E;
    for (int e = lane; e < a.E; e += 32) pos[e] = a.offsets[e] + base[e];
    __syncwarp();
    for (int t = 0; t < nt; t++) {
        if (lane < a.k) {
            const int e = ids[t * a.k + lane];
            if (e >= 0 && e < a.E) {
                const int p = pos[e]++;
                a.perm[p] = (t0 + t) * a.k + lane;
                a.pair_w[p] = wv[t * a.k + lane];
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
    if (step == 0) return launch_pdl(k_perm_hist, blocks, kPermWarps * 32, perm_smem(c, false), s, a, h.ws.perm_hist);
    if (step == 1) return launch_pdl(k_perm_scan, 1, 1024, 0, s, a, h.ws.perm_hist, nch);
    return launch_pdl(k_perm_place, blocks, kPermWarps * 32, perm_smem(c, true), s, a,
                      (const int *)h.ws.perm_hist);
}

cudaError_t init_route_kernels(const k3moe_config &c)
{
    cudaError_t e = cudaFuncSetAttribute(k_perm_hist, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)perm_smem(c, false));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_perm_place, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)perm_smem(c, true));
}

}  // namespace k3
