// Expert tier: the routed experts of every loaded layer live in pinned host
// memory, and a pool of device slots caches them (kimi-k3-in-c README,
// Part II section 12, "An LRU cache for the experts": a slot holds one
// (layer, expert) key or is free; a miss takes a free slot first, else the
// least recently used one; all misses of a request are reserved one after
// another, then read in parallel, then published). Host memory over the
// NVLink-C2C link takes the place of the pages' disk, HBM that of their RAM.
//
// Per forward, after routing, on the forward's stream:
//   k_tier_plan  (one block): stamps the slots of the touched experts that are
//                resident (hits), picks for the others (misses) the slots with
//                the oldest stamps among those this forward does not use (free
//                slots carry stamp 0, so they go first; equal stamps: lower
//                slot first), retires the victims' old keys, publishes the new
//                ones and writes the (slot, expert) fill list;
//   k_tier_fill  (every SM): copies the listed experts' nine arrays from the
//                device-mapped host block into their slots.
// The expert kernels then address expert e at slot slot_of[layer][e]. A pool
// of at least n_experts slots always holds one forward's experts, since the
// slots a forward hits carry its own stamp and are never victims.
#include "k3moe_internal.cuh"

namespace k3 {

constexpr int kPlanThreads = 1024;
constexpr int kPlanPer = kTierMaxSlots / kPlanThreads;   // slots per thread
constexpr int kFillThreads = 512;
constexpr int kFillVec = 8;                              // 16-byte loads in flight per thread
constexpr size_t kFillChunk = (size_t)kFillThreads * kFillVec * 16;   // 64 KB

static_assert(kMaxExperts <= kPlanThreads, "one touched expert per plan thread");

// Stamp of a pinned slot: above every forward's stamp, so never a victim.
constexpr uint32_t kPinned = 0xFFFFFFFFu;

struct TierPlanArgs {
    const int *touched, *n_touched;
    int pin;                // 1: the listed experts' slots become pinned
    int *slot_of;           // [max_layers * E]
    int *slot_key;          // [slots]
    uint32_t *slot_used;    // [slots]
    int2 *fill;             // [E]
    int *n_fill;
    unsigned long long *stats;
    int layer, E, slots;
    uint32_t stamp;
    unsigned long long expert_bytes;
    int *err;
};

// Block-wide exclusive prefix sum (kPlanThreads threads); *total gets the sum.
__device__ int plan_excl_scan(int v, int *wsum, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    __syncthreads();   // wsum may still be read by a previous call
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        wsum[lane] = wi - w;   // exclusive over warps
        if (lane == 31) wsum[32] = wi;
    }
    __syncthreads();
    *total = wsum[32];
    return wsum[warp] + inc - v;
}

__device__ int plan_sum(int v, int *wsum)
{
    int t;
    plan_excl_scan(v, wsum, &t);
    return t;
}

__global__ void __launch_bounds__(kPlanThreads) k_tier_plan(TierPlanArgs a)
{
    __shared__ int wsum[33];
    __shared__ int victims[kMaxExperts];
    pdl_launch_dependents();
    pdl_wait();   // the touched list comes from the routing kernels
    const int tid = threadIdx.x;
    int *slot_of_l = a.slot_of + (size_t)a.layer * a.E;
    int nt = *a.n_touched;
    if (nt < 0 || nt > a.E) {
        if (tid == 0) {
            set_err(a.err, kErrBounds, 700);
            *a.n_fill = 0;
        }
        return;
    }
    // 1. hits stamp their slots; misses are ranked in touched order
    int e = -1, miss = 0, hit = 0;
    if (tid < nt) {
        e = a.touched[tid];
        if (e < 0 || e >= a.E) {
            set_err(a.err, kErrBounds, 701);
            e = -1;
        } else {
            const int s = slot_of_l[e];
            if (s >= 0 && s < a.slots) {
                if (a.pin) a.slot_used[s] = kPinned;
                else if (a.slot_used[s] != kPinned) a.slot_used[s] = a.stamp;
                hit = 1;
            } else {
                miss = 1;
            }
        }
    }
    int n_miss;
    const int rank = plan_excl_scan(miss, wsum, &n_miss);   // its barriers order the stamps
    const int n_hit = plan_sum(hit, wsum);
    int n_fill = n_miss;
    if (n_miss > 0) {
        // 2. victims: the n_miss slots of smallest stamp below this forward's
        //    (ties: lower slot index), found as the smallest threshold tau with
        //    #{stamp <= tau} >= n_miss over this thread's contiguous slots
        const int s0 = tid * kPlanPer;
        uint32_t u[kPlanPer];
#pragma unroll
        for (int j = 0; j < kPlanPer; j++)
            u[j] = (s0 + j < a.slots) ? a.slot_used[s0 + j] : 0xFFFFFFFFu;
        int avail = 0;
#pragma unroll
        for (int j = 0; j < kPlanPer; j++) avail += u[j] < a.stamp;
        if (plan_sum(avail, wsum) < n_miss) {   // cannot happen with slots >= E
            if (tid == 0) {
                set_err(a.err, kErrBounds, 702);
                *a.n_fill = 0;
            }
            return;
        }
        uint32_t lo = 0, hi = a.stamp - 1;   // #{stamp <= hi} >= n_miss (pinned slots never count)
        while (lo < hi) {
            const uint32_t mid = lo + (hi - lo) / 2;
            int c = 0;
#pragma unroll
            for (int j = 0; j < kPlanPer; j++) c += u[j] <= mid;
            if (plan_sum(c, wsum) >= n_miss) hi = mid;
            else lo = mid + 1;
        }
        const uint32_t tau = lo;
        int lt = 0, eq = 0;
#pragma unroll
        for (int j = 0; j < kPlanPer; j++) {
            lt += u[j] < tau;
            eq += u[j] == tau;
        }
        const int n_lt = plan_sum(lt, wsum);
        int n_eq_all;
        int eq_before = plan_excl_scan(eq, wsum, &n_eq_all);
        const int need_eq = n_miss - n_lt;   // >= 1 by the choice of tau
        int mine = 0;
        bool take[kPlanPer];
#pragma unroll
        for (int j = 0; j < kPlanPer; j++) {
            take[j] = u[j] < tau || (u[j] == tau && eq_before < need_eq);
            if (u[j] == tau) eq_before++;
            mine += take[j];
        }
        int n_taken;
        int at = plan_excl_scan(mine, wsum, &n_taken);
#pragma unroll
        for (int j = 0; j < kPlanPer; j++)
            if (take[j] && at < kMaxExperts) victims[at++] = s0 + j;
        __syncthreads();
        // 3. publish: retire each victim's old key, install the new one
        if (miss && n_taken == n_miss) {
            const int s = victims[rank];
            const int old = a.slot_key[s];
            if (old >= 0) a.slot_of[old] = -1;
            a.slot_key[s] = a.layer * a.E + e;
            slot_of_l[e] = s;
            a.slot_used[s] = a.pin ? kPinned : a.stamp;
            a.fill[rank] = make_int2(s, e);
        }
        if (n_taken != n_miss) {
            n_fill = 0;
            if (tid == 0) set_err(a.err, kErrBounds, 703);
        }
    }
    if (tid == 0) {
        *a.n_fill = n_fill;
        a.stats[0] += (unsigned long long)n_hit;
        a.stats[1] += (unsigned long long)n_miss;
        a.stats[2] += (unsigned long long)n_miss * a.expert_bytes;
    }
}

struct TierFillArgs {
    const int2 *fill;
    const int *n_fill;
    const uint8_t *src[kTierPieces];   // device-mapped host arrays [E][size]
    uint8_t *dst[kTierPieces];         // slot arrays [slots][size]
    unsigned long long size[kTierPieces];
    int chunk0[kTierPieces + 1];       // first chunk of each piece within one expert
    int E, slots;
    int *err;
};

__global__ void __launch_bounds__(kFillThreads) k_tier_fill(TierFillArgs a)
{
    pdl_launch_dependents();
    pdl_wait();   // the fill list comes from k_tier_plan
    const int nf = *a.n_fill;
    const int C = a.chunk0[kTierPieces];
    const long long total = (long long)nf * C;
    for (long long u = blockIdx.x; u < total; u += gridDim.x) {
        const int i = (int)(u / C), r = (int)(u - (long long)i * C);
        // the piece holding chunk r (constant parameter indices only)
        const uint8_t *sp = a.src[0];
        uint8_t *dp = a.dst[0];
        size_t sz = a.size[0];
        int c0 = 0;
#pragma unroll
        for (int q = 1; q < kTierPieces; q++)
            if (r >= a.chunk0[q]) {
                sp = a.src[q];
                dp = a.dst[q];
                sz = a.size[q];
                c0 = a.chunk0[q];
            }
        const int2 f = a.fill[i];
        if (f.x < 0 || f.x >= a.slots || f.y < 0 || f.y >= a.E) {
            if (threadIdx.x == 0) set_err(a.err, kErrBounds, 710);
            return;
        }
        const size_t off = (size_t)(r - c0) * kFillChunk;
        const int nv = (int)((sz - off < kFillChunk ? sz - off : kFillChunk) / 16);
        const uint4 *src = reinterpret_cast<const uint4 *>(sp + (size_t)f.y * sz + off);
        uint4 *dst = reinterpret_cast<uint4 *>(dp + (size_t)f.x * sz + off);
        uint4 v[kFillVec] = {};
#pragma unroll
        for (int j = 0; j < kFillVec; j++) {
            const int q = threadIdx.x + j * kFillThreads;
            if (q < nv) v[j] = __ldcs(src + q);   // host memory, read once
        }
#pragma unroll
        for (int j = 0; j < kFillVec; j++) {
            const int q = threadIdx.x + j * kFillThreads;
            if (q < nv) dst[q] = v[j];
        }
    }
}

// The ids 0 .. E-1 followed by E: the expert list of a whole layer (pinning).
__global__ void k_tier_iota(int *ids, int E)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < E) ids[i] = i;
    if (i == E) ids[E] = E;
}

cudaError_t launch_tier_iota(const k3moe &h)
{
    const int E = h.cfg.n_experts;
    k_tier_iota<<<(E + 256) / 256, 256>>>(h.tier.all_ids, E);
    return cudaGetLastError();
}

// Shifts every used, unpinned slot's stamp down by `shift` (stamps at or
// below it become 1: used, and older than every later stamp).
__global__ void k_tier_rebase(uint32_t *slot_used, int slots, uint32_t shift)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= slots) return;
    const uint32_t u = slot_used[i];
    if (u != 0u && u != kPinned) slot_used[i] = u > shift ? u - shift : 1u;
}

// A reloaded layer gives up its slots: they become free and its table empty.
__global__ void k_tier_forget(int *slot_of, int *slot_key, uint32_t *slot_used, int layer, int E,
                              int slots)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < E) slot_of[(size_t)layer * E + i] = -1;
    if (i < slots && slot_key[i] >= 0 && slot_key[i] / E == layer) {
        slot_key[i] = -1;
        slot_used[i] = 0;
    }
}

cudaError_t launch_tier_plan(k3moe &h, int layer, cudaStream_t s, bool pin)
{
    TierDev &t = h.tier;
    if (t.stamp >= t.rebase_at) {
        // stream-ordered behind the previous forward's plan (a plain launch
        // starts after the kernel before it has finished)
        const uint32_t shift = t.stamp - t.rebase_keep;
        k_tier_rebase<<<(t.slots + 255) / 256, 256, 0, s>>>(t.slot_used, t.slots, shift);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        t.stamp -= shift;
    }
    TierPlanArgs a;
    // a pin lists every expert of the layer (the table's iota), else the
    // forward's touched experts
    a.touched = pin ? t.all_ids : h.ws.touched;
    a.n_touched = pin ? t.all_ids + h.cfg.n_experts : h.ws.n_touched;
    a.pin = pin ? 1 : 0;
    a.slot_of = t.slot_of;
    a.slot_key = t.slot_key;
    a.slot_used = t.slot_used;
    a.fill = t.fill;
    a.n_fill = t.n_fill;
    a.stats = t.stats;
    a.layer = layer;
    a.E = h.cfg.n_experts;
    a.slots = t.slots;
    a.stamp = ++t.stamp;   // stamp 0 marks a slot never used
    a.expert_bytes = t.expert_bytes;
    a.err = h.ws.err;
    return launch_pdl(k_tier_plan, 1, kPlanThreads, 0, s, a);
}

cudaError_t launch_tier_fill(const k3moe &h, const LayerDev &w, cudaStream_t s)
{
    const TierDev &t = h.tier;
    TierFillArgs a;
    a.fill = t.fill;
    a.n_fill = t.n_fill;
    int c = 0;
    for (int p = 0; p < kTierPieces; p++) {
        a.src[p] = w.hsrc[p];
        a.dst[p] = t.arr[p];
        a.size[p] = t.piece[p];
        a.chunk0[p] = c;
        c += (int)((t.piece[p] + kFillChunk - 1) / kFillChunk);
    }
    a.chunk0[kTierPieces] = c;
    a.E = h.cfg.n_experts;
    a.slots = t.slots;
    a.err = h.ws.err;
    // one CTA per SM: it fits beside a CTA of the T = 1 shared-expert kernel
    // (registers and threads), which launches behind it and overlaps the copy
    return launch_pdl(k_tier_fill, h.sm_count, kFillThreads, 0, s, a);
}

cudaError_t launch_tier_forget(const k3moe &h, int layer, cudaStream_t s)
{
    const int n = h.tier.slots > h.cfg.n_experts ? h.tier.slots : h.cfg.n_experts;
    k_tier_forget<<<(n + 255) / 256, 256, 0, s>>>(h.tier.slot_of, h.tier.slot_key, h.tier.slot_used,
                                                  layer, h.cfg.n_experts, h.tier.slots);
    return cudaGetLastError();
}

}  // namespace k3
