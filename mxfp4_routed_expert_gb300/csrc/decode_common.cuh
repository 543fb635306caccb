// Device code shared by the decode kernels: the router epilogue of one token
// and the bf16 / MXFP4 dot-product steps of the weight-streaming GEMVs.
#pragma once
#include <climits>

#include "k3moe_internal.cuh"

namespace k3 {

// acc += dot(8 bf16 weights, 8 bf16 activations): fp32 fused multiply-adds on
// bf16 operands, two chains for instruction-level parallelism.
__device__ __forceinline__ void dot8_bf16(const uint4 &w, const uint4 &x, float &a0, float &a1)
{
    asm("{\n\t.reg .b16 w0, w1, w2, w3, w4, w5, w6, w7, x0, x1, x2, x3, x4, x5, x6, x7;\n\t"
        "mov.b32 {w0, w1}, %2;\n\tmov.b32 {w2, w3}, %3;\n\tmov.b32 {w4, w5}, %4;\n\tmov.b32 {w6, w7}, %5;\n\t"
        "mov.b32 {x0, x1}, %6;\n\tmov.b32 {x2, x3}, %7;\n\tmov.b32 {x4, x5}, %8;\n\tmov.b32 {x6, x7}, %9;\n\t"
        "fma.rn.f32.bf16 %0, w0, x0, %0;\n\tfma.rn.f32.bf16 %1, w1, x1, %1;\n\t"
        "fma.rn.f32.bf16 %0, w2, x2, %0;\n\tfma.rn.f32.bf16 %1, w3, x3, %1;\n\t"
        "fma.rn.f32.bf16 %0, w4, x4, %0;\n\tfma.rn.f32.bf16 %1, w5, x5, %1;\n\t"
        "fma.rn.f32.bf16 %0, w6, x6, %0;\n\tfma.rn.f32.bf16 %1, w7, x7, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
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
    uint32_t h;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(h0), "r"(h1));
    return f16x2_sum(h);
}

// ---- router epilogue (kimi-k3-in-c README, Part II section 9, k3_router;
//      colibri docs/kimi_k3.md "Stable LatentMoE") ----

struct RouteArgs {
    const float *logits;   // [T, E]
    const float *bias;     // [E]
    int T, E, k, renorm;
    float routed_scale;
    int *ids;              // [T, k]
    float *wts;            // [T, k]
    const float *z;        // [T, L]
    __half *z16;           // [T, L + kZPad]: scaled fp16 z, then the exponent (int32)
    uint8_t *zq, *zqs;     // null, or two-term MXFP8 z: [2][zq_rows][L] e4m3, [2][zq_rows][L/32] scales
    int zq_rows;
    float *acc;            // [T, L]
    int L;
    float topp;            // > 0: keep the picks up to cumulative weight topp (0: all k)
    int fuse_perm;         // T == 1: also write counts/offsets/perm/touched
    int *counts, *offsets, *perm, *touched, *n_touched;
    float *pair_w;
    int *err;
};

constexpr int kRouteThreads = 256;   // threads that run route_token
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kZPer = 4096 / kRouteThreads;          // latent <= 4096
constexpr int kEPer = kMaxExperts / kRouteThreads;   // experts per thread (contiguous ids)

// Float -> unsigned key with the same order (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Barrier over the kRouteThreads threads that run the router epilogue.
struct RouteBlockSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Sum of one int per thread over the route threads; `buf` holds kRouteWarps ints.
template <class Sync>
__device__ __forceinline__ int block_sum(int v, int *buf, Sync sync)
{
    v = __reduce_add_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) buf[threadIdx.x >> 5] = v;
    sync();
    int s = 0;
#pragma unroll
    for (int w = 0; w < kRouteWarps; w++) s += buf[w];
    return s;
}

// Exclusive prefix sum in thread order over the route threads; `buf` holds kRouteWarps ints.
template <class Sync>
__device__ __forceinline__ int block_excl(int v, int *buf, Sync sync)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) buf[warp] = incl;
    sync();
    int base = 0;
    for (int w = 0; w < warp; w++) base += buf[w];
    return base + incl - v;
}

// Shared-memory scratch of route_token.
struct RouteSmem {
    float red[kRouteWarps];
    int cnt[2][kRouteWarps];
    int scan_buf[kRouteWarps];
    float sel_ch[kMaxTopk], sel_sc[kMaxTopk];
    int sel_e[kMaxTopk];
    int sel_keep[kMaxTopk];   // 1: the pick survives the cumulative-weight cut
};

// The router epilogue of token t on threads 0 .. kRouteThreads-1 (which all
// call it), `sync` their barrier. `ready()` runs after the selection bias is
// read and before the logits and z are: the wait for the kernel that wrote them.
template <class Sync, class Ready>
__device__ __forceinline__ void route_token(const RouteArgs &a, int t, RouteSmem &rs, Sync sync, Ready ready)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *red = rs.red;
    int(*cnt)[kRouteWarps] = rs.cnt;
    int *scan_buf = rs.scan_buf;
    float *sel_ch = rs.sel_ch, *sel_sc = rs.sel_sc;
    int *sel_e = rs.sel_e;
    int *sel_keep = rs.sel_keep;
    // the selection bias is a layer weight: read it before waiting on the router
    float bv[kEPer];
#pragma unroll
    for (int j = 0; j < kEPer; j++) {
        const int e = kEPer * tid + j;
        bv[j] = e < a.E ? a.bias[e] : 0.f;
    }
    ready();

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
        sync();
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
    const int packed_before = block_excl(gt | (eq << 16), scan_buf, sync);
    sync();
    const int n_gt = block_sum(gt, scan_buf, sync);
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
    sync();

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
    if (a.zq) {
        // the tensor-core expert path's copy of z: the 32 lanes of a warp hold
        // 32 consecutive latent values, one scale group (L % 32 == 0)
        const size_t pl = (size_t)a.zq_rows * a.L;
#pragma unroll
        for (int q = 0; q < kZPer; q++) {
            const int i0 = (tid & ~31) + q * kRouteThreads;
            if (i0 < a.L) {
                const int i = i0 + (tid & 31);
                uint32_t qh, ql;
                int eh, el;
                mx8_hilo(zv[q], qh, ql, eh, el);
                a.zq[(size_t)t * a.L + i] = (uint8_t)qh;
                a.zq[pl + (size_t)t * a.L + i] = (uint8_t)ql;
                if ((tid & 31) == 0) {
                    a.zqs[((size_t)t * a.L + i) / kGroup] = (uint8_t)(eh + 127);
                    a.zqs[(pl + (size_t)t * a.L + i) / kGroup] = (uint8_t)(el + 127);
                }
            }
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
        const bool rn = a.renorm && ssum > 0.f;
        float wv = have ? (rn ? sc / ssum : sc) * a.routed_scale : 0.f;
        // Cumulative-weight cut (the pages' K3_TOPP: the low-weight tail of
        // the picks is dropped and the rest renormalised): in weight order
        // (larger first, equal: lower id), a pick is kept while the weight
        // before it is below topp of the total; the kept weights are scaled
        // back to the total.
        bool keep = have;
        if (a.topp > 0.f) {
            float total = 0.f, before = 0.f;
            for (int q = 0; q < a.k; q++) {
                const float wq = __shfl_sync(0xffffffffu, wv, q);
                const int eq_ = __shfl_sync(0xffffffffu, e, q);
                total += wq;
                if (q != lane && (wq > wv || (wq == wv && eq_ < e))) before += wq;
            }
            keep = have && (total <= 0.f || before < a.topp * total);
            float kept = 0.f;
            for (int q = 0; q < a.k; q++) {
                const float wq = __shfl_sync(0xffffffffu, wv, q);
                const bool kq = __shfl_sync(0xffffffffu, keep ? 1 : 0, q) != 0;
                if (kq) kept += wq;
            }
            if (keep && kept > 0.f) wv = wv * (total / kept);
        }
        // positions: kept picks first in selection order, dropped ones after
        // (without a cut: the selection rank and the id rank)
        const unsigned kmask = __ballot_sync(0xffffffffu, keep);
        int pos = rank, kid = id_rank;
        if (a.topp > 0.f) {
            pos = 0;
            kid = 0;
            for (int q = 0; q < a.k; q++) {
                const bool kq = (kmask >> q) & 1u;
                const float vq = __shfl_sync(0xffffffffu, v, q);
                const int eq_ = __shfl_sync(0xffffffffu, e, q);
                const bool q_first = vq > v || (vq == v && eq_ < e);   // q before this lane (selection order)
                if (keep ? (kq && q_first) : (kq || q_first)) pos++;
                if (kq && eq_ < e) kid++;
            }
        }
        const int m_kept = __popc(kmask);
        if (have) {
            a.ids[(size_t)t * a.k + pos] = keep ? e : -1;
            a.wts[(size_t)t * a.k + pos] = keep ? wv : 0.f;
            if (a.fuse_perm && keep) {   // single token: one pair per kept expert, in id order
                a.perm[kid] = pos;
                a.pair_w[kid] = wv;
                a.touched[kid] = e;
            }
            sel_keep[lane] = keep ? 1 : 0;   // lane q holds pick sel_e[q]
        }
        if (a.fuse_perm && lane == 0) *a.n_touched = m_kept;
    }
    if (a.fuse_perm) {
        if (a.topp > 0.f) sync();   // sel_keep from warp 0
        // counts/offsets for every expert: offsets[e] = #kept picks below e
        for (int e = tid; e <= a.E; e += kRouteThreads) {
            int below = 0, here = 0;
            if (a.topp > 0.f) {
                for (int q = 0; q < a.k; q++) {
                    const int kq = sel_keep[q];
                    below += (kq && sel_e[q] < e) ? 1 : 0;
                    here += (kq && sel_e[q] == e) ? 1 : 0;
                }
            } else {
                for (int q = 0; q < a.k; q++) {
                    below += sel_e[q] < e ? 1 : 0;
                    here += sel_e[q] == e ? 1 : 0;
                }
            }
            a.offsets[e] = below;
            if (e < a.E) a.counts[e] = here;
        }
    }
}


}  // namespace k3
