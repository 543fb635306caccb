// bf16 weight-streaming GEMVs for small token counts (decode):
//  - k_dense_x: everything that reads the layer input x in one pass over the
//    weights: router logits (x . Wr), the latent down projection z (x . Wd)
//    and the shared experts' gate/up pair with SiTU-GLU fused (x . Ws1, x . Ws3).
//  - k_up: y = Wup . n + Ws2 . s, one K-concatenated pass over the up
//    projection and the shared experts' down projection.
// kimi-k3-in-c README, Part II section 9 (k3_moe steps 1, 2, 5, 6) and
// section 5 (k3_matmul_bf16: bf16 widening is a 16-bit shift).
//
// Each warp owns 4 weight rows; every lane streams 16-byte chunks of those
// rows (one HBM read per weight), the activations of TB tokens sit in shared
// memory as fp32, and the 4 x TB dot products are reduced across the warp at
// the end. Token counts above TB loop over token chunks.
#include "k3moe_internal.cuh"

namespace k3 {

template <int TB>
__device__ __forceinline__ void fma8(const uint4 &w, const float *xsrow, float &a)
{
    const float4 xa = *reinterpret_cast<const float4 *>(xsrow);
    const float4 xb = *reinterpret_cast<const float4 *>(xsrow + 4);
    a = fmaf(bf16lo(w.x), xa.x, a);
    a = fmaf(bf16hi(w.x), xa.y, a);
    a = fmaf(bf16lo(w.y), xa.z, a);
    a = fmaf(bf16hi(w.y), xa.w, a);
    a = fmaf(bf16lo(w.z), xb.x, a);
    a = fmaf(bf16hi(w.z), xb.y, a);
    a = fmaf(bf16lo(w.w), xb.z, a);
    a = fmaf(bf16hi(w.w), xb.w, a);
}

// The loads of a batch of kBatch chunk columns (4 rows each) are issued
// together before any of them is used, so every lane keeps 4*kBatch 16-byte
// loads in flight.
constexpr int kBatch = 4;

template <int TB>
__device__ __forceinline__ void dot4(const __nv_bfloat16 *const rows[4], int K, const float *xs,
                                     int xs_ld, float (&acc)[4][TB], int lane)
{
    const int nch = K / 8;
    int c = lane;
    for (; c + 32 * (kBatch - 1) < nch; c += 32 * kBatch) {
        uint4 w[kBatch][4];
#pragma unroll
        for (int b = 0; b < kBatch; b++)
#pragma unroll
            for (int r = 0; r < 4; r++) w[b][r] = ld_stream(rows[r] + (size_t)(c + 32 * b) * 8);
#pragma unroll
        for (int b = 0; b < kBatch; b++)
#pragma unroll
            for (int t = 0; t < TB; t++)
#pragma unroll
                for (int r = 0; r < 4; r++)
                    fma8<TB>(w[b][r], xs + t * xs_ld + (c + 32 * b) * 8, acc[r][t]);
    }
    for (; c < nch; c += 32) {
        uint4 w[4];
#pragma unroll
        for (int r = 0; r < 4; r++) w[r] = ld_stream(rows[r] + (size_t)c * 8);
#pragma unroll
        for (int t = 0; t < TB; t++)
#pragma unroll
            for (int r = 0; r < 4; r++) fma8<TB>(w[r], xs + t * xs_ld + c * 8, acc[r][t]);
    }
}

template <int TB>
__device__ __forceinline__ void reduce4(float (&acc)[4][TB])
{
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int t = 0; t < TB; t++) acc[r][t] = warp_sum(acc[r][t]);
}

struct DenseXArgs {
    const __nv_bfloat16 *x;
    int T, H;
    const __nv_bfloat16 *router_w;
    int E;
    float *logits;        // [T, E]
    const __nv_bfloat16 *down_w;
    int L;
    float *z;             // [T, L]
    const __nv_bfloat16 *sh_w1, *sh_w3;
    int S;
    float *shared_out;    // cat + L, row pitch cat_ld
    int cat_ld;
    float b1, b2;
    int u_begin, u_end;   // unit range of this launch: router, then down, then shared pairs
    int wait;             // wait for the previous kernel (0: the launch reads only x)
};

constexpr int kGemvWarps = 8;
constexpr size_t kGemvSmemMax = 227 * 1024;
constexpr int kStageUnroll = 8;   // staging loads in flight per thread

template <int TB>
__global__ void __launch_bounds__(kGemvWarps * 32) k_dense_x(DenseXArgs a)
{
    extern __shared__ float xs[];   // [TB][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    if (a.wait) pdl_wait();
    const int nA = (a.E + 3) / 4, nB = a.L / 4;
    for (int t0 = 0; t0 < a.T; t0 += TB) {
        const int tb = min(TB, a.T - t0);
        // stage x as fp32: 16-byte loads, all issued before any is used
        const uint4 *xsrc = reinterpret_cast<const uint4 *>(a.x + (size_t)t0 * a.H);
        const int nv = TB * a.H / 8;
        for (int i0 = threadIdx.x; i0 < nv; i0 += kStageUnroll * blockDim.x) {
            uint4 v[kStageUnroll];
#pragma unroll
            for (int j = 0; j < kStageUnroll; j++) {
                const int i = i0 + j * blockDim.x;
                v[j] = (i < nv && (8 * i) / a.H < tb) ? xsrc[i] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < kStageUnroll; j++) {
                const int i = i0 + j * blockDim.x;
                if (i < nv) {
                    float4 *d = reinterpret_cast<float4 *>(xs + 8 * i);
                    d[0] = make_float4(bf16lo(v[j].x), bf16hi(v[j].x), bf16lo(v[j].y), bf16hi(v[j].y));
                    d[1] = make_float4(bf16lo(v[j].z), bf16hi(v[j].z), bf16lo(v[j].w), bf16hi(v[j].w));
                }
            }
        }
        __syncthreads();
        for (int u = a.u_begin + blockIdx.x * kGemvWarps + warp; u < a.u_end;
             u += gridDim.x * kGemvWarps) {
            const __nv_bfloat16 *rows[4];
            float acc[4][TB];
#pragma unroll
            for (int r = 0; r < 4; r++)
#pragma unroll
                for (int t = 0; t < TB; t++) acc[r][t] = 0.f;
            if (u < nA) {
                const int e0 = 4 * u;
#pragma unroll
                for (int r = 0; r < 4; r++)
                    rows[r] = a.router_w + (size_t)min(e0 + r, a.E - 1) * a.H;
            } else if (u < nA + nB) {
                const int l0 = 4 * (u - nA);
#pragma unroll
                for (int r = 0; r < 4; r++) rows[r] = a.down_w + (size_t)(l0 + r) * a.H;
            } else {
                const int s0 = 2 * (u - nA - nB);
                rows[0] = a.sh_w1 + (size_t)s0 * a.H;
                rows[1] = a.sh_w1 + (size_t)(s0 + 1) * a.H;
                rows[2] = a.sh_w3 + (size_t)s0 * a.H;
                rows[3] = a.sh_w3 + (size_t)(s0 + 1) * a.H;
            }
            dot4<TB>(rows, a.H, xs, a.H, acc, lane);
            reduce4<TB>(acc);
            if (lane == 0) {
                for (int t = 0; t < tb; t++) {
                    const size_t tt = (size_t)(t0 + t);
                    if (u < nA) {
                        for (int r = 0; r < 4; r++)
                            if (4 * u + r < a.E) a.logits[tt * a.E + 4 * u + r] = acc[r][t];
                    } else if (u < nA + nB) {
                        const int l0 = 4 * (u - nA);
                        for (int r = 0; r < 4; r++) a.z[tt * a.L + l0 + r] = acc[r][t];
                    } else {
                        const int s0 = 2 * (u - nA - nB);
                        for (int q = 0; q < 2; q++)
                            a.shared_out[tt * a.cat_ld + s0 + q] =
                                situ_f(acc[q][t], acc[2 + q][t], a.b1, a.b2);
                    }
                }
            }
        }
        __syncthreads();
    }
    // Without the dependency wait at the start, wait before exiting: the next
    // kernel waits only for this one, whose completion must imply that of
    // every earlier kernel of the forward.
    if (!a.wait && threadIdx.x == 0) pdl_wait();
}

struct UpArgs {
    const float *cat;     // [T, L+S]; the shared-expert part cat[:, L:] is read
    const float *acc;     // [T, L] weighted sum of the routed experts
    const __nv_bfloat16 *gain;   // [L] latent norm gain, or null for no norm
    float eps;
    int T, L, S, H;
    const __nv_bfloat16 *up_w;    // [H, L]
    const __nv_bfloat16 *sh_w2;   // [H, S]
    __nv_bfloat16 *y;             // [T, H]
};

// The activations of k_up are [RMSNorm(acc) * gain | shared SiTU]: each block
// normalises the aggregate of its own tokens while staging it (README
// section 9, k3_moe step 4: the norm is taken on the aggregate).
template <int TB>
__global__ void __launch_bounds__(kGemvWarps * 32) k_up(UpArgs a)
{
    extern __shared__ float xs[];   // [TB][L+S]
    __shared__ float red[TB][kGemvWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.L + a.S;
    const int nunits = a.H / 4;
    pdl_launch_dependents();
    pdl_wait();
    for (int t0 = 0; t0 < a.T; t0 += TB) {
        const int tb = min(TB, a.T - t0);
        float ss[TB];
#pragma unroll
        for (int t = 0; t < TB; t++) {
            ss[t] = 0.f;
            // row t of the activations: [acc (L) | shared SiTU (S)], 16-byte loads
            // issued kStageUnroll at a time before any is used
            const float *src_a = a.acc + (size_t)(t0 + t) * a.L;
            const float *src_s = a.cat + (size_t)(t0 + t) * K + a.L;
            float4 *dst = reinterpret_cast<float4 *>(xs + t * K);
            const int nv = K / 4, nl = a.L / 4;
            for (int i0 = threadIdx.x; i0 < nv; i0 += kStageUnroll * blockDim.x) {
                float4 v[kStageUnroll];
#pragma unroll
                for (int j = 0; j < kStageUnroll; j++) {
                    const int i = i0 + j * blockDim.x;
                    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (i < nv && t < tb)
                        v[j] = i < nl ? reinterpret_cast<const float4 *>(src_a)[i]
                                      : reinterpret_cast<const float4 *>(src_s)[i - nl];
                }
#pragma unroll
                for (int j = 0; j < kStageUnroll; j++) {
                    const int i = i0 + j * blockDim.x;
                    if (i < nv) {
                        if (i < nl) ss[t] += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
                        dst[i] = v[j];
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TB; t++) {
            ss[t] = warp_sum(ss[t]);
            if (lane == 0) red[t][warp] = ss[t];
        }
        __syncthreads();
        if (a.gain) {
#pragma unroll
            for (int t = 0; t < TB; t++) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < kGemvWarps; w++) tot += red[t][w];
                const float inv = 1.0f / sqrtf(tot / (float)a.L + a.eps);
                for (int i = threadIdx.x; i < a.L; i += blockDim.x)
                    xs[t * K + i] *= inv * __bfloat162float(a.gain[i]);
            }
            __syncthreads();
        }
        for (int u = blockIdx.x * kGemvWarps + warp; u < nunits; u += gridDim.x * kGemvWarps) {
            const int o0 = 4 * u;
            float acc[4][TB];
#pragma unroll
            for (int r = 0; r < 4; r++)
#pragma unroll
                for (int t = 0; t < TB; t++) acc[r][t] = 0.f;
            const __nv_bfloat16 *rows[4];
#pragma unroll
            for (int r = 0; r < 4; r++) rows[r] = a.up_w + (size_t)(o0 + r) * a.L;
            dot4<TB>(rows, a.L, xs, K, acc, lane);
#pragma unroll
            for (int r = 0; r < 4; r++) rows[r] = a.sh_w2 + (size_t)(o0 + r) * a.S;
            dot4<TB>(rows, a.S, xs + a.L, K, acc, lane);
            reduce4<TB>(acc);
            if (lane == 0) {
                for (int t = 0; t < tb; t++)
                    for (int r = 0; r < 4; r++)
                        a.y[(size_t)(t0 + t) * a.H + o0 + r] = __float2bfloat16_rn(acc[r][t]);
            }
        }
        __syncthreads();
    }
}

template <typename Kern>
static int grid_for(const k3moe &h, Kern kern, size_t smem, int units)
{
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvWarps * 32, smem);
    if (per_sm < 1) per_sm = 1;
    const int want = (units + kGemvWarps - 1) / kGemvWarps;
    return want < h.sm_count * per_sm ? want : h.sm_count * per_sm;
}

template <int TB>
static cudaError_t init_tb(k3moe &h, int slot)
{
    const k3moe_config &c = h.cfg;
    const size_t sx = (size_t)TB * c.hidden * sizeof(float);
    const size_t su = (size_t)TB * (c.latent + c.shared_inter) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_dense_x<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sx);
    if (e != cudaSuccess) return e;
    h.grid_dense[slot] = grid_for(h, k_dense_x<TB>, sx, 1 << 30);   // resident-block cap
    // k_up stages TB rows of L+S floats: a wide dense feed-forward layer does
    // not fit (it never runs k_up); grid 0 marks the width unusable
    h.grid_up[slot] = 0;
    if (su <= kGemvSmemMax) {
        e = cudaFuncSetAttribute(k_up<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)su);
        if (e != cudaSuccess) return e;
        h.grid_up[slot] = grid_for(h, k_up<TB>, su, c.hidden / 4);
    }
    return cudaGetLastError();
}

cudaError_t init_dense_kernels(k3moe &h)
{
    cudaError_t e = init_tb<1>(h, 0);
    if (e == cudaSuccess) e = init_tb<2>(h, 1);
    if (e == cudaSuccess) e = init_tb<4>(h, 2);
    return e;
}

template <int TB>
static cudaError_t run_dense_x(const k3moe &h, const DenseXArgs &a, int slot, cudaStream_t s)
{
    const size_t smem = (size_t)TB * a.H * sizeof(float);
    const int want = (a.u_end - a.u_begin + kGemvWarps - 1) / kGemvWarps;
    const int grid = want < h.grid_dense[slot] ? want : h.grid_dense[slot];
    // router+down opens the layer in plain stream order; the shared gate/up
    // alone (u_begin > 0) reads only x and needs no wait
    if (a.u_begin == 0) return launch_ordered(k_dense_x<TB>, grid, kGemvWarps * 32, smem, s, a);
    return launch_pdl(k_dense_x<TB>, grid, kGemvWarps * 32, smem, s, a);
}

cudaError_t launch_dense_x(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x, int T,
                           cudaStream_t s, int part, bool wait_x)
{
    const k3moe_config &c = h.cfg;
    DenseXArgs a;
    a.x = x;
    a.T = T;
    a.H = c.hidden;
    a.router_w = w.router_w;
    a.E = c.n_experts;
    a.logits = h.ws.logits;
    a.down_w = w.down_w;
    a.L = c.latent;
    a.z = h.ws.z;
    a.sh_w1 = w.sh_w1;
    a.sh_w3 = w.sh_w3;
    a.S = c.shared_inter;
    a.cat_ld = c.latent + c.shared_inter;
    a.shared_out = h.ws.cat + c.latent;
    a.b1 = c.situ_b1;
    a.b2 = c.situ_b2;
    const int nAB = (c.n_experts + 3) / 4 + c.latent / 4, nC = c.shared_inter / 2;
    a.u_begin = part == 1 ? nAB : 0;
    a.u_end = part == 0 ? nAB : nAB + nC;
    a.wait = part != 1 || wait_x;
    if (T == 1) return run_dense_x<1>(h, a, 0, s);
    if (T == 2) return run_dense_x<2>(h, a, 1, s);
    return run_dense_x<4>(h, a, 2, s);
}

template <int TB>
static cudaError_t run_up(const k3moe &h, const UpArgs &a, int slot, cudaStream_t s)
{
    if (h.grid_up[slot] == 0) return cudaErrorInvalidValue;
    const size_t smem = (size_t)TB * (a.L + a.S) * sizeof(float);
    return launch_pdl(k_up<TB>, h.grid_up[slot], kGemvWarps * 32, smem, s, a);
}

cudaError_t launch_up(const k3moe &h, const LayerDev &w, __nv_bfloat16 *y, int T, cudaStream_t s)
{
    const k3moe_config &c = h.cfg;
    UpArgs a;
    a.cat = h.ws.cat;
    a.acc = h.ws.acc;
    a.gain = c.latent_norm ? w.gain : nullptr;
    a.eps = c.rms_eps;
    a.T = T;
    a.L = c.latent;
    a.S = c.shared_inter;
    a.H = c.hidden;
    a.up_w = w.up_w;
    a.sh_w2 = w.sh_w2;
    a.y = y;
    if (T == 1) return run_up<1>(h, a, 0, s);
    if (T == 2) return run_up<2>(h, a, 1, s);
    return run_up<4>(h, a, 2, s);
}

}  // namespace k3
