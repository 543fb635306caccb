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
__device__ __forceinline__ void dot4(const __nv_bfloat16 *const rows[4], int K, const float *xs,
                                     int xs_ld, float (&acc)[4][TB], int lane)
{
    const int nch = K / 8;
#pragma unroll 4
    for (int c = lane; c < nch; c += 32) {
        uint4 w[4];
#pragma unroll
        for (int r = 0; r < 4; r++) w[r] = ld_stream(rows[r] + (size_t)c * 8);
#pragma unroll
        for (int t = 0; t < TB; t++) {
            const float4 xa = *reinterpret_cast<const float4 *>(xs + t * xs_ld + c * 8);
            const float4 xb = *reinterpret_cast<const float4 *>(xs + t * xs_ld + c * 8 + 4);
#pragma unroll
            for (int r = 0; r < 4; r++) {
                float a = acc[r][t];
                a = fmaf(bf16lo(w[r].x), xa.x, a);
                a = fmaf(bf16hi(w[r].x), xa.y, a);
                a = fmaf(bf16lo(w[r].y), xa.z, a);
                a = fmaf(bf16hi(w[r].y), xa.w, a);
                a = fmaf(bf16lo(w[r].z), xb.x, a);
                a = fmaf(bf16hi(w[r].z), xb.y, a);
                a = fmaf(bf16lo(w[r].w), xb.z, a);
                a = fmaf(bf16hi(w[r].w), xb.w, a);
                acc[r][t] = a;
            }
        }
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
};

constexpr int kGemvWarps = 8;

template <int TB>
__global__ void __launch_bounds__(kGemvWarps * 32) k_dense_x(DenseXArgs a)
{
    extern __shared__ float xs[];   // [TB][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nA = (a.E + 3) / 4, nB = a.L / 4, nC = a.S / 2;
    const int nunits = nA + nB + nC;
    for (int t0 = 0; t0 < a.T; t0 += TB) {
        const int tb = min(TB, a.T - t0);
        const uint32_t *xsrc = reinterpret_cast<const uint32_t *>(a.x + (size_t)t0 * a.H);
        for (int i = threadIdx.x; i < TB * a.H / 2; i += blockDim.x) {
            const int t = (2 * i) / a.H;
            const uint32_t v = (t < tb) ? xsrc[i] : 0u;
            xs[2 * i] = bf16lo(v);
            xs[2 * i + 1] = bf16hi(v);
        }
        __syncthreads();
        for (int u = blockIdx.x * kGemvWarps + warp; u < nunits; u += gridDim.x * kGemvWarps) {
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
}

struct UpArgs {
    const float *cat;     // [T, L+S]
    int T, L, S, H;
    const __nv_bfloat16 *up_w;    // [H, L]
    const __nv_bfloat16 *sh_w2;   // [H, S]
    __nv_bfloat16 *y;             // [T, H]
};

template <int TB>
__global__ void __launch_bounds__(kGemvWarps * 32) k_up(UpArgs a)
{
    extern __shared__ float xs[];   // [TB][L+S]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.L + a.S;
    const int nunits = a.H / 4;
    for (int t0 = 0; t0 < a.T; t0 += TB) {
        const int tb = min(TB, a.T - t0);
        const float4 *src = reinterpret_cast<const float4 *>(a.cat + (size_t)t0 * K);
        float4 *dst = reinterpret_cast<float4 *>(xs);
        for (int i = threadIdx.x; i < TB * K / 4; i += blockDim.x) {
            const int t = (4 * i) / K;
            dst[i] = (t < tb) ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
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
static cudaError_t run_dense_x(const k3moe &h, const DenseXArgs &a, cudaStream_t s)
{
    const size_t smem = (size_t)TB * a.H * sizeof(float);
    cudaFuncSetAttribute(k_dense_x<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const int units = (a.E + 3) / 4 + a.L / 4 + a.S / 2;
    const int grid = grid_for(h, k_dense_x<TB>, smem, units);
    k_dense_x<TB><<<grid, kGemvWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_dense_x(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x, int T,
                           cudaStream_t s)
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
    if (T == 1) return run_dense_x<1>(h, a, s);
    if (T == 2) return run_dense_x<2>(h, a, s);
    return run_dense_x<4>(h, a, s);
}

template <int TB>
static cudaError_t run_up(const k3moe &h, const UpArgs &a, cudaStream_t s)
{
    const size_t smem = (size_t)TB * (a.L + a.S) * sizeof(float);
    cudaFuncSetAttribute(k_up<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const int grid = grid_for(h, k_up<TB>, smem, a.H / 4);
    k_up<TB><<<grid, kGemvWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_up(const k3moe &h, const LayerDev &w, __nv_bfloat16 *y, int T, cudaStream_t s)
{
    const k3moe_config &c = h.cfg;
    UpArgs a;
    a.cat = h.ws.cat;
    a.T = T;
    a.L = c.latent;
    a.S = c.shared_inter;
    a.H = c.hidden;
    a.up_w = w.up_w;
    a.sh_w2 = w.sh_w2;
    a.y = y;
    if (T == 1) return run_up<1>(h, a, s);
    if (T == 2) return run_up<2>(h, a, s);
    return run_up<4>(h, a, s);
}

}  // namespace k3
