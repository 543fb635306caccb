// The glue between stacked layers, the RMSNorm in front of the MoE and the
// load-time scale-byte check.
//
// RMSNorm: out = x / sqrt(mean(x^2) + eps) * gain, eps inside the square root
// (kimi-k3-in-c README, Part II section 5, k3_rmsnorm).
#include "k3moe_internal.cuh"

namespace k3 {

__device__ __forceinline__ float block_sum_256(float v, float *red)
{
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; w++) s += red[w];
    __syncthreads();
    return s;
}

// x_next[t] = bf16(y[t] / sqrt(mean(y[t]^2) + eps)), unit gain.
__global__ void __launch_bounds__(256) k_chain_glue(const __nv_bfloat16 *y, __nv_bfloat16 *xn,
                                                    int H, float eps)
{
    __shared__ float red[8];
    const int t = blockIdx.x;
    const __nv_bfloat16 *a = y + (size_t)t * H;
    pdl_launch_dependents();
    pdl_wait();
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const float v = __bfloat162float(a[i]);
        ss = fmaf(v, v, ss);
    }
    ss = block_sum_256(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x)
        xn[(size_t)t * H + i] = __float2bfloat16_rn(__bfloat162float(a[i]) * inv);
}

cudaError_t launch_chain_glue(const k3moe &h, const __nv_bfloat16 *y, __nv_bfloat16 *x_next,
                              int T, cudaStream_t s)
{
    return launch_pdl(k_chain_glue, T, 256, 0, s, y, x_next, h.cfg.hidden, h.cfg.rms_eps);
}

// x[t] = bf16(h[t] * inv * g), inv = (float)(1 / sqrt(mean(h[t]^2) + eps)): the
// post-attention RMSNorm that feeds the MoE (the decoder layer's post_norm in
// front of k3_moe, kimi-k3-in-c README, Part II; k3_rmsnorm of section 5 sums
// the squares in double and forms inv in double). Each thread sums its
// squares in fp32 and the partial sums meet in double (fp64 is slow here).
__global__ void __launch_bounds__(256) k_residual_norm(const float *hin, const __nv_bfloat16 *g,
                                                       __nv_bfloat16 *x, int H, float eps)
{
    __shared__ double red[8];
    __shared__ float inv_s;
    const int t = blockIdx.x;
    const float *a = hin + (size_t)t * H;
    pdl_launch_dependents();
    const double ss = warp_sum_d((double)residual_sumsq<8>(a, H / 4, threadIdx.x, blockDim.x));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {   // one thread: the double divide and root are slow here
        double tot = 0.0;
#pragma unroll
        for (int w = 0; w < 8; w++) tot += red[w];
        inv_s = (float)(1.0 / sqrt(tot / (double)H + (double)eps));
    }
    __syncthreads();
    residual_write<8>(a, g, inv_s, x + (size_t)t * H, nullptr, H / 4, threadIdx.x, blockDim.x);
}

cudaError_t launch_residual_norm(const k3moe &h, const float *hin, const __nv_bfloat16 *gain, int T,
                                 cudaStream_t s)
{
    // the layer's first kernel: plain stream order, like every layer's first
    return launch_ordered(k_residual_norm, T, 256, 0, s, hin, gain, h.ws.xn, h.cfg.hidden,
                          h.cfg.rms_eps);
}

// flag[0] += number of bytes equal to 255 in p[0, n).
__global__ void k_scale_scan(const uint8_t *p, size_t n, int *flag)
{
    int found = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        found += (p[i] == 255u);
    found = __syncthreads_count(found > 0);
    if (threadIdx.x == 0 && found) atomicAdd(flag, found);
}

cudaError_t launch_scale_scan(const uint8_t *p, size_t n, int *flag, cudaStream_t s)
{
    k_scale_scan<<<1024, 256, 0, s>>>(p, n, flag);
    return cudaGetLastError();
}

}  // namespace k3
