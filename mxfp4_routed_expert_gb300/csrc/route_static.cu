// k3moe_route_static: the router step on its own, for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs where it may not call cudaMalloc -- for
// instance a plugin inside a host framework that owns all device memory
// through its own pool, or a serving loop that forbids allocation after
// start-up so that its memory use stays fixed. Such a caller can hand in
// its inputs and output buffers but cannot give the library a workspace.
//
// The router's only scratch is the [T, E] table of fp32 logits. Here it
// lives in one file-scope device array of fixed size, created when the
// library is loaded and kept by every GPU that loads it until the process
// exits. Host code may not use the array's name as a device address (in host
// code it names a host-side stand-in), so the first call on each device looks
// the address up with cudaGetSymbolAddress while that device is current and
// caches it for the life of the process (the cache does not follow a
// cudaDeviceReset, after which the array may sit elsewhere: call no further
// k3moe_route_static on a device after resetting it). Every call shares the
// array: two calls that overlap on the GPU
// (on different streams, or on different host threads) overwrite each
// other's logits. Each call writes every logit it later reads, so nothing in
// the array has to start at zero.
//
// The arithmetic is the router of the layer (kimi-k3-in-c README, Part II
// section 9, k3_router): logit = x . Wr_e, sc = sigmoid(logit),
// ch = sc + bias_e picks the top k (equal ch: lower expert id first), and the
// weights are the picked sc, renormalised when renorm is set, times
// routed_scale.
#include <climits>
#include <cmath>
#include <mutex>

#include "k3moe_internal.cuh"

namespace {

static __device__ __align__(256) float g_route_logits[K3MOE_ROUTE_STATIC_MAX_LOGITS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_logits_addr[kMaxDevices] = {};

// Device address of g_route_logits on the current device (looked up once).
int static_logits(float **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return K3MOE_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_logits_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_logits) != cudaSuccess || !p) {
            cudaGetLastError();
            return K3MOE_ERR_CUDA;
        }
        g_logits_addr[dev] = static_cast<float *>(p);
    }
    *out = g_logits_addr[dev];
    return K3MOE_OK;
}

// One warp per (token, expert) dot product over 16-byte chunks of x and Wr.
__global__ void __launch_bounds__(256) k_static_logits(const __nv_bfloat16 *x,
                                                       const __nv_bfloat16 *W, float *logits,
                                                       int T, int H, int E)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long id = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         id < (long long)T * E; id += warps) {
        const int t = (int)(id / E), e = (int)(id % E);
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)e * H);
        float acc = 0.f;
        for (int c = lane; c < H / 8; c += 32) {
            const uint4 a = xr[c], b = k3::ld_stream(wr + c);
            acc = fmaf(k3::bf16lo(a.x), k3::bf16lo(b.x), acc);
            acc = fmaf(k3::bf16hi(a.x), k3::bf16hi(b.x), acc);
            acc = fmaf(k3::bf16lo(a.y), k3::bf16lo(b.y), acc);
            acc = fmaf(k3::bf16hi(a.y), k3::bf16hi(b.y), acc);
            acc = fmaf(k3::bf16lo(a.z), k3::bf16lo(b.z), acc);
            acc = fmaf(k3::bf16hi(a.z), k3::bf16hi(b.z), acc);
            acc = fmaf(k3::bf16lo(a.w), k3::bf16lo(b.w), acc);
            acc = fmaf(k3::bf16hi(a.w), k3::bf16hi(b.w), acc);
        }
        acc = k3::warp_sum(acc);
        if (lane == 0) logits[id] = acc;
    }
}

// One warp per token: k rounds of a warp arg-max over the biased scores.
__global__ void __launch_bounds__(32) k_static_topk(const float *logits, const float *bias,
                                                    int E, int k, int renorm, float routed_scale,
                                                    int *ids, float *w)
{
    const int t = blockIdx.x, lane = threadIdx.x;
    constexpr int kPer = k3::kMaxExperts / 32;
    float ch[kPer], sc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int e = lane + 32 * i;
        sc[i] = e < E ? k3::sigmoid_f(logits[(size_t)t * E + e]) : 0.f;
        ch[i] = e < E ? sc[i] + (bias ? bias[e] : 0.f) : 0.f;
        // a NaN score (from a NaN or infinite input) ranks below every number, so
        // that the comparisons below stay a total order and all lanes agree on
        // every pick
        if (isnan(ch[i])) ch[i] = -INFINITY;
    }
    uint32_t taken = 0u;
    float wsum = 0.f, wsel = 0.f;
    int esel = 0;
    for (int j = 0; j < k; j++) {
        float bv = 0.f, bs = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (be == INT_MAX || ch[i] > bv)) {
                bv = ch[i];
                bs = sc[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                bs = os;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        wsum += bs;
        if (lane == j) {
            esel = be;
            wsel = bs;
        }
    }
    if (lane < k) {
        const float v = (renorm && wsum > 0.f) ? wsel / wsum : wsel;
        ids[(size_t)t * k + lane] = esel;
        w[(size_t)t * k + lane] = v * routed_scale;
    }
}

}  // namespace

extern "C" int k3moe_route_static(const void *x, const void *router_w, const float *router_bias,
                                  int T, int hidden, int n_experts, int topk, int renorm,
                                  float routed_scale, int32_t *ids, float *w, void *stream)
{
    if (!x || !router_w || !ids || !w) return K3MOE_ERR_INVALID_ARG;
    if (T < 1 || hidden < 8 || hidden % 8 || n_experts < 1) return K3MOE_ERR_INVALID_ARG;
    // the dot products read x and Wr in 16-byte chunks
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(router_w)) % 16 != 0)
        return K3MOE_ERR_INVALID_ARG;
    if ((renorm != 0 && renorm != 1) || !std::isfinite(routed_scale) || routed_scale <= 0.f)
        return K3MOE_ERR_CONFIG;
    if (topk < 1 || topk > k3::kMaxTopk || topk > n_experts || n_experts > k3::kMaxExperts)
        return K3MOE_ERR_SHAPE;
    if ((unsigned long long)T * (unsigned long long)n_experts > K3MOE_ROUTE_STATIC_MAX_LOGITS)
        return K3MOE_ERR_SHAPE;   // the logits would not fit the static scratch array
    float *logits = nullptr;
    const int rc = static_logits(&logits);
    if (rc != K3MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = (long long)T * n_experts;
    const int grid = (int)((rows + 7) / 8 < 4096 ? (rows + 7) / 8 : 4096);
    // each launch's own error is taken right after it (a launch error is not sticky)
    k_static_logits<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(x),
                                         static_cast<const __nv_bfloat16 *>(router_w), logits, T,
                                         hidden, n_experts);
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ERR_CUDA;
    k_static_topk<<<T, 32, 0, s>>>(logits, router_bias, n_experts, topk, renorm, routed_scale, ids,
                                   w);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}
