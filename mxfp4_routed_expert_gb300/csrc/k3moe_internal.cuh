// Internal declarations of libk3moe: the handle, device buffers, kernel
// launchers and small device helpers shared by the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/k3moe.h"

namespace k3 {

constexpr int kGroup = 32;          // MXFP4 columns per ue8m0 scale
constexpr int kMaxExperts = 1024;   // router select keeps 32 scores per lane
constexpr int kMaxTopk = 32;

// Device error codes latched in Workspace::err (first one wins).
enum : int { kErrNone = 0, kErrBounds = 1, kErrTimeout = 2 };

struct LayerDev {
    bool loaded = false;
    void *block = nullptr;   // single allocation holding every tensor below
    size_t bytes = 0;
    const __nv_bfloat16 *router_w = nullptr;   // [E, H]
    const float *bias = nullptr;               // [E] (zeros when the caller gave none)
    const __nv_bfloat16 *down_w = nullptr;     // [L, H]
    const __nv_bfloat16 *up_w = nullptr;       // [H, L]
    const __nv_bfloat16 *gain = nullptr;       // [L] or nullptr
    const __nv_bfloat16 *sh_w1 = nullptr;      // [S, H]
    const __nv_bfloat16 *sh_w3 = nullptr;      // [S, H]
    const __nv_bfloat16 *sh_w2 = nullptr;      // [H, S]
    const uint8_t *w1p = nullptr, *w1s = nullptr;   // [E][I][L/2], [E][I][L/32]
    const uint8_t *w3p = nullptr, *w3s = nullptr;
    const uint8_t *w2p = nullptr, *w2s = nullptr;   // [E][L][I/2], [E][L][I/32]
};

// Per-handle scratch, sized for max_tokens (Tm).
struct Workspace {
    void *block = nullptr;
    size_t bytes = 0;
    float *logits = nullptr;      // [Tm, E]
    float *z = nullptr;           // [Tm, L]   latent (fp32, from the down projection)
    __half *z16 = nullptr;        // [Tm, L]   z * 2^-zexp[t] in fp16 (expert GEMV input)
    int *zexp = nullptr;          // [Tm]
    float *cat = nullptr;         // [Tm, L+S] normalised latent | shared SiTU
    int *ids = nullptr;           // [Tm, k]
    float *wts = nullptr;         // [Tm, k]
    int *counts = nullptr;        // [E]
    int *offsets = nullptr;       // [E+1]
    int *perm = nullptr;          // [Tm*k]
    int *touched = nullptr;       // [E]  experts with at least one token, ascending
    int *n_touched = nullptr;     // [1]
    __half *h16 = nullptr;        // [Tm*k, I] SiTU output per (token, expert) pair, perm order
    float *acc = nullptr;         // [Tm, L]
    __nv_bfloat16 *xbuf0 = nullptr;   // [Tm, H] staging (host forward, chain)
    __nv_bfloat16 *xbuf1 = nullptr;   // [Tm, H]
    int *err = nullptr;           // [4] device error word + detail
};

struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
};

}  // namespace k3

struct k3moe {
    k3moe_config cfg;
    int sm_count = 0;
    std::vector<k3::LayerDev> layers;
    k3::Workspace ws;
    int last_T = 0;
    bool profiling = false;
    std::vector<k3::ProfRec> prof;
    std::vector<cudaEvent_t> event_pool;
    int err_sticky = 0;
};

namespace k3 {

// ---- launchers (each returns cudaGetLastError()) -----------------------------
cudaError_t launch_dense_x(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x, int T,
                           cudaStream_t s);
cudaError_t launch_route(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_perm(const k3moe &h, int T, cudaStream_t s);
cudaError_t launch_expert_w13(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_expert_w2(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_latent_norm(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_up(const k3moe &h, const LayerDev &w, __nv_bfloat16 *y, int T,
                      cudaStream_t s);
cudaError_t launch_chain_glue(const k3moe &h, const __nv_bfloat16 *y, __nv_bfloat16 *x_next,
                              int T, cudaStream_t s);
cudaError_t launch_scale_scan(const uint8_t *p, size_t n, int *flag, cudaStream_t s);

// ---- device helpers -----------------------------------------------------------
__device__ __forceinline__ void set_err(int *err, int code, int detail)
{
    if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// 16-byte streaming load: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two e2m1 values in one byte -> f16x2 (low nibble -> low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(r)
        : "r"(byte));
    return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float f16x2_sum(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    return __low2float(h) + __high2float(h);
}

// 2^(s-127) for a ue8m0 byte s in [0, 254] (s = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s)
{
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + expf(-v)); }

__device__ __forceinline__ float situ_f(float g, float u, float b1, float b2)
{
    return (b1 * tanhf(g / b1)) * sigmoid_f(g) * (b2 * tanhf(u / b2));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace k3
