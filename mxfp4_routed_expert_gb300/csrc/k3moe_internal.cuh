// Internal declarations of libk3moe: the handle, device buffers, kernel
// launchers and small device helpers shared by the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <deque>
#include <string>
#include <vector>

#include "../../include/k3moe.h"

namespace k3 {

constexpr int kGroup = 32;          // MXFP4 columns per ue8m0 scale
constexpr int kMaxExperts = 1024;   // router select keeps 32 scores per lane
constexpr int kMaxTopk = 32;
constexpr int kMaxLayers = 1024;     // per handle (the model has 93)
constexpr int kZPad = 16;           // fp16 padding after each z16 row (holds its exponent)
constexpr int kSplitTokensMax = 128;  // tensor-core GEMMs split K only up to this many tokens
constexpr int kGemmMinTokens = 16;    // tensor-core dense GEMMs from this many tokens on

// A configuration with n_experts = topk = latent = moe_inter = 0 is a dense
// feed-forward layer (the model's layer 0): y = W2 . SiTU(W1 x, W3 x) with
// the shared-expert weights and width shared_inter.
inline bool is_dense(const k3moe_config &c) { return c.n_experts == 0; }

// Device error codes latched in Workspace::err (first one wins).
enum : int { kErrNone = 0, kErrBounds = 1, kErrTimeout = 2 };

struct LayerDev {
    bool loaded = false;
    int index = -1;          // layer index in the handle
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
    // largest scale byte of each expert row (tensor-core expert GEMM operand rebasing)
    const uint8_t *w1max = nullptr, *w3max = nullptr;   // [E][I]
    const uint8_t *w2max = nullptr;                     // [E][L]
    // row tensor maps of the dense decode GEMVs (router+down, shared gate/up,
    // up+shared down; six each), built once at load
    CUtensorMap dense_maps[3][6];
    bool dense_maps_ok = false;
    // Expert arrays above hold n_wslots experts; expert e sits at index
    // wslot[e] (expert tier: a slot of the handle's device pool) or at e
    // (wslot == nullptr: the layer's own copy of all experts).
    const int *wslot = nullptr;
    int n_wslots = 0;
    // expert tier: the layer's routed experts in one pinned, device-mapped
    // host block, the nine expert arrays in the layout of the device copy
    void *host_block = nullptr;
    const uint8_t *hsrc[9] = {};
    bool pinned = false;     // k3moe_tier_pin_layer: its experts hold pinned slots
    // RMSNorm gain in front of the MoE (k3moe_load_post_norm), own allocation
    const __nv_bfloat16 *post_gain = nullptr;
    void *post_block = nullptr;
};

// Expert tier (k3moe_set_expert_tier): device slots caching routed experts
// whose home is pinned host memory.
constexpr int kTierPieces = 9;          // w1p w1s w3p w3s w2p w2s w1max w3max w2max
constexpr int kTierMaxSlots = 16384;
// Stamps are 32-bit and 0xFFFFFFFF marks a pinned slot: once the counter
// reaches kTierRebaseAt, the slots' stamps are shifted down so that the last
// kTierRebaseKeep stamps keep their order (older ones tie at 1).
constexpr uint32_t kTierRebaseAt = 0x80000000u;
constexpr uint32_t kTierRebaseKeep = 1u << 24;
// Every buffer the kernels write is followed by a band of kGuardBytes bytes
// set to kGuardByte; k3moe_sync_status reports a changed band.
constexpr size_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;

struct TierDev {
    int slots = 0;
    void *block = nullptr;              // device: slot arrays, then the tables
    uint8_t *arr[kTierPieces] = {};     // [slots][piece size]
    size_t piece[kTierPieces] = {};     // bytes of one expert's piece
    size_t expert_bytes = 0;
    int *slot_of = nullptr;             // [max_layers][E]: slot or -1
    int *slot_key = nullptr;            // [slots]: layer * E + expert, or -1 (free)
    uint32_t *slot_used = nullptr;      // [slots]: stamp of the last forward that used it
    int2 *fill = nullptr;               // [E]: (slot, expert) per miss of the current forward
    int *n_fill = nullptr;
    unsigned long long *stats = nullptr;   // hits, misses, bytes filled
    int *all_ids = nullptr;             // [E + 1]: 0 .. E-1, then E (a layer's list, for pinning)
    std::vector<size_t> guards;         // guard bands after each array of the block
    uint32_t stamp = 0;                 // last stamp given to a forward
    uint32_t rebase_at = kTierRebaseAt;
    uint32_t rebase_keep = kTierRebaseKeep;
    int pinned = 0;                     // slots held by pinned layers
};

// Per-handle scratch, sized for max_tokens (Tm).
struct Workspace {
    void *block = nullptr;
    size_t bytes = 0;
    float *logits = nullptr;      // [Tm, E]
    float *z = nullptr;           // [Tm, L]   latent (fp32, from the down projection)
    __half *z16 = nullptr;        // [Tm, L + kZPad]: z * 2^-e in fp16, then e as an int32
                                  //   in the row's padding (expert GEMV input)
    float *cat = nullptr;         // [Tm, L+S] normalised latent | shared SiTU
    int *ids = nullptr;           // [Tm, k]
    float *wts = nullptr;         // [Tm, k]
    int *counts = nullptr;        // [E]
    int *offsets = nullptr;       // [E+1]
    int *perm = nullptr;          // [Tm*k]
    float *pair_w = nullptr;      // [Tm*k] routing weight of each pair slot (perm order)
    int *touched = nullptr;       // [E]  experts with at least one token, ascending
    int *n_touched = nullptr;     // [1]
    __half *h16 = nullptr;        // [Tm*k, I] SiTU output per (token, expert) pair, perm order
    __half *zperm = nullptr;      // [Tm*k, L + kZPad] z16 rows gathered in pair order (expert GEMM)
    // Block-scaled expert path activations in two-term MXFP8 (plane 0: hi,
    // plane 1: lo; e4m3 bytes, then one ue8m0 scale byte per 32 of them):
    uint8_t *zq = nullptr, *zqs = nullptr;   // latent per token [2][Tm][L], [2][Tm][L/32]
    uint8_t *zp8 = nullptr, *zps = nullptr;  // latent per pair  [2][Tm*k][L], [2][Tm*k][L/32]
    uint8_t *h8 = nullptr, *h8s = nullptr;   // SiTU per pair    [2][Tm*k][I], [2][Tm*k][I/32]
    float *acc = nullptr;         // [Tm, L]
    int2 *tiles = nullptr;        // (expert, n-tile) list of the expert GEMM
    int *perm_hist = nullptr;     // [ceil(Tm/32), E] per-chunk expert counts, then chunk bases
    int *n_tiles = nullptr;       // length of the list
    int *eg_ticket = nullptr;     // [2] items handed out so far by the W1/W3 and the W2 grouped
                                  //   GEMM launch (zeroed with the tile list)
    float *gu = nullptr;          // [min(Tm*k, kSplitPairsMax), 2, I] K-split W1/W3 partial sums (kept zeroed)
    int *gu_cnt = nullptr;        // [max tiles * I/128] their arrival counters (kept at zero)
    __nv_bfloat16 *act = nullptr;     // [Tm, L+S] bf16 [normed latent | shared SiTU] (GEMM path)
    float *gemm_part = nullptr;       // split-K partial sums (kept zeroed between launches)
    int *gemm_tiles = nullptr;        // split-K arrival counters (kept at zero)
    __nv_bfloat16 *xbuf0 = nullptr;   // [Tm, H] staging (host forward, chain)
    __nv_bfloat16 *xbuf1 = nullptr;   // [Tm, H]
    __nv_bfloat16 *xn = nullptr;      // [Tm, H] layer input made from the residual (forward_residual)
    int *err = nullptr;           // [4] device error word + detail
    std::vector<size_t> guards;   // byte offsets of the guard bands after each buffer
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
    bool last_x = false;   // the last forward made its input from a residual (Workspace::xn)
    // launch shapes fixed at create time (no per-launch host queries)
    int grid_dense[3] = {0, 0, 0};   // k_dense_x resident-block cap for TB = 1, 2, 4
    // side stream for the shared experts, which overlap routing and permutation
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    int grid_up[3] = {0, 0, 0};      // k_up for TB = 1, 2, 4
    bool dense_tma_ok[2] = {false, false};   // TMA-fed dense GEMVs usable for T = 1, 2
    bool gemm_ok = false;                    // tensor-core dense GEMMs usable (T >= 16)
    bool egemm_ok = false;                   // tensor-core expert GEMM usable (shape)
    bool mx_ok = false;                      // block-scaled expert path usable at any batch (shape)
    int expert_path = K3MOE_EXPERT_AUTO;     // k3moe_set_expert_path
    k3::TierDev tier;                        // k3moe_set_expert_tier
    float topp = 0.f;                        // k3moe_set_topp (0: keep every pick)
    // per-kernel timing (k3moe_set_profiling)
    bool profiling = false;
    std::deque<k3::ProfRec> prof;
    std::vector<cudaEvent_t> event_pool;
    std::vector<std::string> prof_names;
    std::vector<int> prof_launches;
    std::vector<double> prof_ms;
};

namespace k3 {

// ---- launchers (each returns cudaGetLastError()) -----------------------------
// part 0: router logits and latent down projection; part 1: shared-expert
// gate/up with SiTU; part 2: both.
// wait_x: the shared gate/up (part 1) waits for the previous kernel, which
// wrote its input x (else it reads the caller's x without waiting).
cudaError_t launch_dense_x(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x, int T,
                           cudaStream_t s, int part, bool wait_x = false);
cudaError_t launch_route(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_perm(const k3moe &h, int T, cudaStream_t s, int step);
int perm_chunks(int T);
cudaError_t launch_expert_w13(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_expert_w2(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
cudaError_t launch_up(const k3moe &h, const LayerDev &w, __nv_bfloat16 *y, int T,
                      cudaStream_t s);
cudaError_t launch_chain_glue(const k3moe &h, const __nv_bfloat16 *y, __nv_bfloat16 *x_next,
                              int T, cudaStream_t s);
// x = bf16(RMSNorm(h_in) * gain) per token into Workspace::xn, the layer's
// first kernel (stream order)
cudaError_t launch_residual_norm(const k3moe &h, const float *hin, const __nv_bfloat16 *gain, int T,
                                 cudaStream_t s);
cudaError_t launch_scale_scan(const uint8_t *p, size_t n, int *flag, cudaStream_t s);

// ---- one-time set-up at k3moe_create (attributes, grid sizes) -------------------
cudaError_t init_dense_kernels(k3moe &h);
cudaError_t init_route_kernels(const k3moe_config &c);
cudaError_t init_expert_kernels(const k3moe_config &c);
cudaError_t init_dense_tma(const k3moe_config &c);
cudaError_t init_dense_gemm();
size_t dense_gemm_part_floats(const k3moe_config &c);
size_t dense_gemm_tile_counters(const k3moe_config &c);
// tcgen05 dense GEMMs (T >= 16). part 0: router + down; 1: shared gate/up;
// 2: up + shared down (reads Workspace::act).
cudaError_t launch_dense_gemm(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x,
                              __nv_bfloat16 *y, int T, cudaStream_t s, int part);
cudaError_t launch_norm_act(const k3moe &h, const LayerDev &w, int T, cudaStream_t s);
// tcgen05 grouped expert GEMM (many pairs per expert): the n-tile list, the
// latent gathered into pair order, then W1/W3 (w13) or W2.
bool expert_gemm_ok(const k3moe_config &c);
size_t expert_gemm_max_tiles(const k3moe_config &c);
// the block-scaled grouped GEMM's shapes (weight rows and widths in whole tiles)
bool expert_mx_ok(const k3moe_config &c);
int expert_gemm_min_pairs();
cudaError_t init_expert_gemm();
// whether a grouped batch of T tokens runs the block-scaled GEMM (else the f16 one)
bool expert_gemm_mx(const k3moe &h, int T);
// Batches below the grouped GEMMs' smallest (decode): the block-scaled grouped
// GEMM with each item's K range split (true), or the per-pair GEMVs (false)
bool use_expert_split(const k3moe &h, int T);
constexpr int kSplitPairsMax = 256;   // largest batch (pairs) the K-split path takes
// n-tile width for a batch of T tokens (mx: the block-scaled path's widths)
int expert_gemm_bn(const k3moe &h, int T, bool mx);
cudaError_t launch_expert_tiles(const k3moe &h, int T, cudaStream_t s, bool mx);
cudaError_t launch_gather_latent(const k3moe &h, int T, cudaStream_t s);
cudaError_t launch_expert_gemm(const k3moe &h, const LayerDev &w, int T, cudaStream_t s, bool w13);
// largest scale byte over each row's groups that hold a nonzero nibble
cudaError_t launch_row_scale_max(const uint8_t *packed, const uint8_t *s, size_t rows, int G, uint8_t *out);
// The grouped expert GEMM on block-scaled tensor cores (MXFP4 weights x
// two-term MXFP8 activations): the latent gathered into pair order, then
// W1/W3 with SiTU (w13) or W2 with the weighted scatter-add.
cudaError_t init_expert_mx();
cudaError_t launch_gather_zq(const k3moe &h, int T, cudaStream_t s);
cudaError_t launch_expert_mx(const k3moe &h, const LayerDev &w, int T, cudaStream_t s, bool w13);
bool dense_tma_fits(const k3moe_config &c, int TB);
bool build_dense_tma_maps(const k3moe_config &c, LayerDev &w);
// TMA-fed dense GEMVs for T <= 2. part 0: router + down; 1: shared gate/up;
// 2: latent norm + up + shared down.
// hin (parts 0 and 1): the kernel makes its input x = bf16(RMSNorm(hin) *
// post_gain) itself from the fp32 residual (x unused); part 0 also stores it
// in Workspace::xn.
// t0: the launch covers tokens t0.. of the batch (x and y already offset; the
// workspace rows are offset here). ordered: launch in plain stream order (the
// first kernel of a dense feed-forward layer).
// spare_sm: leave one SM to a block that runs beside this kernel (the
// expert tier's planning block, which fills an SM's register file).
cudaError_t launch_dense_tma(const k3moe &h, const LayerDev &w, const __nv_bfloat16 *x,
                             __nv_bfloat16 *y, int T, cudaStream_t s, int part,
                             const float *hin = nullptr, int t0 = 0, bool ordered = false,
                             bool wait = false, bool spare_sm = false);
bool expert_smem_fits(const k3moe_config &c);
// expert tier: which touched experts are resident and which slots the others
// take (one block), then the copy of the missed experts into their slots
cudaError_t launch_tier_plan(k3moe &h, int layer, cudaStream_t s, bool pin = false);
cudaError_t launch_tier_iota(const k3moe &h);
cudaError_t launch_tier_fill(const k3moe &h, const LayerDev &w, cudaStream_t s);
cudaError_t launch_tier_forget(const k3moe &h, int layer, cudaStream_t s);
// the detail word a k3moe_check_wait_timeout launch latches
constexpr int kWaitCheckWhere = 900;
cudaError_t launch_wait_check(const k3moe &h, cudaStream_t s);

// ---- device helpers -----------------------------------------------------------
__device__ __forceinline__ void set_err(int *err, int code, int detail)
{
    if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// 16-byte streaming load: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
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

// Four bytes of e2m1 pairs -> four f16x2 (byte b -> o_b; low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t &o0, uint32_t &o1,
                                                  uint32_t &o2, uint32_t &o3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(w));
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

// 2^n for an integer n in [-127, 127] (n = -127 gives the subnormal 2^-127).
__device__ __forceinline__ float exp2i(int n)
{
    return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(0x00400000u);
}

// ---- MXFP8 activations: e4m3 elements, one ue8m0 scale per 32 ----------------
// Exponent e of the scale 2^e of a group whose largest magnitude has the fp32
// bit pattern amax: the smallest e with amax <= 448 * 2^e (448 = 1.75 * 2^8,
// the largest e4m3 value), so that no element saturates; clamped to the
// ue8m0 range [-127, 127] (byte = e + 127).
__device__ __forceinline__ int mx_group_exponent(uint32_t amax)
{
    if (amax == 0u) return -127;
    const int e = (int)(amax >> 23) - 127 - 8 + ((amax & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return max(-127, min(127, e));
}

// fp32 -> e4m3 byte, round to nearest even (both lanes of the x2 conversion
// get v, so the byte order of the pair does not matter).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v), "f"(v));
    return r & 0xFFu;
}

// e4m3 byte -> fp32 (exact; through f16, which holds every e4m3 value).
__device__ __forceinline__ float e4m3_to_f32(uint32_t q)
{
    uint32_t h2;
    const uint16_t b = (uint16_t)(q | (q << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Two-term MXFP8 of v, one value per lane of a converged warp whose 32 lanes
// hold one scale group: hi = e4m3(v / 2^eh), eh chosen by mx_group_exponent
// over the group, and lo = e4m3((v - hi 2^eh) / 2^el) with el = eh - 4. The
// scaled values of hi lie within 448, so their rounding error is at most 16
// (half the e4m3 spacing 32 of the top binade); times 2^4 that stays within
// 448 and keeps the residual's own e4m3 precision without a second group
// maximum. hi 2^eh + lo 2^el carries about 8 significant bits more than hi
// alone.
__device__ __forceinline__ void mx8_hilo(float v, uint32_t &qh, uint32_t &ql, int &eh, int &el)
{
    eh = mx_group_exponent(__reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu));
    el = max(eh - 4, -127);
    qh = f32_to_e4m3(v * exp2i(-eh));
    const float r = v - e4m3_to_f32(qh) * exp2i(eh);
    ql = f32_to_e4m3(r * exp2i(-el));
}

__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + expf(-v)); }

__device__ __forceinline__ float tanh_hw(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// SiTU with the hardware tanh (relative error about 2^-11), sigma(g) written
// as (1 + tanh(g / 2)) / 2: b1 tanh(g / b1) sigma(g) b2 tanh(u / b2); ib1 and
// ib2 are 1/b1 and 1/b2. The routed experts' epilogues use it.
__device__ __forceinline__ float situ_hw(float g, float u, float b1, float b2, float ib1, float ib2)
{
    return (b1 * b2) * tanh_hw(g * ib1) * tanh_hw(u * ib2) * fmaf(0.5f, tanh_hw(0.5f * g), 0.5f);
}

__device__ __forceinline__ float situ_f(float g, float u, float b1, float b2)
{
    return (b1 * tanhf(g / b1)) * sigmoid_f(g) * (b2 * tanhf(u / b2));
}

// SiTU from three exponentials and one division: with a = exp(-2|g|/b1),
// b = exp(-2|u|/b2) and c = exp(-g),
//   tanh(g / b1) sigma(g) tanh(u / b2) = sign(g u) (1 - a)(1 - b) / ((1 + a)(1 + b)(1 + c))
// (tanh(x) = sign(x) (1 - e^-2|x|) / (1 + e^-2|x|), sigma(g) = 1 / (1 + e^-g)),
// times b1 b2; ib1 and ib2 are 1/b1 and 1/b2. __expf has a relative error of
// about 2^-21; near g = 0 or u = 0 the error stays absolute (about 1e-7)
// rather than relative. Four special-function operations against about
// twelve for situ_f, for the shared experts' GEMM epilogue, which evaluates
// it for every (token, row) of its tiles.
__device__ __forceinline__ float situ_exp(float g, float u, float b1, float b2, float ib1, float ib2)
{
    const float a = __expf(-2.f * fabsf(g) * ib1);
    const float b = __expf(-2.f * fabsf(u) * ib2);
    const float c = __expf(-g);
    const float r = __fdividef((1.f - a) * (1.f - b), (1.f + a) * (1.f + b) * (1.f + c));
    const uint32_t sgn = (__float_as_uint(g) ^ __float_as_uint(u)) & 0x80000000u;
    return (b1 * b2) * __uint_as_float(__float_as_uint(r) ^ sgn);
}

// ---- mbarrier / bulk-copy (TMA) helpers --------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `parity` to complete, for at most about two seconds;
// on time-out latches kErrTimeout with `where` and returns false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err, int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            set_err(err, kErrTimeout, where);
            return false;
        }
    }
    return true;
}

// Bulk (non-tensor) TMA copy global -> shared, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- programmatic dependent launch ----------------------------------------------
// Every kernel of a forward lets the next one start launching at once, and
// waits for the previous one to finish (and flush) before it reads anything
// that kernel wrote. The wait covers only the immediately preceding kernel,
// so a kernel whose inputs need no wait (it reads only the layer input)
// still waits before it exits: every kernel's completion then implies the
// completion of all earlier kernels of the stream.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem,
                              cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The same without programmatic serialization: the kernel starts only after
// all earlier work on the stream has completed. A layer's first kernel uses
// it, so that every later kernel of the layer may rely on the layer input
// and on the previous forward having finished with the workspace.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ordered(void (*kern)(KArgs...), int grid, int block, size_t smem,
                                  cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ double warp_sum_d(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- RMSNorm of one fp32 residual row into bf16 (the norm in front of the MoE)
// Both passes keep V 16-byte loads in flight per thread (a row is read from
// L2 by many CTAs; one load at a time would be latency-bound).

// This thread's share of sum(h^2) over a row of n4 float4 (fp32 partial sum).
template <int V>
__device__ __forceinline__ float residual_sumsq(const float *row, int n4, int tid, int nthr)
{
    const float4 *hp = reinterpret_cast<const float4 *>(row);
    float sf = 0.f;
    for (int i0 = tid; i0 < n4; i0 += V * nthr) {
        float4 v[V];
#pragma unroll
        for (int u = 0; u < V; u++) {
            const int i = i0 + u * nthr;
            v[u] = i < n4 ? hp[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < V; u++) {
            sf = fmaf(v[u].x, v[u].x, sf);
            sf = fmaf(v[u].y, v[u].y, sf);
            sf = fmaf(v[u].z, v[u].z, sf);
            sf = fmaf(v[u].w, v[u].w, sf);
        }
    }
    return sf;
}

// out[i] = bf16(row[i] * inv * gain[i]) for this thread's float4 groups; a
// second copy goes to out2 when it is not null.
template <int V>
__device__ __forceinline__ void residual_write(const float *row, const __nv_bfloat16 *gain, float inv,
                                               __nv_bfloat16 *out, __nv_bfloat16 *out2, int n4, int tid,
                                               int nthr)
{
    const float4 *hp = reinterpret_cast<const float4 *>(row);
    const uint2 *gp = reinterpret_cast<const uint2 *>(gain);
    for (int i0 = tid; i0 < n4; i0 += V * nthr) {
        float4 v[V];
        uint2 g[V];
#pragma unroll
        for (int u = 0; u < V; u++) {
            const int i = i0 + u * nthr;
            if (i < n4) {
                v[u] = hp[i];
                g[u] = gp[i];
            }
        }
#pragma unroll
        for (int u = 0; u < V; u++) {
            const int i = i0 + u * nthr;
            if (i < n4) {
                const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162 *>(&g[u].x);
                const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162 *>(&g[u].y);
                const __nv_bfloat162 a = __floats2bfloat162_rn(v[u].x * inv * __low2float(g01),
                                                               v[u].y * inv * __high2float(g01));
                const __nv_bfloat162 b = __floats2bfloat162_rn(v[u].z * inv * __low2float(g23),
                                                               v[u].w * inv * __high2float(g23));
                uint2 o;
                o.x = *reinterpret_cast<const uint32_t *>(&a);
                o.y = *reinterpret_cast<const uint32_t *>(&b);
                reinterpret_cast<uint2 *>(out)[i] = o;
                if (out2) reinterpret_cast<uint2 *>(out2)[i] = o;
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace k3
