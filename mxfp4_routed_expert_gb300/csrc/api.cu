// Host side of the C ABI declared in include/k3moe.h: argument and
// configuration checks, device allocation, weight loading and validation, the
// launch sequence of one layer, routing/intermediate readback and timing.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <new>
#include <utility>
#include <string>

#include "k3moe_internal.cuh"

using namespace k3;

namespace {

size_t al256(size_t n) { return (n + 255) & ~size_t(255); }

int check_config(const k3moe_config *c)
{
    if (!c) return K3MOE_ERR_INVALID_ARG;
    if (c->struct_size != sizeof(k3moe_config)) return K3MOE_ERR_CONFIG;
    // all four routed-part sizes 0: a dense feed-forward layer
    const bool dense = c->n_experts == 0 && c->topk == 0 && c->latent == 0 && c->moe_inter == 0;
    const int32_t pos[] = {c->hidden, c->latent, c->n_experts, c->topk, c->moe_inter,
                           c->shared_inter, c->max_layers, c->max_tokens};
    for (int32_t v : pos)
        if (v <= 0 && !(dense && v == 0)) return K3MOE_ERR_CONFIG;
    if (c->hidden <= 0 || c->shared_inter <= 0) return K3MOE_ERR_CONFIG;
    if (c->device < 0) return K3MOE_ERR_CONFIG;
    if ((c->renorm != 0 && c->renorm != 1) || (c->latent_norm != 0 && c->latent_norm != 1))
        return K3MOE_ERR_CONFIG;
    const float fl[] = {c->rms_eps, c->situ_b1, c->situ_b2, c->routed_scale};
    for (float v : fl)
        if (!std::isfinite(v) || v <= 0.f) return K3MOE_ERR_CONFIG;
    if (c->hidden % 64 || c->latent % 64 || c->moe_inter % 64 || c->shared_inter % 64)
        return K3MOE_ERR_SHAPE;
    if (c->topk > kMaxTopk || c->topk > c->n_experts || c->n_experts > kMaxExperts)
        return K3MOE_ERR_SHAPE;
    // the expert GEMVs keep 4 column groups of 32 per lane in registers
    if (c->latent > 4096 || c->moe_inter > 4096) return K3MOE_ERR_SHAPE;
    if (!expert_smem_fits(*c)) return K3MOE_ERR_SHAPE;
    if ((long long)c->max_tokens * c->topk > 65536) return K3MOE_ERR_SHAPE;
    if (c->max_layers > kMaxLayers) return K3MOE_ERR_SHAPE;
    // fp16 partial sums in the expert GEMVs: |SiTU| <= b1*b2 must stay small
    if ((double)c->situ_b1 * c->situ_b2 > 512.0) return K3MOE_ERR_SHAPE;
    // the dense layer runs decode batches through the TMA-fed kernels, two
    // tokens at a time
    if (dense && (!dense_tma_fits(*c, 1) || !dense_tma_fits(*c, 2))) return K3MOE_ERR_SHAPE;
    return K3MOE_OK;
}

struct Carve {
    char *base;
    size_t off = 0;
    std::vector<size_t> *guards = nullptr;   // non-null: a guard band after each buffer
    template <typename T>
    T *take(size_t count)
    {
        T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
        off += al256(count * sizeof(T));
        if (guards) {
            if (base) guards->push_back(off);
            off += kGuardBytes;
        }
        return p;
    }
};

// Writes the guard pattern into every band.
cudaError_t set_guards(void *block, const std::vector<size_t> &guards)
{
    for (size_t g : guards) {
        const cudaError_t e = cudaMemset((char *)block + g, kGuardByte, kGuardBytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// K3MOE_OK when every band still holds the pattern (device idle).
int check_guards(const void *block, const std::vector<size_t> &guards)
{
    unsigned char band[kGuardBytes];
    for (size_t g : guards) {
        if (cudaMemcpy(band, (const char *)block + g, kGuardBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
            return K3MOE_ERR_CUDA;
        for (size_t i = 0; i < kGuardBytes; i++)
            if (band[i] != kGuardByte) return K3MOE_ERR_GUARD;
    }
    return K3MOE_OK;
}

// Lays out the workspace; with base == nullptr only measures it.
size_t carve_workspace(const k3moe_config &c, char *base, Workspace *ws)
{
    const size_t Tm = (size_t)c.max_tokens, E = c.n_experts, L = c.latent, S = c.shared_inter;
    const size_t H = c.hidden, K = c.topk, I = c.moe_inter;
    Workspace w;
    Carve cv{base};
    cv.guards = &w.guards;
    w.logits = cv.take<float>(Tm * E);
    w.z = cv.take<float>(Tm * L);
    w.z16 = cv.take<__half>(Tm * (L + kZPad));
    w.cat = cv.take<float>(Tm * (L + S));
    w.ids = cv.take<int>(Tm * K);
    w.wts = cv.take<float>(Tm * K);
    w.counts = cv.take<int>(E);
    w.offsets = cv.take<int>(E + 1);
    w.perm = cv.take<int>(Tm * K);
    w.pair_w = cv.take<float>(Tm * K);
    w.touched = cv.take<int>(E);
    w.n_touched = cv.take<int>(1);
    w.h16 = cv.take<__half>(Tm * K * I);
    w.acc = cv.take<float>(Tm * L);
    const bool eg = expert_gemm_ok(c), mx = expert_mx_ok(c);
    w.zperm = cv.take<__half>(eg ? Tm * K * (L + kZPad) : 0);
    // two-term MXFP8 activations of the block-scaled grouped expert path
    w.zq = cv.take<uint8_t>(mx ? 2 * Tm * L : 0);
    w.zqs = cv.take<uint8_t>(mx ? 2 * Tm * L / kGroup : 0);
    w.zp8 = cv.take<uint8_t>(mx ? 2 * Tm * K * L : 0);
    w.zps = cv.take<uint8_t>(mx ? 2 * Tm * K * L / kGroup : 0);
    w.h8 = cv.take<uint8_t>(mx ? 2 * Tm * K * I : 0);
    w.h8s = cv.take<uint8_t>(mx ? 2 * Tm * K * I / kGroup : 0);
    w.tiles = cv.take<int2>(mx ? expert_gemm_max_tiles(c) : 0);
    w.n_tiles = cv.take<int>(1);
    w.eg_ticket = cv.take<int>(mx ? 2 : 0);
    w.gu = cv.take<float>(mx ? std::min<size_t>(Tm * K, kSplitPairsMax) * 2 * I : 0);
    w.gu_cnt = cv.take<int>(mx ? expert_gemm_max_tiles(c) * (I / 128) : 0);
    w.perm_hist = cv.take<int>((size_t)perm_chunks(c.max_tokens) * E);
    w.act = cv.take<__nv_bfloat16>(Tm * (L + S));
    w.gemm_part = cv.take<float>(dense_gemm_part_floats(c));
    w.gemm_tiles = cv.take<int>(dense_gemm_tile_counters(c));
    w.xbuf0 = cv.take<__nv_bfloat16>(Tm * H);
    w.xbuf1 = cv.take<__nv_bfloat16>(Tm * H);
    w.xn = cv.take<__nv_bfloat16>(Tm * H);
    w.err = cv.take<int>(4);
    w.block = base;
    w.bytes = cv.off;
    if (ws) *ws = std::move(w);
    return cv.off;
}

struct LayerSizes {
    size_t router, bias, down, up, gain, sh13, sh2, e13p, e13s, e2p, e2s, e13m, e2m;
    size_t dense;     // bf16 weights, bias and gain
    size_t experts;   // the nine routed-expert arrays
    size_t total;
};

LayerSizes layer_sizes(const k3moe_config &c)
{
    const size_t E = c.n_experts, H = c.hidden, L = c.latent, S = c.shared_inter, I = c.moe_inter;
    LayerSizes z;
    z.router = E * H * 2;
    z.bias = E * 4;
    z.down = L * H * 2;
    z.up = H * L * 2;
    z.gain = L * 2;
    z.sh13 = S * H * 2;
    z.sh2 = H * S * 2;
    z.e13p = E * I * (L / 2);
    z.e13s = E * I * (L / kGroup);
    z.e2p = E * L * (I / 2);
    z.e2s = E * L * (I / kGroup);
    z.e13m = E * I;
    z.e2m = E * L;
    z.dense = al256(z.router) + al256(z.bias) + al256(z.down) + al256(z.up) + al256(z.gain) +
              2 * al256(z.sh13) + al256(z.sh2);
    z.experts = 2 * al256(z.e13p) + 2 * al256(z.e13s) + al256(z.e2p) + al256(z.e2s) +
                2 * al256(z.e13m) + al256(z.e2m);
    z.total = z.dense + z.experts;
    return z;
}

// Moves finished event pairs into the per-kernel totals and back into the
// pool. Records complete in stream order, so a non-blocking harvest stops at
// the first one still pending.
int harvest(k3moe *h, bool blocking)
{
    int rc = K3MOE_OK;
    while (!h->prof.empty()) {
        ProfRec r = h->prof.front();
        if (blocking) {
            if (cudaEventSynchronize(r.b) != cudaSuccess) rc = K3MOE_ERR_CUDA;
        } else if (cudaEventQuery(r.b) != cudaSuccess) {
            cudaGetLastError();   // cudaErrorNotReady is not an error here
            break;
        }
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) rc = K3MOE_ERR_CUDA;
        size_t i = 0;
        while (i < h->prof_names.size() && h->prof_names[i] != r.name) i++;
        if (i == h->prof_names.size()) {
            h->prof_names.push_back(r.name);
            h->prof_launches.push_back(0);
            h->prof_ms.push_back(0.0);
        }
        h->prof_launches[i] += 1;
        h->prof_ms[i] += ms;
        h->event_pool.push_back(r.a);
        h->event_pool.push_back(r.b);
        h->prof.pop_front();
    }
    return rc;
}

cudaEvent_t get_event(k3moe *h)
{
    if (h->event_pool.empty()) harvest(h, false);
    if (!h->event_pool.empty()) {
        cudaEvent_t e = h->event_pool.back();
        h->event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return e;
}

// Brackets one kernel launch with events when profiling is on.
struct Prof {
    k3moe *h;
    const char *name;
    cudaStream_t s;
    cudaEvent_t a = nullptr;
    Prof(k3moe *h_, const char *n, cudaStream_t s_) : h(h_), name(n), s(s_)
    {
        if (h->profiling) {
            a = get_event(h);
            if (a) cudaEventRecord(a, s);
        }
    }
    ~Prof()
    {
        if (!a) return;
        cudaEvent_t b = get_event(h);
        if (!b) {   // no event to close the bracket: this launch goes untimed
            h->event_pool.push_back(a);
            return;
        }
        cudaEventRecord(b, s);
        h->prof.push_back({name, a, b});
    }
};

// Grouped tensor-core expert GEMM or per-pair GEMVs for this batch.
bool use_expert_gemm(const k3moe &h, int T)
{
    if (!h.egemm_ok || h.expert_path == K3MOE_EXPERT_GEMV) return false;
    if (T * h.cfg.topk < expert_gemm_min_pairs()) return false;
    return h.expert_path == K3MOE_EXPERT_GEMM || h.expert_path == K3MOE_EXPERT_MX || T >= kGemmMinTokens;
}

// hin != nullptr: the layer input is made from the fp32 residual hin by the
// RMSNorm in front of the MoE (inside the decode dense kernels at T <= 2, else
// by a first kernel into Workspace::xn); x is then unused.
int run_layer(k3moe *h, const LayerDev &w, const __nv_bfloat16 *x, __nv_bfloat16 *y, int T,
              cudaStream_t s, const float *hin = nullptr)
{
    cudaError_t e;
    const bool tier = h->tier.slots > 0;
#define K3_STEP(name, call)                        \
    {                                              \
        Prof p_(h, name, s);                       \
        e = (call);                                \
    }                                              \
    if (e != cudaSuccess) return K3MOE_ERR_CUDA;
    // Decode (T <= 15), one stream with programmatic dependent launch:
    //   router+down -> route -> shared gate/up -> experts -> up
    // The shared gate/up kernel's producers stream weights before their wait
    // on the router, so it runs alongside the single-block router on the
    // other SMs; a side stream would add an event fork and join for no
    // overlap (the experts need every SM once the shared experts hold them).
    // Batched (T >= 16): the shared gate/up GEMM on a side stream after
    // router+down, joined before the experts.
    const bool gemm = T >= kGemmMinTokens && h->gemm_ok;
    if (is_dense(h->cfg)) {
        // dense feed-forward layer: gate/up with SiTU, then the down projection
        if (hin) {
            K3_STEP("residual_rmsnorm", launch_residual_norm(*h, hin, w.post_gain, T, s));
            x = h->ws.xn;
        }
        if (gemm) {
            K3_STEP("dense_gate_up_gemm", launch_dense_gemm(*h, w, x, nullptr, T, s, 1));
            K3_STEP("dense_down_gemm", launch_dense_gemm(*h, w, nullptr, y, T, s, 2));
        } else {
            // decode: two tokens per pass of the TMA-fed kernels; the first
            // kernel opens the layer in stream order unless it follows the norm
            const size_t H = h->cfg.hidden;
            for (int t0 = 0; t0 < T; t0 += 2) {
                const int n = T - t0 < 2 ? T - t0 : 2;
                K3_STEP("dense_gate_up_gemv", launch_dense_tma(*h, w, x + t0 * H, nullptr, n, s, 1, nullptr, t0,
                                                               t0 == 0 && !hin, hin != nullptr));
                K3_STEP("dense_down_gemv", launch_dense_tma(*h, w, nullptr, y + t0 * H, n, s, 2, nullptr, t0));
            }
        }
        h->last_T = T;
        h->last_x = hin != nullptr;
        return K3MOE_OK;
    }
    const bool tma = T <= 2 && h->dense_tma_ok[T - 1];
    const bool egemm = use_expert_gemm(*h, T);
    const float *fused = (hin && tma) ? hin : nullptr;   // made inside the dense kernels
    if (hin && !tma) {
        K3_STEP("residual_rmsnorm", launch_residual_norm(*h, hin, w.post_gain, T, s));
        x = h->ws.xn;
    }
    if (gemm) {
        K3_STEP("router_down_gemm", launch_dense_gemm(*h, w, x, nullptr, T, s, 0));
        if (cudaEventRecord(h->ev_fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(h->side, h->ev_fork, 0) != cudaSuccess)
            return K3MOE_ERR_CUDA;
        {
            Prof p_(h, "shared_gate_up_gemm", h->side);
            e = launch_dense_gemm(*h, w, x, nullptr, T, h->side, 1);
        }
        if (e != cudaSuccess || cudaEventRecord(h->ev_join, h->side) != cudaSuccess)
            return K3MOE_ERR_CUDA;
        K3_STEP("route_topk", launch_route(*h, w, T, s));
    } else {
        K3_STEP("router_down_gemv", tma ? launch_dense_tma(*h, w, x, nullptr, T, s, 0, fused)
                                        : launch_dense_x(*h, w, x, T, s, 0));
        K3_STEP("route_topk", launch_route(*h, w, T, s));
        if (tier && T == 1) {
            // the copy of missed experts over the host link overlaps the
            // shared experts' HBM stream, which launches behind it
            K3_STEP("tier_plan", launch_tier_plan(*h, w.index, s));
            K3_STEP("tier_fill", launch_tier_fill(*h, w, s));
        }
        K3_STEP("shared_gate_up_gemv", tma ? launch_dense_tma(*h, w, x, nullptr, T, s, 1, fused, 0, false,
                                                              false, tier && T == 1)
                                           : launch_dense_x(*h, w, x, T, s, 1, hin != nullptr));
    }
    if (T > 1) {   // T == 1: written by route_topk
        K3_STEP("perm_count", launch_perm(*h, T, s, 0));
        K3_STEP("perm_scan", launch_perm(*h, T, s, 1));
        K3_STEP("perm_place", launch_perm(*h, T, s, 2));
        if (tier) {
            K3_STEP("tier_plan", launch_tier_plan(*h, w.index, s));
            K3_STEP("tier_fill", launch_tier_fill(*h, w, s));
        }
    }
    if (gemm && cudaStreamWaitEvent(s, h->ev_join, 0) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (egemm && expert_gemm_mx(*h, T)) {
        K3_STEP("expert_tiles", launch_expert_tiles(*h, T, s, true));
        K3_STEP("gather_latent", launch_gather_zq(*h, T, s));
        K3_STEP("expert_w13_gemm", launch_expert_mx(*h, w, T, s, true));
        K3_STEP("expert_w2_gemm", launch_expert_mx(*h, w, T, s, false));
    } else if (egemm) {
        K3_STEP("expert_tiles", launch_expert_tiles(*h, T, s, false));
        K3_STEP("gather_latent", launch_gather_latent(*h, T, s));
        K3_STEP("expert_w13_gemm", launch_expert_gemm(*h, w, T, s, true));
        K3_STEP("expert_w2_gemm", launch_expert_gemm(*h, w, T, s, false));
    } else if (use_expert_split(*h, T)) {
        K3_STEP("expert_tiles", launch_expert_tiles(*h, T, s, true));
        K3_STEP("gather_latent", launch_gather_zq(*h, T, s));
        K3_STEP("expert_w13_gemm", launch_expert_mx(*h, w, T, s, true));
        K3_STEP("expert_w2_gemm", launch_expert_mx(*h, w, T, s, false));
    } else {
        K3_STEP("expert_w13_gemv", launch_expert_w13(*h, w, T, s));
        K3_STEP("expert_w2_gemv", launch_expert_w2(*h, w, T, s));
    }
    if (gemm) {
        K3_STEP("latent_rmsnorm", launch_norm_act(*h, w, T, s));
        K3_STEP("up_shared_gemm", launch_dense_gemm(*h, w, nullptr, y, T, s, 2));
    } else {
        K3_STEP("norm_up_shared_gemv", tma ? launch_dense_tma(*h, w, nullptr, y, T, s, 2)
                                           : launch_up(*h, w, y, T, s));
    }
#undef K3_STEP
    h->last_T = T;
    h->last_x = hin != nullptr;
    return K3MOE_OK;
}

// Free device memory as the size checks see it: the runtime's figure, capped
// at K3MOE_DEVICE_BUDGET_MB megabytes when that variable holds a number.
cudaError_t free_device_bytes(size_t *fr)
{
    size_t tot = 0;
    const cudaError_t e = cudaMemGetInfo(fr, &tot);
    if (e != cudaSuccess) return e;
    if (const char *env = std::getenv("K3MOE_DEVICE_BUDGET_MB")) {
        char *end = nullptr;
        const unsigned long long mb = std::strtoull(env, &end, 10);
        if (end != env && *end == '\0' && mb < (1ull << 40)) {
            const size_t cap = (size_t)mb << 20;
            if (cap < *fr) *fr = cap;
        }
    }
    return cudaSuccess;
}

// The error code for a C++ exception caught at an entry point: host memory
// ran out (std::bad_alloc), or anything else the runtime's C++ layer threw.
int abi_exception()
{
    try {
        throw;
    } catch (const std::bad_alloc &) {
        return K3MOE_ERR_OOM;
    } catch (...) {
        return K3MOE_ERR_CUDA;
    }
}

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const char *pa = (const char *)a, *pb = (const char *)b;
    return pa < pb + nb && pb < pa + na;
}

// The kernels read and write activations in 16-byte vectors (and through TMA
// maps at T >= 16, whose base must be 16-byte aligned).
bool misaligned(const void *p) { return (uintptr_t)p % 16 != 0; }

void free_layer(LayerDev &l)
{
    if (l.block) cudaFree(l.block);
    if (l.host_block) cudaFreeHost(l.host_block);
    if (l.post_block) cudaFree(l.post_block);
    l = LayerDev();
}

void free_tier(k3::TierDev &t)
{
    if (t.block) cudaFree(t.block);
    t = k3::TierDev();
}

}  // namespace

extern "C" {

int k3moe_abi_version(void) { return K3MOE_ABI_VERSION; }

const char *k3moe_strerror(int code)
{
    switch (code) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_INVALID_ARG: return "invalid argument";
    case K3MOE_ERR_CONFIG: return "configuration field missing or invalid";
    case K3MOE_ERR_SHAPE: return "unsupported layer shape";
    case K3MOE_ERR_OOM: return "not enough device memory";
    case K3MOE_ERR_BAD_SCALE: return "expert scale byte 255 (NaN) found";
    case K3MOE_ERR_NOT_LOADED: return "layer not loaded";
    case K3MOE_ERR_CUDA: return "CUDA runtime error";
    case K3MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case K3MOE_ERR_DEVICE: return "device-side index check failed";
    case K3MOE_ERR_GUARD: return "guard band after a library buffer overwritten";
    default: return "unknown error";
    }
}

int k3moe_create(const k3moe_config *cfg, k3moe **out)
{
    if (!out) return K3MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const int rc = check_config(cfg);
    if (rc != K3MOE_OK) return rc;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || cfg->device >= ndev) return K3MOE_ERR_CUDA;
    if (cudaSetDevice(cfg->device) != cudaSuccess) return K3MOE_ERR_CUDA;
    k3moe *h = new (std::nothrow) k3moe();
    if (!h) return K3MOE_ERR_OOM;
    h->cfg = *cfg;
    cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, cfg->device);
    const size_t need = carve_workspace(*cfg, nullptr, nullptr);
    size_t fr = 0;
    if (free_device_bytes(&fr) != cudaSuccess) {
        delete h;
        return K3MOE_ERR_CUDA;
    }
    if (need + (64u << 20) > fr) {
        delete h;
        return K3MOE_ERR_OOM;
    }
    void *blk = nullptr;
    if (cudaMalloc(&blk, need) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return K3MOE_ERR_OOM;
    }
    try {
        carve_workspace(*cfg, (char *)blk, &h->ws);
    } catch (const std::bad_alloc &) {   // no C++ exception crosses the C ABI
        cudaFree(blk);
        delete h;
        return K3MOE_ERR_OOM;
    }
    int prio_lo = 0, prio_hi = 0;
    cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi);
    if (cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, prio_lo) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        if (h->side) cudaStreamDestroy(h->side);
        if (h->ev_fork) cudaEventDestroy(h->ev_fork);
        if (h->ev_join) cudaEventDestroy(h->ev_join);
        cudaFree(blk);
        delete h;
        return K3MOE_ERR_CUDA;
    }
    if (cudaMemset(blk, 0, need) != cudaSuccess || set_guards(blk, h->ws.guards) != cudaSuccess ||
        init_dense_kernels(*h) != cudaSuccess ||
        init_route_kernels(*cfg) != cudaSuccess || init_expert_kernels(*cfg) != cudaSuccess ||
        init_dense_tma(*cfg) != cudaSuccess || init_dense_gemm() != cudaSuccess ||
        init_expert_gemm() != cudaSuccess || init_expert_mx() != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        cudaStreamDestroy(h->side);
        cudaEventDestroy(h->ev_fork);
        cudaEventDestroy(h->ev_join);
        cudaFree(blk);
        delete h;
        return K3MOE_ERR_CUDA;
    }
    h->dense_tma_ok[0] = dense_tma_fits(*cfg, 1);
    h->dense_tma_ok[1] = dense_tma_fits(*cfg, 2);
    // every TMA box of the GEMMs must lie inside its tensor: 128-row weight tiles
    h->gemm_ok = is_dense(*cfg) ? (cfg->shared_inter >= 128 && cfg->hidden >= 128)
                                : (cfg->n_experts >= 128 && cfg->latent >= 128 && cfg->shared_inter >= 128 &&
                                   cfg->hidden >= 128);
    h->egemm_ok = expert_gemm_ok(*cfg);
    h->mx_ok = expert_mx_ok(*cfg);
    try {
        h->layers.resize((size_t)cfg->max_layers);
    } catch (const std::bad_alloc &) {   // no C++ exception crosses the C ABI
        k3moe_destroy(h);
        return K3MOE_ERR_OOM;
    }
    *out = h;
    return K3MOE_OK;
}

void k3moe_destroy(k3moe *h)
{
    if (!h) return;
    cudaSetDevice(h->cfg.device);
    for (auto &l : h->layers) free_layer(l);
    free_tier(h->tier);
    if (h->ws.block) cudaFree(h->ws.block);
    for (auto &r : h->prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    for (auto e : h->event_pool) cudaEventDestroy(e);
    if (h->side) {
        cudaStreamSynchronize(h->side);
        cudaStreamDestroy(h->side);
    }
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    delete h;
}

int k3moe_load_layer(k3moe *h, int layer, const k3moe_layer_weights *w)
{
    try {
        if (!h || !w) return K3MOE_ERR_INVALID_ARG;
        if (w->struct_size != sizeof(k3moe_layer_weights)) return K3MOE_ERR_INVALID_ARG;
        if (layer < 0 || layer >= h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
        if (w->where != K3MOE_HOST && w->where != K3MOE_DEVICE) return K3MOE_ERR_INVALID_ARG;
        const k3moe_config &c = h->cfg;
        const bool dense = is_dense(c);   // only the three feed-forward matrices
        if (!w->shared_w1 || !w->shared_w3 || !w->shared_w2) return K3MOE_ERR_INVALID_ARG;
        if (!dense && (!w->router_w || !w->down_w || !w->up_w || !w->w1_packed || !w->w1_scale ||
                       !w->w3_packed || !w->w3_scale || !w->w2_packed || !w->w2_scale))
            return K3MOE_ERR_INVALID_ARG;
        if (!dense && c.latent_norm && !w->latent_gain) return K3MOE_ERR_INVALID_ARG;
        for (int e = 0; e < c.n_experts; e++)
            if (!w->w1_packed[e] || !w->w1_scale[e] || !w->w3_packed[e] || !w->w3_scale[e] ||
                !w->w2_packed[e] || !w->w2_scale[e])
                return K3MOE_ERR_INVALID_ARG;
        if (cudaSetDevice(c.device) != cudaSuccess) return K3MOE_ERR_CUDA;

        const LayerSizes z = layer_sizes(c);
        // Expert tier: the routed experts go to one pinned, device-mapped host
        // block and reach the device through the slots; else all of the layer
        // lives in device memory.
        const bool tiered = h->tier.slots > 0;
        const size_t dev_bytes = tiered ? z.dense : z.total;
        size_t fr = 0;
        if (free_device_bytes(&fr) != cudaSuccess) return K3MOE_ERR_CUDA;
        if (dev_bytes + (256u << 20) > fr) return K3MOE_ERR_OOM;   // checked before any allocation
        void *blk = nullptr;
        if (cudaMalloc(&blk, dev_bytes) != cudaSuccess) {
            cudaGetLastError();
            return K3MOE_ERR_OOM;
        }
        void *hblk = nullptr, *hdev = nullptr;
        if (tiered) {
            if (cudaHostAlloc(&hblk, z.experts, cudaHostAllocMapped) != cudaSuccess) {
                cudaGetLastError();
                cudaFree(blk);
                return K3MOE_ERR_OOM;
            }
            if (cudaHostGetDevicePointer(&hdev, hblk, 0) != cudaSuccess) {
                cudaGetLastError();
                cudaFreeHost(hblk);
                cudaFree(blk);
                return K3MOE_ERR_CUDA;
            }
        }
        LayerDev L;
        L.block = blk;
        L.bytes = dev_bytes;
        L.index = layer;
        Carve cv{(char *)blk};
        __nv_bfloat16 *router = cv.take<__nv_bfloat16>(z.router / 2);
        float *bias = cv.take<float>(z.bias / 4);
        __nv_bfloat16 *down = cv.take<__nv_bfloat16>(z.down / 2);
        __nv_bfloat16 *up = cv.take<__nv_bfloat16>(z.up / 2);
        __nv_bfloat16 *gain = cv.take<__nv_bfloat16>(z.gain / 2);
        __nv_bfloat16 *sh1 = cv.take<__nv_bfloat16>(z.sh13 / 2);
        __nv_bfloat16 *sh3 = cv.take<__nv_bfloat16>(z.sh13 / 2);
        __nv_bfloat16 *sh2 = cv.take<__nv_bfloat16>(z.sh2 / 2);
        // the nine expert arrays [E][...]: after the dense tensors, or in the host
        // block (ex: where the copies go; exd: the same arrays as kernels see them)
        const size_t asz[kTierPieces] = {z.e13p, z.e13s, z.e13p, z.e13s, z.e2p, z.e2s, z.e13m, z.e13m, z.e2m};
        uint8_t *ex[kTierPieces], *exd[kTierPieces];
        {
            Carve ce{tiered ? (char *)hblk : (char *)blk, tiered ? 0 : z.dense};
            Carve cd{tiered ? (char *)hdev : (char *)blk, tiered ? 0 : z.dense};
            for (int p = 0; p < kTierPieces; p++) {
                ex[p] = ce.take<uint8_t>(asz[p]);
                exd[p] = cd.take<uint8_t>(asz[p]);
            }
        }

        const cudaMemcpyKind kind =
            w->where == K3MOE_HOST ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
        // expert pieces: into device memory, or into the pinned host block
        const cudaMemcpyKind ekind = tiered ? cudaMemcpyDefault : kind;
        int rc = K3MOE_OK;
        int *flag = h->ws.err + 2;   // scratch word for the scale scan
    #define K3_CP(dst, src, n, k)                                             \
        if (rc == K3MOE_OK && cudaMemcpy((dst), (src), (n), (k)) != cudaSuccess) \
            rc = K3MOE_ERR_CUDA;
        if (!dense) K3_CP(router, w->router_w, z.router, kind);
        if (w->router_bias && !dense) {
            K3_CP(bias, w->router_bias, z.bias, kind);
        } else if (rc == K3MOE_OK && cudaMemset(bias, 0, z.bias) != cudaSuccess) {
            rc = K3MOE_ERR_CUDA;
        }
        if (!dense) {
            K3_CP(down, w->down_w, z.down, kind);
            K3_CP(up, w->up_w, z.up, kind);
            if (w->latent_gain) K3_CP(gain, w->latent_gain, z.gain, kind);
        }
        K3_CP(sh1, w->shared_w1, z.sh13, kind);
        K3_CP(sh3, w->shared_w3, z.sh13, kind);
        K3_CP(sh2, w->shared_w2, z.sh2, kind);
        const size_t pe13 = (size_t)c.moe_inter * (c.latent / 2), se13 = (size_t)c.moe_inter * (c.latent / kGroup);
        const size_t pe2 = (size_t)c.latent * (c.moe_inter / 2), se2 = (size_t)c.latent * (c.moe_inter / kGroup);
        for (int e = 0; e < c.n_experts && rc == K3MOE_OK; e++) {
            K3_CP(ex[0] + e * pe13, w->w1_packed[e], pe13, ekind);
            K3_CP(ex[1] + e * se13, w->w1_scale[e], se13, ekind);
            K3_CP(ex[2] + e * pe13, w->w3_packed[e], pe13, ekind);
            K3_CP(ex[3] + e * se13, w->w3_scale[e], se13, ekind);
            K3_CP(ex[4] + e * pe2, w->w2_packed[e], pe2, ekind);
            K3_CP(ex[5] + e * se2, w->w2_scale[e], se2, ekind);
        }
    #undef K3_CP
        if (rc == K3MOE_OK && !dense) {
            // scale checks and row maxima read the arrays where they live (the
            // host block through its device mapping in the tier)
            int bad = 0;
            if (cudaMemset(flag, 0, sizeof(int)) != cudaSuccess ||
                launch_scale_scan(exd[1], z.e13s, flag, 0) != cudaSuccess ||
                launch_scale_scan(exd[3], z.e13s, flag, 0) != cudaSuccess ||
                launch_scale_scan(exd[5], z.e2s, flag, 0) != cudaSuccess ||
                launch_row_scale_max(exd[0], exd[1], z.e13m, c.latent / kGroup, exd[6]) != cudaSuccess ||
                launch_row_scale_max(exd[2], exd[3], z.e13m, c.latent / kGroup, exd[7]) != cudaSuccess ||
                launch_row_scale_max(exd[4], exd[5], z.e2m, c.moe_inter / kGroup, exd[8]) != cudaSuccess ||
                cudaMemcpy(&bad, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
                rc = K3MOE_ERR_CUDA;
            else if (bad)
                rc = K3MOE_ERR_BAD_SCALE;
            cudaMemset(flag, 0, sizeof(int));
        }
        // a reloaded tiered layer gives up its slots before its old block goes
        if (rc == K3MOE_OK && tiered && h->layers[(size_t)layer].loaded &&
            (launch_tier_forget(*h, layer, 0) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess))
            rc = K3MOE_ERR_CUDA;
        if (rc == K3MOE_OK && tiered && h->layers[(size_t)layer].pinned)
            h->tier.pinned -= c.n_experts;   // the forget freed its pinned slots
        if (rc != K3MOE_OK) {
            cudaFree(blk);
            if (hblk) cudaFreeHost(hblk);
            return rc;
        }
        L.router_w = router;
        L.bias = bias;
        L.down_w = down;
        L.up_w = up;
        L.gain = c.latent_norm ? gain : nullptr;
        L.sh_w1 = sh1;
        L.sh_w3 = sh3;
        L.sh_w2 = sh2;
        // expert arrays as the expert kernels address them: the handle's slots
        // (tier) or the layer's own copy
        const uint8_t *const *arr = tiered ? (const uint8_t *const *)h->tier.arr : (const uint8_t *const *)exd;
        L.w1p = arr[0];
        L.w1s = arr[1];
        L.w3p = arr[2];
        L.w3s = arr[3];
        L.w2p = arr[4];
        L.w2s = arr[5];
        L.w1max = arr[6];
        L.w3max = arr[7];
        L.w2max = arr[8];
        if (tiered) {
            L.wslot = h->tier.slot_of + (size_t)layer * c.n_experts;
            L.n_wslots = h->tier.slots;
            L.host_block = hblk;
            for (int p = 0; p < kTierPieces; p++) L.hsrc[p] = exd[p];
        } else {
            L.wslot = nullptr;
            L.n_wslots = c.n_experts;
        }
        if (dense_tma_fits(c, 1)) build_dense_tma_maps(c, L);   // else the maps are never used
        L.loaded = true;
        free_layer(h->layers[(size_t)layer]);
        h->layers[(size_t)layer] = L;
        return K3MOE_OK;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_forward(k3moe *h, int layer, const void *x, void *y, int T, void *stream)
{
    try {
        if (!h || !x || !y) return K3MOE_ERR_INVALID_ARG;
        if (layer < 0 || layer >= h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
        if (T < 1 || T > h->cfg.max_tokens) return K3MOE_ERR_INVALID_ARG;
        const size_t nb = (size_t)T * h->cfg.hidden * 2;
        if (overlap(x, nb, y, nb) || misaligned(x) || misaligned(y)) return K3MOE_ERR_INVALID_ARG;
        const LayerDev &w = h->layers[(size_t)layer];
        if (!w.loaded) return K3MOE_ERR_NOT_LOADED;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        return run_layer(h, w, (const __nv_bfloat16 *)x, (__nv_bfloat16 *)y, T, (cudaStream_t)stream);
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_load_post_norm(k3moe *h, int layer, const void *gain, int where)
{
    if (!h || !gain) return K3MOE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
    if (where != K3MOE_HOST && where != K3MOE_DEVICE) return K3MOE_ERR_INVALID_ARG;
    LayerDev &w = h->layers[(size_t)layer];
    if (!w.loaded) return K3MOE_ERR_NOT_LOADED;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
    const size_t nb = (size_t)h->cfg.hidden * 2;
    void *p = w.post_block;
    if (!p && cudaMalloc(&p, nb) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ERR_OOM;
    }
    if (cudaMemcpy(p, gain, nb, where == K3MOE_HOST ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice) !=
        cudaSuccess) {
        cudaGetLastError();
        if (!w.post_block) cudaFree(p);
        return K3MOE_ERR_CUDA;
    }
    w.post_block = p;
    w.post_gain = (const __nv_bfloat16 *)p;
    return K3MOE_OK;
}

int k3moe_forward_residual(k3moe *h, int layer, const float *h_in, void *y, int T, void *stream)
{
    try {
        if (!h || !h_in || !y) return K3MOE_ERR_INVALID_ARG;
        if (layer < 0 || layer >= h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
        if (T < 1 || T > h->cfg.max_tokens) return K3MOE_ERR_INVALID_ARG;
        if (misaligned(h_in) || misaligned(y)) return K3MOE_ERR_INVALID_ARG;
        if (overlap(h_in, (size_t)T * h->cfg.hidden * 4, y, (size_t)T * h->cfg.hidden * 2))
            return K3MOE_ERR_INVALID_ARG;
        const LayerDev &w = h->layers[(size_t)layer];
        if (!w.loaded || !w.post_gain) return K3MOE_ERR_NOT_LOADED;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        return run_layer(h, w, nullptr, (__nv_bfloat16 *)y, T, (cudaStream_t)stream, h_in);
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_forward_chain(k3moe *h, int first_layer, int n_layers, const void *x, void *y, int T,
                        void *stream)
{
    try {
        if (!h || !x || !y || n_layers < 1) return K3MOE_ERR_INVALID_ARG;
        if (first_layer < 0 || first_layer + n_layers > h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
        if (T < 1 || T > h->cfg.max_tokens) return K3MOE_ERR_INVALID_ARG;
        const size_t nb = (size_t)T * h->cfg.hidden * 2;
        if (overlap(x, nb, y, nb) || misaligned(x) || misaligned(y)) return K3MOE_ERR_INVALID_ARG;
        for (int l = first_layer; l < first_layer + n_layers; l++)
            if (!h->layers[(size_t)l].loaded) return K3MOE_ERR_NOT_LOADED;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        cudaStream_t s = (cudaStream_t)stream;
        const __nv_bfloat16 *cur = (const __nv_bfloat16 *)x;
        for (int i = 0; i < n_layers; i++) {
            const bool last = i == n_layers - 1;
            __nv_bfloat16 *out = last ? (__nv_bfloat16 *)y : h->ws.xbuf0;
            int rc = run_layer(h, h->layers[(size_t)(first_layer + i)], cur, out, T, s);
            if (rc != K3MOE_OK) return rc;
            if (!last) {
                cudaError_t e;
                {
                    Prof p(h, "chain_glue_rmsnorm", s);
                    e = launch_chain_glue(*h, h->ws.xbuf0, h->ws.xbuf1, T, s);
                }
                if (e != cudaSuccess) return K3MOE_ERR_CUDA;
                cur = h->ws.xbuf1;
            }
        }
        return K3MOE_OK;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_forward_host(k3moe *h, int layer, const void *x_host, void *y_host, int T, void *stream)
{
    try {
        if (!h || !x_host || !y_host) return K3MOE_ERR_INVALID_ARG;
        if (layer < 0 || layer >= h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
        if (T < 1 || T > h->cfg.max_tokens) return K3MOE_ERR_INVALID_ARG;
        if (!h->layers[(size_t)layer].loaded) return K3MOE_ERR_NOT_LOADED;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        cudaStream_t s = (cudaStream_t)stream;
        const size_t nb = (size_t)T * h->cfg.hidden * 2;
        // The layer's last kernel writes each output element once with a plain
        // store: a pinned (device-mapped) y is written in place, saving the copy
        // back. (x stays a copy: the first kernels read it from many CTAs.)
        {
            cudaPointerAttributes ay{};
            if (cudaPointerGetAttributes(&ay, y_host) == cudaSuccess && ay.type == cudaMemoryTypeHost &&
                ay.devicePointer && !misaligned(ay.devicePointer)) {
                if (cudaMemcpyAsync(h->ws.xbuf0, x_host, nb, cudaMemcpyHostToDevice, s) != cudaSuccess)
                    return K3MOE_ERR_CUDA;
                const int rc =
                    run_layer(h, h->layers[(size_t)layer], h->ws.xbuf0, (__nv_bfloat16 *)ay.devicePointer, T, s);
                if (rc != K3MOE_OK) return rc;
                return cudaStreamSynchronize(s) == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
            }
            cudaGetLastError();   // pageable or unaligned y: the copy path below
        }
        if (cudaMemcpyAsync(h->ws.xbuf0, x_host, nb, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return K3MOE_ERR_CUDA;
        int rc = run_layer(h, h->layers[(size_t)layer], h->ws.xbuf0, h->ws.xbuf1, T, s);
        if (rc != K3MOE_OK) return rc;
        if (cudaMemcpyAsync(y_host, h->ws.xbuf1, nb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return K3MOE_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return K3MOE_ERR_CUDA;
        return K3MOE_OK;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_get_routing(k3moe *h, int32_t *ids, float *w, int32_t *counts, int32_t *offsets,
                      int32_t *perm, void *stream)
{
    if (!h) return K3MOE_ERR_INVALID_ARG;
    if (h->last_T <= 0) return K3MOE_ERR_NOT_LOADED;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t TK = (size_t)h->last_T * h->cfg.topk, E = h->cfg.n_experts;
    const cudaMemcpyKind d2d = cudaMemcpyDeviceToDevice;
    if ((ids && cudaMemcpyAsync(ids, h->ws.ids, TK * 4, d2d, s) != cudaSuccess) ||
        (w && cudaMemcpyAsync(w, h->ws.wts, TK * 4, d2d, s) != cudaSuccess) ||
        (counts && cudaMemcpyAsync(counts, h->ws.counts, E * 4, d2d, s) != cudaSuccess) ||
        (offsets && cudaMemcpyAsync(offsets, h->ws.offsets, (E + 1) * 4, d2d, s) != cudaSuccess) ||
        (perm && cudaMemcpyAsync(perm, h->ws.perm, TK * 4, d2d, s) != cudaSuccess))
        return K3MOE_ERR_CUDA;
    return K3MOE_OK;
}

int k3moe_get_intermediate(k3moe *h, int which, void *dst, size_t bytes, void *stream)
{
    if (!h || !dst) return K3MOE_ERR_INVALID_ARG;
    if (h->last_T <= 0) return K3MOE_ERR_NOT_LOADED;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t T = (size_t)h->last_T, L = h->cfg.latent, S = h->cfg.shared_inter;
    const size_t E = h->cfg.n_experts;
    cudaError_t e;
    switch (which) {
    case K3MOE_T_Z:
        if (bytes > T * L * 4) return K3MOE_ERR_INVALID_ARG;
        e = cudaMemcpyAsync(dst, h->ws.z, bytes, cudaMemcpyDeviceToDevice, s);
        break;
    case K3MOE_T_ACC:
        if (bytes > T * L * 4) return K3MOE_ERR_INVALID_ARG;
        e = cudaMemcpyAsync(dst, h->ws.acc, bytes, cudaMemcpyDeviceToDevice, s);
        break;
    case K3MOE_T_LOGITS:
        if (bytes > T * E * 4) return K3MOE_ERR_INVALID_ARG;
        e = cudaMemcpyAsync(dst, h->ws.logits, bytes, cudaMemcpyDeviceToDevice, s);
        break;
    case K3MOE_T_X:
        if (!h->last_x) return K3MOE_ERR_INVALID_ARG;
        if (bytes > T * h->cfg.hidden * 2) return K3MOE_ERR_INVALID_ARG;
        e = cudaMemcpyAsync(dst, h->ws.xn, bytes, cudaMemcpyDeviceToDevice, s);
        break;
    case K3MOE_T_SHARED: {
        if (bytes != T * S * 4) return K3MOE_ERR_INVALID_ARG;
        e = cudaMemcpy2DAsync(dst, S * 4, h->ws.cat + L, (L + S) * 4, S * 4, T,
                              cudaMemcpyDeviceToDevice, s);
        break;
    }
    default:
        return K3MOE_ERR_INVALID_ARG;
    }
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3moe_sync_status(k3moe *h)
{
    if (!h) return K3MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ERR_CUDA;
    }
    int word[2] = {0, 0};
    if (cudaMemcpy(word, h->ws.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return K3MOE_ERR_CUDA;
    if (word[0] != kErrNone) {
        cudaMemset(h->ws.err, 0, 2 * sizeof(int));
        return word[0] == kErrTimeout ? K3MOE_ERR_TIMEOUT : K3MOE_ERR_DEVICE;
    }
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ERR_CUDA;
    int rc = check_guards(h->ws.block, h->ws.guards);
    if (rc == K3MOE_OK && h->tier.block) rc = check_guards(h->tier.block, h->tier.guards);
    return rc;
}

int k3moe_set_expert_path(k3moe *h, int mode)
{
    if (!h) return K3MOE_ERR_INVALID_ARG;
    if (mode != K3MOE_EXPERT_AUTO && mode != K3MOE_EXPERT_GEMV && mode != K3MOE_EXPERT_GEMM &&
        mode != K3MOE_EXPERT_MX)
        return K3MOE_ERR_INVALID_ARG;
    if (mode == K3MOE_EXPERT_GEMM && !h->egemm_ok) return K3MOE_ERR_SHAPE;
    if (mode == K3MOE_EXPERT_MX && !h->mx_ok) return K3MOE_ERR_SHAPE;
    h->expert_path = mode;
    return K3MOE_OK;
}

int k3moe_set_expert_tier(k3moe *h, int slots)
{
    try {
        if (!h) return K3MOE_ERR_INVALID_ARG;
        for (const auto &l : h->layers)
            if (l.loaded) return K3MOE_ERR_INVALID_ARG;
        const k3moe_config &c = h->cfg;
        if (slots != 0 && (is_dense(c) || slots < c.n_experts || slots > kTierMaxSlots))
            return K3MOE_ERR_INVALID_ARG;
        if (cudaSetDevice(c.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        free_tier(h->tier);
        if (slots == 0) return K3MOE_OK;
        TierDev t;
        const size_t I = c.moe_inter, L = c.latent, E = c.n_experts;
        const size_t piece[kTierPieces] = {I * (L / 2), I * (L / kGroup), I * (L / 2), I * (L / kGroup),
                                           L * (I / 2), L * (I / kGroup), I, I, L};
        for (int p = 0; p < kTierPieces; p++) {
            if (piece[p] % 16) return K3MOE_ERR_SHAPE;   // the fill copies 16-byte words
            t.piece[p] = piece[p];
            t.expert_bytes += piece[p];
        }
        // the slot arrays, then the tables, each followed by a guard band; the
        // first pass (no base) only measures
        auto carve = [&](char *base) {
            Carve cv{base};
            cv.guards = &t.guards;
            for (int p = 0; p < kTierPieces; p++) t.arr[p] = cv.take<uint8_t>((size_t)slots * piece[p]);
            t.slot_of = cv.take<int>((size_t)c.max_layers * E);
            t.slot_key = cv.take<int>((size_t)slots);
            t.slot_used = cv.take<uint32_t>((size_t)slots);
            t.fill = cv.take<int2>(E);
            t.n_fill = cv.take<int>(1);
            t.stats = cv.take<unsigned long long>(3);
            t.all_ids = cv.take<int>(E + 1);
            return cv.off;
        };
        const size_t bytes = carve(nullptr);
        size_t fr = 0;
        if (free_device_bytes(&fr) != cudaSuccess) return K3MOE_ERR_CUDA;
        if (bytes + (256u << 20) > fr) return K3MOE_ERR_OOM;
        if (cudaMalloc(&t.block, bytes) != cudaSuccess) {
            cudaGetLastError();
            return K3MOE_ERR_OOM;
        }
        try {
            carve((char *)t.block);   // records the guard offsets (host memory)
        } catch (const std::bad_alloc &) {
            cudaFree(t.block);
            return K3MOE_ERR_OOM;
        }
        // every slot free (key -1, stamp 0), no expert resident, counters 0
        if (cudaMemset(t.block, 0, bytes) != cudaSuccess ||
            cudaMemset(t.slot_of, 0xFF, (size_t)c.max_layers * E * 4) != cudaSuccess ||
            cudaMemset(t.slot_key, 0xFF, (size_t)slots * 4) != cudaSuccess ||
            set_guards(t.block, t.guards) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(t.block);
            return K3MOE_ERR_CUDA;
        }
        // K3MOE_TIER_REBASE="at,keep" moves the stamp rebase from its defaults
        // (2^31, 2^24) to small counts, so that a short run goes through it
        if (const char *env = std::getenv("K3MOE_TIER_REBASE")) {
            unsigned long at = 0, keep = 0;
            if (std::sscanf(env, "%lu,%lu", &at, &keep) != 2 || keep < 1 || keep >= at || at > kTierRebaseAt) {
                cudaFree(t.block);
                return K3MOE_ERR_INVALID_ARG;
            }
            t.rebase_at = (uint32_t)at;
            t.rebase_keep = (uint32_t)keep;
        }
        t.slots = slots;
        h->tier = std::move(t);
        if (launch_tier_iota(*h) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            free_tier(h->tier);
            return K3MOE_ERR_CUDA;
        }
        return K3MOE_OK;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_tier_pin_layer(k3moe *h, int layer)
{
    try {
        if (!h || layer < 0 || layer >= h->cfg.max_layers) return K3MOE_ERR_INVALID_ARG;
        TierDev &t = h->tier;
        const int E = h->cfg.n_experts;
        if (t.slots == 0) return K3MOE_ERR_INVALID_ARG;
        LayerDev &w = h->layers[(size_t)layer];
        if (!w.loaded) return K3MOE_ERR_NOT_LOADED;
        if (w.pinned) return K3MOE_OK;
        // every forward of an unpinned layer must still find E free-able slots
        if (t.slots - t.pinned - E < E) return K3MOE_ERR_INVALID_ARG;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        if (launch_tier_plan(*h, layer, 0, true) != cudaSuccess || launch_tier_fill(*h, w, 0) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            return K3MOE_ERR_CUDA;
        }
        int word = 0;
        if (cudaMemcpy(&word, h->ws.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return K3MOE_ERR_CUDA;
        if (word != kErrNone) return K3MOE_ERR_DEVICE;
        t.pinned += E;
        w.pinned = true;
        return K3MOE_OK;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_get_tier_stats(k3moe *h, k3moe_tier_stats *out)
{
    if (!h || !out || out->struct_size != (int32_t)sizeof(k3moe_tier_stats)) return K3MOE_ERR_INVALID_ARG;
    out->slots = h->tier.slots;
    out->hits = out->misses = out->bytes_filled = 0;
    if (h->tier.slots == 0) return K3MOE_OK;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
    unsigned long long v[3] = {0, 0, 0};
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(v, h->tier.stats, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ERR_CUDA;
    }
    out->hits = (int64_t)v[0];
    out->misses = (int64_t)v[1];
    out->bytes_filled = (int64_t)v[2];
    return K3MOE_OK;
}

int k3moe_set_topp(k3moe *h, float p)
{
    if (!h || !(p >= 0.f && p <= 1.f)) return K3MOE_ERR_INVALID_ARG;   // NaN fails too
    h->topp = p;
    return K3MOE_OK;
}

int k3moe_check_wait_timeout(k3moe *h, void *stream)
{
    if (!h) return K3MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
    return launch_wait_check(*h, (cudaStream_t)stream) == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3moe_set_profiling(k3moe *h, int enable)
{
    try {
        if (!h) return K3MOE_ERR_INVALID_ARG;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        h->profiling = enable != 0;
        while (h->profiling && h->event_pool.size() < 512) {   // created outside any timed region
            cudaEvent_t e = nullptr;
            if (cudaEventCreate(&e) != cudaSuccess) return K3MOE_ERR_CUDA;
            h->event_pool.push_back(e);
        }
        return K3MOE_OK;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

int k3moe_profile_read(k3moe *h, k3moe_kernel_stat *out, int max_entries, int *n_entries)
{
    try {
        if (!h || (!out && max_entries > 0)) return K3MOE_ERR_INVALID_ARG;
        if (cudaSetDevice(h->cfg.device) != cudaSuccess) return K3MOE_ERR_CUDA;
        const int rc = harvest(h, true);
        const int n = (int)h->prof_names.size();
        for (int i = 0; i < n && i < max_entries; i++) {
            std::memset(&out[i], 0, sizeof(k3moe_kernel_stat));
            std::strncpy(out[i].name, h->prof_names[(size_t)i].c_str(), sizeof(out[i].name) - 1);
            out[i].launches = h->prof_launches[(size_t)i];
            out[i].total_ms = h->prof_ms[(size_t)i];
        }
        if (n_entries) *n_entries = n;
        h->prof_names.clear();
        h->prof_launches.clear();
        h->prof_ms.clear();
        return rc;
    } catch (...) {   // no C++ exception crosses the C ABI
        return abi_exception();
    }
}

}  // extern "C"
