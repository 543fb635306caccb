/*
 * k3moe: the Kimi K3 LatentMoE routed-expert layer on one GB300 (sm_103a).
 *
 * C ABI of libk3moe.so. Plain pointers and sizes only.
 *
 * What one layer computes (kimi-k3-in-c README, Part II section 9 "Picking 16
 * experts of 896", k3_router and k3_moe; colibri docs/kimi_k3.md, "Stable
 * LatentMoE"), for every token x (a row of x[T, hidden]):
 *   1. router: logit_e = x . Wr_e, sc_e = sigmoid(logit_e), ch_e = sc_e + bias_e;
 *      the topk experts with the largest ch (equal ch: lower id first) are
 *      picked and weighted by their UNBIASED sc, renormalised to sum 1 (when
 *      renorm is set) and multiplied by routed_scale;
 *   2. z = Wdown . x                                   (hidden -> latent);
 *   3. acc = sum_j w_j * W2_e(SiTU(W1_e z, W3_e z))    over the picked experts,
 *      whose weights are MXFP4 (README section 4: e2m1 nibbles, two per byte,
 *      low nibble = even column, bit 3 = sign, one ue8m0 scale per 32 columns,
 *      w = v * 2^(scale - 127)) and are used as stored, never re-encoded;
 *   4. n = RMSNorm(acc) * latent_gain                  (norm of the aggregate);
 *   5. y = Wup . n + Ws2 . SiTU(Ws1 x, Ws3 x)          (shared experts on the
 *      original x, added unweighted);
 *   SiTU(g, u) = b1*tanh(g/b1)*sigmoid(g) * b2*tanh(u/b2).
 *
 * Conventions (taken from the README's engine): refuse rather than guess a
 * missing configuration value; never drop an expert silently; never leave a
 * half-built state behind after an error.
 *
 * All entry points return 0 (K3MOE_OK) or a negative K3MOE_ERR_* code.
 * Errors found on the host are returned immediately. Errors found by a kernel
 * (an index out of range, a bounded wait that ran out) are latched in a device
 * word and returned by k3moe_sync_status, which also reports an overwritten
 * guard band (a write past the end of a library buffer).
 *
 * Device memory: k3moe_create, k3moe_load_layer and k3moe_set_expert_tier
 * check what they need (plus a margin: 64 MB for the workspace, 256 MB for a
 * layer or the tier's slots) against free device memory before allocating,
 * and return K3MOE_ERR_OOM with nothing allocated when it does not fit. The
 * environment variable K3MOE_DEVICE_BUDGET_MB, read at each check, caps the
 * free memory those checks assume at that many megabytes (a budget on a
 * shared GPU).
 *
 * Threading: a handle may be used by one host thread at a time.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3MOE_ABI_VERSION 1

#if defined(__GNUC__)
#define K3MOE_API __attribute__((visibility("default")))
#else
#define K3MOE_API
#endif

enum {
    K3MOE_OK = 0,
    K3MOE_ERR_INVALID_ARG = -1,   /* NULL handle/pointer, bad layer index, T out of range */
    K3MOE_ERR_CONFIG = -2,        /* a configuration field is missing (0), NaN or negative */
    K3MOE_ERR_SHAPE = -3,         /* sizes the kernels do not support (see k3moe_config) */
    K3MOE_ERR_OOM = -4,           /* not enough free device memory; nothing was allocated */
    K3MOE_ERR_BAD_SCALE = -5,     /* an expert holds scale byte 255 (NaN in MX); layer not loaded */
    K3MOE_ERR_NOT_LOADED = -6,    /* forward on a layer that was never loaded */
    K3MOE_ERR_CUDA = -7,          /* a CUDA runtime call failed */
    K3MOE_ERR_TIMEOUT = -8,       /* a device-side bounded wait gave up */
    K3MOE_ERR_DEVICE = -9,        /* a device-side index check failed */
    K3MOE_ERR_GUARD = -10         /* a guard band after a library buffer was overwritten */
};

/* Where the pointees of a k3moe_layer_weights live. */
enum { K3MOE_HOST = 0, K3MOE_DEVICE = 1 };

typedef struct k3moe k3moe;

/* Layer configuration (the MoE fields of the README's K3Cfg). Every field is
 * required: a zero, negative or NaN value returns K3MOE_ERR_CONFIG, except the
 * two flags, which must be 0 or 1.
 * Supported sizes (else K3MOE_ERR_SHAPE): hidden, latent, moe_inter and
 * shared_inter multiples of 64; latent and moe_inter at most 4096;
 * 1 <= topk <= 32; topk <= n_experts <= 1024; max_tokens <= 65536 / topk;
 * max_layers <= 1024 (the model has 93); situ_b1 * situ_b2 <= 512.
 * K3: hidden 7168, latent 3584, n_experts 896, topk 16, moe_inter 3072,
 * shared_inter 6144 (two shared experts fused), rms_eps 1e-5, situ_b1 4,
 * situ_b2 25, routed_scale 1, renorm 1, latent_norm 1.
 * Dense feed-forward layer (the model's layer 0, y = W2 . SiTU(W1 x, W3 x),
 * K3: hidden 7168, width 33792): n_experts, topk, latent and moe_inter all 0,
 * shared_inter the width; load_layer then reads only shared_w1/w3/w2, and the
 * decode kernels must fit the width (else K3MOE_ERR_SHAPE). */
typedef struct {
    uint32_t struct_size;   /* sizeof(k3moe_config), checked */
    int32_t hidden;         /* H: width of x and y */
    int32_t latent;         /* L: expert latent width */
    int32_t n_experts;      /* E: routed experts */
    int32_t topk;           /* k: experts per token */
    int32_t moe_inter;      /* I: routed expert inner width */
    int32_t shared_inter;   /* S: fused shared-expert inner width */
    int32_t max_layers;     /* layers this handle can hold */
    int32_t max_tokens;     /* largest T of one forward (sizes the workspace) */
    int32_t device;         /* CUDA device ordinal */
    int32_t renorm;         /* 1: renormalise the picked weights to sum 1 */
    int32_t latent_norm;    /* 1: RMSNorm the aggregate with latent_gain */
    float rms_eps;          /* eps inside the square root of RMSNorm */
    float situ_b1;          /* SiTU gate cap */
    float situ_b2;          /* SiTU up cap */
    float routed_scale;     /* multiplies the routed weights */
} k3moe_config;

/* One layer's weights in the checkpoint layout (row = output, row-major).
 * bf16 tensors are raw bfloat16 bit patterns. The six expert arrays hold one
 * pointer per expert (E entries each; the arrays themselves are host memory);
 * the pointees, like every other pointer here, live where `where` says.
 * Bytes are copied unchanged into library-owned device memory (with the
 * expert tier on, the expert arrays into library-owned pinned host memory). */
typedef struct {
    uint32_t struct_size;          /* sizeof(k3moe_layer_weights), checked */
    int32_t where;                 /* K3MOE_HOST or K3MOE_DEVICE */
    const void *router_w;          /* bf16 [E, H] */
    const float *router_bias;      /* fp32 [E]; NULL means no bias */
    const void *down_w;            /* bf16 [L, H] */
    const void *up_w;              /* bf16 [H, L] */
    const void *latent_gain;       /* bf16 [L]; required when latent_norm = 1 */
    const void *shared_w1;         /* bf16 [S, H] (gate) */
    const void *shared_w3;         /* bf16 [S, H] (up) */
    const void *shared_w2;         /* bf16 [H, S] */
    const uint8_t *const *w1_packed;  /* [E] -> [I, L/2] e2m1 pairs (gate) */
    const uint8_t *const *w1_scale;   /* [E] -> [I, L/32] ue8m0 */
    const uint8_t *const *w3_packed;  /* [E] -> [I, L/2] (up) */
    const uint8_t *const *w3_scale;   /* [E] -> [I, L/32] */
    const uint8_t *const *w2_packed;  /* [E] -> [L, I/2] (down, back to the latent) */
    const uint8_t *const *w2_scale;   /* [E] -> [L, I/32] */
} k3moe_layer_weights;

/* Creates a handle on cfg->device and allocates its workspace (sized by
 * max_tokens). On error *out is NULL and nothing stays allocated. */
K3MOE_API int k3moe_create(const k3moe_config *cfg, k3moe **out);

/* Copies one layer's weights to the device (synchronous). Free device memory
 * is checked against the whole layer before anything is allocated
 * (K3MOE_ERR_OOM). Every scale byte is checked: 255 returns
 * K3MOE_ERR_BAD_SCALE and the layer stays unloaded. Reloading a slot replaces
 * it (and drops its post-norm gain and tier pin). layer is in [0, max_layers).
 * With the expert tier on, the expert arrays go to pinned host memory instead
 * (K3MOE_ERR_OOM when it cannot be pinned). */
K3MOE_API int k3moe_load_layer(k3moe *h, int layer, const k3moe_layer_weights *w);

/* One layer on T tokens: x [T, H] bf16 -> y [T, H] bf16, both device pointers,
 * 16-byte aligned (the kernels move activations in 16-byte vectors), not
 * overlapping; K3MOE_ERR_INVALID_ARG otherwise. Asynchronous on `stream` (a cudaStream_t; NULL
 * is the legacy default stream). 1 <= T <= max_tokens. The routing of the
 * call stays readable through k3moe_get_routing until the next forward. */
K3MOE_API int k3moe_forward(k3moe *h, int layer, const void *x, void *y, int T, void *stream);

/* Layers first_layer .. first_layer + n_layers - 1 applied in sequence, with
 * x_next = bf16(RMSNorm(y) with unit gain and rms_eps) between two layers.
 * x, y: device [T, H] bf16, aligned and disjoint as for k3moe_forward. The
 * routing of the last layer stays readable. */
K3MOE_API int k3moe_forward_chain(k3moe *h, int first_layer, int n_layers, const void *x, void *y,
                        int T, void *stream);

/* k3moe_forward with HOST buffers: copies x to the device, runs the layer,
 * copies y back and synchronises `stream`. Pinned host memory is faster but
 * not required; a pinned (device-mapped), 16-byte aligned y is written in
 * place by the layer's last kernel, without a copy back. Host pointers need
 * no alignment. */
K3MOE_API int k3moe_forward_host(k3moe *h, int layer, const void *x_host, void *y_host, int T,
                       void *stream);

/* Copies the routing of the last forward into caller-owned device buffers
 * (any may be NULL), asynchronously on `stream`:
 *   ids [T, k] int32 and w [T, k] fp32, slot j in descending ch order (with
 *   the top-p cut: the kept picks first, then id -1 / weight 0);
 *   counts [E] int32; offsets [E+1] int32 (exclusive prefix sum of counts);
 *   perm [T*k] int32: flat pair indices t*k+j grouped by expert (ascending),
 *   and by ascending token inside an expert (the first offsets[E] entries).
 * A dense feed-forward layer has no routing (zero-size tables). */
K3MOE_API int k3moe_get_routing(k3moe *h, int32_t *ids, float *w, int32_t *counts, int32_t *offsets,
                      int32_t *perm, void *stream);

/* ---- Forward from the residual stream -------------------------------------------
 * In the model the layer's input is the decoder's residual stream h after the
 * RMSNorm in front of the MoE (kimi-k3-in-c README, Part II, the decoder layer
 * applies its post_norm to h and hands the result to k3_moe; k3_rmsnorm in
 * section 5: x = h * inv * gain, inv = 1/sqrt(mean(h^2) + eps) with the squares
 * summed in double).
 *
 * k3moe_load_post_norm attaches that norm's gain (bf16 [hidden], host or
 * device memory as `where` says) to a loaded layer; loading the layer again
 * drops it. K3MOE_ERR_NOT_LOADED when the layer is not loaded.
 *
 * k3moe_forward_residual takes h_in fp32 [T, hidden] (device memory, 16-byte
 * aligned, as y must be), forms x = bf16(RMSNorm(h_in) * gain) per token (rms_eps of the
 * configuration) and runs the layer on x as k3moe_forward does. At T <= 2 the
 * norm runs inside the first two kernels of the layer (x never goes to
 * memory); otherwise a first kernel writes x to the workspace. The x used can
 * be read back with k3moe_get_intermediate(K3MOE_T_X). Errors as
 * k3moe_forward, and K3MOE_ERR_NOT_LOADED when the layer has no post-norm
 * gain. */
K3MOE_API int k3moe_load_post_norm(k3moe *h, int layer, const void *gain, int where);
K3MOE_API int k3moe_forward_residual(k3moe *h, int layer, const float *h_in, void *y, int T,
                                     void *stream);

/* Intermediates of the last forward, for parity diagnosis. Copies `bytes`
 * bytes (at most the tensor's size for the last T) into caller device memory.
 *   K3MOE_T_Z       fp32 [T, L]   latent down projection
 *   K3MOE_T_ACC     fp32 [T, L]   weighted sum of expert outputs (before the norm)
 *   K3MOE_T_SHARED  fp32 [T, S]   SiTU of the shared experts
 *   K3MOE_T_LOGITS  fp32 [T, E]   router logits
 *   K3MOE_T_X       bf16 [T, H]   the layer input that k3moe_forward_residual made
 *                                 (K3MOE_ERR_INVALID_ARG after any other forward) */
enum { K3MOE_T_Z = 1, K3MOE_T_ACC = 2, K3MOE_T_SHARED = 3, K3MOE_T_LOGITS = 4, K3MOE_T_X = 5 };
K3MOE_API int k3moe_get_intermediate(k3moe *h, int which, void *dst, size_t bytes, void *stream);

/* Synchronises the device and returns (then clears) the first latched
 * device-side error, or the first asynchronous CUDA error. It then reads the
 * guard bands (256 bytes of a fixed pattern after every workspace and tier
 * buffer the kernels write): K3MOE_ERR_GUARD when one has changed, i.e. a
 * kernel wrote past the end of a buffer (the handle should then be
 * destroyed). */
K3MOE_API int k3moe_sync_status(k3moe *h);

/* Check of the device-side failure path (the README's engine reports a
 * failed step by its exit code rather than hanging or returning a half-done
 * result; kimi-k3-in-c README, "Exit codes"). Launches on `stream` one
 * single-thread kernel whose wait on a barrier that nothing completes runs
 * out after the same bounded limit (about two seconds) as every wait in the
 * layer's kernels; it latches the time-out, so the next k3moe_sync_status
 * returns K3MOE_ERR_TIMEOUT and clears it. Nothing faults, traps or hangs;
 * the handle and its loaded layers stay usable. Errors: K3MOE_ERR_INVALID_ARG
 * (NULL handle), K3MOE_ERR_CUDA (the launch failed). */
K3MOE_API int k3moe_check_wait_timeout(k3moe *h, void *stream);

/* Which routed-expert kernels a forward uses (same arithmetic, kimi-k3-in-c
 * README, Part II section 9, k3_moe step 3; results agree to fp32 rounding
 * order and fp16 operand rounding):
 *   K3MOE_EXPERT_AUTO  (default) a grouped tensor-core GEMM when the batch
 *                      holds at least 128 (token, expert) pairs and T >= 16,
 *                      else the per-pair GEMVs; the grouped GEMM is the
 *                      block-scaled one (K3MOE_EXPERT_MX) while the experts
 *                      see fewer than 64 pairs each on average, else the f16
 *                      one (K3MOE_EXPERT_GEMM);
 *   K3MOE_EXPERT_GEMV  always the per-pair GEMVs (streaming dequantisation);
 *   K3MOE_EXPERT_GEMM  the grouped GEMM with f16 operands (the nibbles and
 *                      activations widened on the SM) whenever T * topk >= 128
 *                      (below that the GEMVs run: its n-tile needs 128 pair
 *                      rows);
 *   K3MOE_EXPERT_MX    every batch on the grouped GEMM of the block-scaled
 *                      tensor cores (tcgen05 kind::mxf8f6f4): the stored e2m1
 *                      weights and their ue8m0 scales go to the tensor core as
 *                      they are, against activations in two-term MXFP8 (hi +
 *                      lo e4m3 with a ue8m0 scale per 32, about 12 significant
 *                      bits); every scale byte is applied exactly, whatever a
 *                      row's scale range. Below 128 pairs each work item's K
 *                      range may be split over several items (partial sums
 *                      meet in device memory); at decode sizes this is slower
 *                      than the GEMVs, which is why the automatic choice keeps
 *                      them there.
 * Both grouped GEMMs need latent and moe_inter to be multiples of 128; the f16
 * one also needs max_tokens * topk >= 128. Asking for K3MOE_EXPERT_GEMM or
 * K3MOE_EXPERT_MX on a handle whose shape does not allow it returns
 * K3MOE_ERR_SHAPE and leaves the mode as it was. Returns K3MOE_ERR_INVALID_ARG for an unknown mode. Takes
 * effect at the next forward; not thread-safe with a forward on the same
 * handle. */
enum { K3MOE_EXPERT_AUTO = 0, K3MOE_EXPERT_GEMV = 1, K3MOE_EXPERT_GEMM = 2, K3MOE_EXPERT_MX = 3 };
K3MOE_API int k3moe_set_expert_path(k3moe *h, int mode);

/* ---- Expert tier: host memory holds the routed experts, device slots cache them
 * (kimi-k3-in-c README, Part II section 12, "An LRU cache for the experts";
 * host memory over NVLink-C2C takes the place of the pages' disk, device
 * memory that of their RAM). For a pool of layers whose routed experts do not
 * all fit in device memory.
 *
 * k3moe_set_expert_tier must come before the first k3moe_load_layer. With
 * slots > 0, every layer loaded afterwards keeps its routed-expert tensors
 * (packed nibbles, scales, and the largest scale byte of each row) in one
 * pinned, device-mapped host block that the library allocates and owns; its
 * router, projections and shared experts stay in device memory. The handle
 * keeps `slots` expert slots in device memory (slots * ~17.56 MB at K3 size),
 * shared by all layers. Every forward, after routing, one kernel stamps the
 * slots of the touched experts already resident (hits) and gives each other
 * touched expert (miss) a slot that this forward does not use: a free one
 * first, else the one used longest ago (equal age: the lower slot); a second
 * kernel copies the missed experts from the host block into their slots; the
 * expert kernels then read the slots. The host takes no part (no
 * synchronisation, no copy calls). Results are those of the resident layer.
 * Ages are 32-bit stamps kept by the host and passed to each forward's plan:
 * a tiered forward must be launched, not replayed from a captured CUDA
 * graph. Once the count reaches 2^31 a small kernel shifts the slots' stamps
 * down, keeping the order of the last 2^24 (older slots tie, the lower slot
 * going first); the environment variable K3MOE_TIER_REBASE="at,keep", read
 * here, moves those two counts (1 <= keep < at <= 2^31; else
 * K3MOE_ERR_INVALID_ARG) so that a short run goes through the shift.
 * slots must be >= n_experts (the most one forward touches) and <= 16384;
 * slots = 0 turns the tier off. Reloading a tiered layer frees its slots.
 * Errors: K3MOE_ERR_INVALID_ARG (NULL handle, a layer already loaded, slots
 * out of range), K3MOE_ERR_SHAPE (an expert array of a size not a multiple of
 * 16 bytes), K3MOE_ERR_OOM (the slots do not fit in free device memory; a
 * later load_layer returns it when the host block cannot be pinned),
 * K3MOE_ERR_CUDA. */
K3MOE_API int k3moe_set_expert_tier(k3moe *h, int slots);

/* Pins a loaded layer's routed experts in the tier (the pages' pinned slots,
 * which eviction skips): all n_experts of the layer are copied into slots now
 * (counted as misses) and stay there; its forwards only hit. Synchronous.
 * Needs slots >= (pinned layers + 2) * n_experts, so that any other layer's
 * forward still fits; pinning a pinned layer again does nothing; loading the
 * layer again unpins it. Errors: K3MOE_ERR_INVALID_ARG (no tier, bad layer,
 * too few slots), K3MOE_ERR_NOT_LOADED, K3MOE_ERR_DEVICE, K3MOE_ERR_CUDA. */
K3MOE_API int k3moe_tier_pin_layer(k3moe *h, int layer);

typedef struct {
    int32_t struct_size;    /* sizeof(k3moe_tier_stats), set by the caller */
    int32_t slots;          /* 0: tier off */
    int64_t hits;           /* touched experts found resident, summed over forwards */
    int64_t misses;         /* touched experts copied in */
    int64_t bytes_filled;   /* bytes those copies moved from host to device memory */
} k3moe_tier_stats;
/* Synchronises the device and reads the tier's counters (cumulative since
 * k3moe_set_expert_tier). K3MOE_ERR_INVALID_ARG for NULL or a wrong struct_size. */
K3MOE_API int k3moe_get_tier_stats(k3moe *h, k3moe_tier_stats *out);

/* ---- Dropping the low-weight tail of the picks --------------------------------------
 * The pages' optional K3_TOPP (kimi-k3-in-c README, run-time options): of the
 * topk picks of a token, keep only those up to cumulative weight p and
 * renormalise. In weight order (larger first, equal weights: lower id first)
 * a pick is kept while the sum of the weights before it is below p times the
 * total of all picks; the kept weights are scaled back to that total (with
 * renorm: the kept unbiased scores renormalised, times routed_scale). The
 * first pick is always kept. Dropped picks are never read: the experts they
 * would have touched are skipped. k3moe_get_routing then returns, per token,
 * the kept picks first (selection order) and -1 with weight 0 in the dropped
 * slots; counts, offsets and perm cover the kept pairs only. p = 0 (the
 * default) keeps all topk; with p = 1 only picks of zero weight at the end of
 * the weight order drop. K3MOE_ERR_INVALID_ARG outside [0, 1] or NaN.
 * Takes effect at the next forward. This changes what the layer computes: the
 * pages ask for an accuracy check of any p first. */
K3MOE_API int k3moe_set_topp(k3moe *h, float p);

/* Per-kernel timing: with profiling on, every kernel a forward launches is
 * bracketed by CUDA events on the launching stream. k3moe_profile_read
 * synchronises, aggregates per kernel name and resets the record. */
typedef struct {
    char name[48];        /* kernel name */
    int32_t launches;     /* launches recorded */
    double total_ms;      /* sum of event-timed durations */
} k3moe_kernel_stat;
K3MOE_API int k3moe_set_profiling(k3moe *h, int enable);
K3MOE_API int k3moe_profile_read(k3moe *h, k3moe_kernel_stat *out, int max_entries, int *n_entries);

/* Frees every device allocation of the handle. NULL is ignored. */
K3MOE_API void k3moe_destroy(k3moe *h);

/* Static description of a return code. */
K3MOE_API const char *k3moe_strerror(int code);

/* K3MOE_ABI_VERSION of the library. */
K3MOE_API int k3moe_abi_version(void);

/* ---- Router without allocation ------------------------------------------------
 * The pages describe no such call; it exists for callers that may not
 * allocate device memory (a plugin whose host framework owns every device
 * buffer through its own pool, or a serving loop that forbids allocation
 * after start-up). It needs no handle and calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * Computes the router step of the layer for T tokens on the CURRENT device:
 * logit = x . Wr_e, sc = sigmoid(logit), ch = sc + bias_e; the topk experts
 * with the largest ch (equal ch: lower id first) go to ids [T, topk] int32 in
 * descending ch order, their sc (renormalised to sum 1 when renorm = 1, then
 * times routed_scale) to w [T, topk] fp32. x [T, hidden] and router_w
 * [n_experts, hidden] are bf16, router_bias [n_experts] fp32 or NULL; all
 * pointers are device memory owned by the caller. Asynchronous on `stream`.
 *
 * Scratch: the [T, n_experts] fp32 logits live in one static device array of
 * K3MOE_ROUTE_STATIC_MAX_LOGITS floats (4 MiB) that every GPU loading this
 * library keeps until the process exits. T * n_experts above that limit
 * returns K3MOE_ERR_SHAPE. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture. The address is cached for the life of the process and does
 * not follow a cudaDeviceReset: make no further call on a device after
 * resetting it. All calls share the array, so calls that overlap on the GPU
 * (other streams or host threads) race on it; nothing in it needs to start at
 * zero. A NaN score (from NaN or infinite inputs) ranks below every finite
 * one; the ids stay a set of distinct experts, the weights are then
 * undefined. Errors: K3MOE_ERR_INVALID_ARG (NULL pointer, x or router_w not
 * on a 16-byte boundary, T < 1, hidden not a positive multiple of 8; nothing
 * is launched), K3MOE_ERR_CONFIG (renorm not 0/1, routed_scale not finite and
 * > 0), K3MOE_ERR_SHAPE (topk not in [1, 32], topk > n_experts, n_experts >
 * 1024, or the size limit), K3MOE_ERR_CUDA (address lookup or launch
 * failed). */
#define K3MOE_ROUTE_STATIC_MAX_LOGITS (1u << 20)
K3MOE_API int k3moe_route_static(const void *x, const void *router_w, const float *router_bias,
                                 int T, int hidden, int n_experts, int topk, int renorm,
                                 float routed_scale, int32_t *ids, float *w, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* K3MOE_H */
