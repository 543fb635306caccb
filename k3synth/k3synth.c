/*
 * k3synth: seeded, counter-based synthetic inputs for the K3 LatentMoE layer.
 *
 * This file draws random numbers and nothing else. It holds none of the
 * layer's arithmetic (no router, no MXFP4 decode, no SiTU, no norm): it only
 * fills buffers with bytes, uniform integers and approximately normal values,
 * so that the CPU oracle and the CUDA library can be fed the same inputs.
 *
 * Generator: word i of a stream with key K is SplitMix64's output function
 * (Steele, Lea and Flood, "Fast Splittable Pseudorandom Number Generators",
 * OOPSLA 2014) applied to the counter K + (i+1)*golden_gamma. A stream key is
 * built by feeding (seed, part0, part1, ...) through the same mixer. Every
 * value therefore depends only on (key, index): fills are reproducible at any
 * thread count and on any host.
 *
 * Normal values use the Irwin-Hall construction (the sum of twelve uniforms,
 * minus six), evaluated in integer arithmetic and scaled by a power of two,
 * so no libm call is involved and the bits are identical on x86-64 and
 * aarch64. Its tails stop at +-6 sigma.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define K3S_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t k3s_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t k3s_word(uint64_t key, uint64_t i)
{
    return k3s_mix(key + (i + 1) * K3S_GAMMA);
}

/* Stream key from a seed and up to four parts (tensor id, layer, expert, ...). */
uint64_t k3s_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c, uint64_t d)
{
    uint64_t k = k3s_mix(seed + K3S_GAMMA);
    k = k3s_mix(k ^ (a + 0x1000193ULL));
    k = k3s_mix(k ^ (b + 0x2000391ULL));
    k = k3s_mix(k ^ (c + 0x3000607ULL));
    k = k3s_mix(k ^ (d + 0x4000949ULL));
    return k;
}

/* Irwin-Hall(12): twelve 16-bit uniforms from three words. The result is
 * (S - 393210) / 65536 with S the sum of the twelve draws, exactly
 * representable in a double; its mean is 0 and its variance 1 - 1/65536^2. */
static inline double k3s_normal(uint64_t key, uint64_t i)
{
    uint64_t s = 0;
    for (int w = 0; w < 3; w++) {
        uint64_t v = k3s_word(key, 3 * i + (uint64_t)w);
        s += (v & 0xFFFF) + ((v >> 16) & 0xFFFF) + ((v >> 32) & 0xFFFF) + (v >> 48);
    }
    return ((double)(int64_t)s - 393210.0) * (1.0 / 65536.0);
}

/* float -> bfloat16 bits, round to nearest even (NaN kept quiet). */
static inline uint16_t k3s_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

#define K3S_PAR_MIN (1u << 16)

/* out[i] = bf16(mean + sigma * N_i), i in [0, n). */
void k3s_fill_normal_bf16(uint16_t *out, size_t n, uint64_t key, double mean, double sigma)
{
#pragma omp parallel for schedule(static) if (n > K3S_PAR_MIN)
    for (size_t i = 0; i < n; i++)
        out[i] = k3s_f32_to_bf16((float)(mean + sigma * k3s_normal(key, i)));
}

/* out[i] = float(mean + sigma * N_i). */
void k3s_fill_normal_f32(float *out, size_t n, uint64_t key, double mean, double sigma)
{
#pragma omp parallel for schedule(static) if (n > K3S_PAR_MIN)
    for (size_t i = 0; i < n; i++)
        out[i] = (float)(mean + sigma * k3s_normal(key, i));
}

/* out[i] = mean + sigma * N_i in double (for inputs that are built on further
 * before rounding, e.g. the covering construction). */
void k3s_fill_normal_f64(double *out, size_t n, uint64_t key, double mean, double sigma)
{
#pragma omp parallel for schedule(static) if (n > K3S_PAR_MIN)
    for (size_t i = 0; i < n; i++)
        out[i] = mean + sigma * k3s_normal(key, i);
}

/* Uniform random bytes: byte i is byte (i % 8) of word i / 8, little-endian. */
void k3s_fill_bytes(uint8_t *out, size_t n, uint64_t key)
{
    const size_t nw = n / 8;
#pragma omp parallel for schedule(static) if (nw > K3S_PAR_MIN)
    for (size_t w = 0; w < nw; w++) {
        uint64_t v = k3s_word(key, w);
        for (int b = 0; b < 8; b++) out[8 * w + (size_t)b] = (uint8_t)(v >> (8 * b));
    }
    if (n % 8) {
        uint64_t v = k3s_word(key, nw);
        for (size_t b = 0; b < n % 8; b++) out[8 * nw + b] = (uint8_t)(v >> (8 * b));
    }
}

/* Uniform integers in [lo, hi] (inclusive) stored as bytes. Value i uses the
 * 16-bit chunk i % 4 of word i / 4, mapped by (chunk * range) >> 16. */
void k3s_fill_uniform_u8(uint8_t *out, size_t n, uint64_t key, int lo, int hi)
{
    const uint32_t range = (uint32_t)(hi - lo + 1);
#pragma omp parallel for schedule(static) if (n > K3S_PAR_MIN)
    for (size_t i = 0; i < n; i++) {
        uint64_t v = k3s_word(key, i / 4);
        uint32_t chunk = (uint32_t)((v >> (16 * (i % 4))) & 0xFFFF);
        out[i] = (uint8_t)(lo + (int)((chunk * range) >> 16));
    }
}

/* Uniform 64-bit words (for shuffles and index draws done by the caller). */
void k3s_fill_words(uint64_t *out, size_t n, uint64_t key)
{
#pragma omp parallel for schedule(static) if (n > K3S_PAR_MIN)
    for (size_t i = 0; i < n; i++) out[i] = k3s_word(key, i);
}

/* Expert tensors: expert e of `n_experts` gets its own stream
 * k3s_key(seed, tensor, layer, e, 0), so any single expert can be regenerated
 * alone. mode 0: uniform bytes; mode 1: uniform integers in [lo, hi]. */
void k3s_fill_experts(uint8_t *out, int n_experts, size_t n_per_expert, uint64_t seed,
                      uint64_t tensor, uint64_t layer, int mode, int lo, int hi)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < n_experts; e++) {
        uint8_t *o = out + (size_t)e * n_per_expert;
        const uint64_t key = k3s_key(seed, tensor, layer, (uint64_t)e, 0);
        if (mode == 0) {
            const size_t nw = n_per_expert / 8;
            for (size_t w = 0; w < nw; w++) {
                uint64_t v = k3s_word(key, w);
                uint8_t b8[8];
                for (int b = 0; b < 8; b++) b8[b] = (uint8_t)(v >> (8 * b));
                memcpy(o + 8 * w, b8, 8);
            }
            if (n_per_expert % 8) {
                uint64_t v = k3s_word(key, nw);
                for (size_t b = 0; b < n_per_expert % 8; b++) o[8 * nw + b] = (uint8_t)(v >> (8 * b));
            }
        } else {
            const uint32_t range = (uint32_t)(hi - lo + 1);
            for (size_t w = 0; 4 * w < n_per_expert; w++) {
                const uint64_t v = k3s_word(key, w);
                for (size_t c = 0; c < 4 && 4 * w + c < n_per_expert; c++) {
                    uint32_t chunk = (uint32_t)((v >> (16 * c)) & 0xFFFF);
                    o[4 * w + c] = (uint8_t)(lo + (int)((chunk * range) >> 16));
                }
            }
        }
    }
}

/* Token rows: row t of a [T, width] bf16 matrix of N(mean, sigma) values, with
 * its own stream k3s_key(seed, tensor, stream, t, attempt[t]). A caller that
 * needs to replace one token (for instance to move it away from a routing
 * near-tie) bumps that token's attempt counter and regenerates. */
void k3s_fill_token_rows_bf16(uint16_t *out, int T, int width, uint64_t seed, uint64_t tensor,
                              uint64_t stream, const int32_t *attempt, double mean, double sigma)
{
#pragma omp parallel for schedule(static) if (T > 8)
    for (int t = 0; t < T; t++) {
        const uint64_t key = k3s_key(seed, tensor, stream, (uint64_t)t,
                                     attempt ? (uint64_t)attempt[t] : 0);
        uint16_t *o = out + (size_t)t * (size_t)width;
        for (int i = 0; i < width; i++)
            o[i] = k3s_f32_to_bf16((float)(mean + sigma * k3s_normal(key, (uint64_t)i)));
    }
}

/* Same rows in double, before any rounding. */
void k3s_fill_token_rows_f64(double *out, int T, int width, uint64_t seed, uint64_t tensor,
                             uint64_t stream, const int32_t *attempt, double mean, double sigma)
{
#pragma omp parallel for schedule(static) if (T > 8)
    for (int t = 0; t < T; t++) {
        const uint64_t key = k3s_key(seed, tensor, stream, (uint64_t)t,
                                     attempt ? (uint64_t)attempt[t] : 0);
        double *o = out + (size_t)t * (size_t)width;
        for (int i = 0; i < width; i++) o[i] = mean + sigma * k3s_normal(key, (uint64_t)i);
    }
}

/* double -> bf16 bits through float, both steps round-to-nearest-even. */
void k3s_round_bf16(uint16_t *out, const double *in, size_t n)
{
#pragma omp parallel for schedule(static) if (n > K3S_PAR_MIN)
    for (size_t i = 0; i < n; i++) out[i] = k3s_f32_to_bf16((float)in[i]);
}
