"""Seeded synthetic inputs for the K3 LatentMoE layer.

Both sides of every comparison draw their inputs from here: the CPU oracle
(tests, the CPU baseline) and the CUDA library (tests, bench.py). The module
fills arrays with random bytes, uniform integers and approximately normal
values from a counter-based generator (``k3synth.c``) and lays them out in the
checkpoint's shapes. It holds none of the layer's arithmetic.

Layer shapes and value distributions follow the workloads the pages name for
the Kimi K3 "Stable LatentMoE" block (kimi-k3-in-c README, Part II section 9
"Picking 16 experts of 896"; colibri "docs/kimi_k3.md", "Model" list):
hidden 7168, latent 3584, 896 routed experts, top-16, expert inter 3072, two
shared experts fused to inter 6144, MXFP4 experts with one ue8m0 scale per 32
columns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3synth.c")
_LIB_PATH = os.path.join(_HERE, "libk3synth.so")
_lib = None

# Tensor ids used in stream keys. They only name streams; changing one changes
# every generated value of that tensor.
TX, TROUTER, TBIAS, TDOWN, TUP, TGAIN, TSH1, TSH3, TSH2 = 1, 2, 3, 4, 5, 6, 7, 8, 9
TW1P, TW1S, TW3P, TW3S, TW2P, TW2S = 10, 11, 12, 13, 14, 15
TPERM, TCOVER = 16, 17
TRESID, TRESID_SCALE, TPOSTGAIN = 18, 19, 20
TD1, TD3, TD2 = 21, 22, 23

MXFP4_GROUP = 32


def build(force: bool = False, out: str | None = None, flags=("-O2",)) -> str:
    """Compile the generator to `out` (default: libk3synth.so next to its
    source; atomic rename, so parallel builders never see a half-written file).
    K3SYNTH_LIB names an already built library to load instead."""
    if out is None and os.environ.get("K3SYNTH_LIB"):
        return os.environ["K3SYNTH_LIB"]
    out = out or _LIB_PATH
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    try:
        subprocess.check_call(["gcc", *flags, "-std=c99", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, sz, p = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
        lib.k3s_key.restype = u64
        lib.k3s_key.argtypes = [u64] * 5
        lib.k3s_fill_normal_bf16.argtypes = [p, sz, u64, ctypes.c_double, ctypes.c_double]
        lib.k3s_fill_normal_f32.argtypes = [p, sz, u64, ctypes.c_double, ctypes.c_double]
        lib.k3s_fill_normal_f64.argtypes = [p, sz, u64, ctypes.c_double, ctypes.c_double]
        lib.k3s_fill_bytes.argtypes = [p, sz, u64]
        lib.k3s_fill_uniform_u8.argtypes = [p, sz, u64, ctypes.c_int, ctypes.c_int]
        lib.k3s_fill_words.argtypes = [p, sz, u64]
        lib.k3s_fill_experts.argtypes = [p, ctypes.c_int, sz, u64, u64, u64,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.k3s_fill_token_rows_bf16.argtypes = [p, ctypes.c_int, ctypes.c_int, u64, u64, u64,
                                                 p, ctypes.c_double, ctypes.c_double]
        lib.k3s_fill_token_rows_f64.argtypes = [p, ctypes.c_int, ctypes.c_int, u64, u64, u64,
                                                p, ctypes.c_double, ctypes.c_double]
        lib.k3s_round_bf16.argtypes = [p, p, sz]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def key(seed: int, a: int = 0, b: int = 0, c: int = 0, d: int = 0) -> int:
    return int(_L().k3s_key(seed, a, b, c, d))


def normal_bf16(shape, k: int, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _L().k3s_fill_normal_bf16(_ptr(out), out.size, k, mean, sigma)
    return out


def normal_f32(shape, k: int, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().k3s_fill_normal_f32(_ptr(out), out.size, k, mean, sigma)
    return out


def normal_f64(shape, k: int, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _L().k3s_fill_normal_f64(_ptr(out), out.size, k, mean, sigma)
    return out


def uniform_bytes(shape, k: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint8)
    _L().k3s_fill_bytes(_ptr(out), out.size, k)
    return out


def uniform_u8(shape, k: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint8)
    _L().k3s_fill_uniform_u8(_ptr(out), out.size, k, lo, hi)
    return out


def words(n: int, k: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _L().k3s_fill_words(_ptr(out), n, k)
    return out


def round_bf16(a: np.ndarray) -> np.ndarray:
    """double -> bf16 bits (through float32, both steps round-to-nearest-even)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _L().k3s_round_bf16(_ptr(out), _ptr(a), a.size)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a 16-bit left shift)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Shape:
    """Sizes of one LatentMoE layer (notation of the pages' K3Cfg)."""
    hidden: int
    latent: int
    n_experts: int
    topk: int
    moe_inter: int
    shared_inter: int
    rms_eps: float = 1e-5
    situ_b1: float = 4.0
    situ_b2: float = 25.0
    routed_scale: float = 1.0
    renorm: int = 1
    topp: float = 0.0      # cumulative-weight cut of the picks (0: off)

    @property
    def expert_bytes(self) -> int:
        L, I = self.latent, self.moe_inter
        return 2 * (I * L // 2 + I * L // MXFP4_GROUP) + (L * I // 2 + L * I // MXFP4_GROUP)


# Kimi K3 layer (K3Cfg values printed in the pages' config section).
K3 = Shape(hidden=7168, latent=3584, n_experts=896, topk=16, moe_inter=3072, shared_inter=6144)
# The small layer the oracle runs in well under a second.
TINY = Shape(hidden=256, latent=128, n_experts=32, topk=4, moe_inter=128, shared_inter=256)
# The model's dense feed-forward layer 0: hidden 7168, dense_inter 33792.
K3_DENSE = Shape(hidden=7168, latent=0, n_experts=0, topk=0, moe_inter=0, shared_inter=33792)


@dataclass(frozen=True)
class WeightRecipe:
    """Value distributions of one synthetic layer."""
    dense_sigma: float = 0.02      # router, down, up and shared weights: N(0, sigma) -> bf16
    bias_sigma: float = 0.1        # score-correction bias: N(0, sigma) fp32
    gain_sigma: float = 0.1        # latent RMSNorm gain: 1 + N(0, sigma) -> bf16
    scale_lo: int = 117            # ue8m0 scale bytes: uniform integers in [lo, hi]
    scale_hi: int = 123
    zero_bias: bool = False        # bias all zeros (covering construction)


TINY_RECIPE = WeightRecipe(scale_lo=118, scale_hi=124)
K3_RECIPE = WeightRecipe(scale_lo=117, scale_hi=123)


def make_layer(shape: Shape, seed: int, layer: int = 0,
               recipe: WeightRecipe = K3_RECIPE) -> dict:
    """All tensors of one layer, in the checkpoint layout (row = output):

    router_w [E,H] bf16, router_bias [E] f32, down_w [L,H] bf16, up_w [H,L] bf16,
    latent_gain [L] bf16, sh_w1/sh_w3 [S,H] bf16, sh_w2 [H,S] bf16,
    w1p/w3p [E,I,L/2] u8 with w1s/w3s [E,I,L/32] u8, w2p [E,L,I/2] u8 with w2s [E,L,I/32] u8.
    bf16 tensors are uint16 bit patterns.
    """
    H, L, E, I, S = shape.hidden, shape.latent, shape.n_experts, shape.moe_inter, shape.shared_inter
    r = recipe
    d = {}
    d["router_w"] = normal_bf16((E, H), key(seed, TROUTER, layer), 0.0, r.dense_sigma)
    d["router_bias"] = (np.zeros(E, np.float32) if r.zero_bias
                        else normal_f32((E,), key(seed, TBIAS, layer), 0.0, r.bias_sigma))
    d["down_w"] = normal_bf16((L, H), key(seed, TDOWN, layer), 0.0, r.dense_sigma)
    d["up_w"] = normal_bf16((H, L), key(seed, TUP, layer), 0.0, r.dense_sigma)
    d["latent_gain"] = normal_bf16((L,), key(seed, TGAIN, layer), 1.0, r.gain_sigma)
    d["sh_w1"] = normal_bf16((S, H), key(seed, TSH1, layer), 0.0, r.dense_sigma)
    d["sh_w3"] = normal_bf16((S, H), key(seed, TSH3, layer), 0.0, r.dense_sigma)
    d["sh_w2"] = normal_bf16((H, S), key(seed, TSH2, layer), 0.0, r.dense_sigma)
    lib = _L()

    def experts(shape3, tensor, mode):
        out = np.empty(shape3, dtype=np.uint8)
        per = int(np.prod(shape3[1:]))
        lib.k3s_fill_experts(_ptr(out), E, per, seed, tensor, layer, mode, r.scale_lo, r.scale_hi)
        return out

    G = MXFP4_GROUP
    d["w1p"] = experts((E, I, L // 2), TW1P, 0)
    d["w1s"] = experts((E, I, L // G), TW1S, 1)
    d["w3p"] = experts((E, I, L // 2), TW3P, 0)
    d["w3s"] = experts((E, I, L // G), TW3S, 1)
    d["w2p"] = experts((E, L, I // 2), TW2P, 0)
    d["w2s"] = experts((E, L, I // G), TW2S, 1)
    return d


def make_router(shape: Shape, seed: int, layer: int = 0,
                recipe: WeightRecipe = K3_RECIPE) -> dict:
    """Only the router tensors of make_layer (same streams, same values)."""
    E, H = shape.n_experts, shape.hidden
    return {"router_w": normal_bf16((E, H), key(seed, TROUTER, layer), 0.0, recipe.dense_sigma),
            "router_bias": (np.zeros(E, np.float32) if recipe.zero_bias
                            else normal_f32((E,), key(seed, TBIAS, layer), 0.0, recipe.bias_sigma))}


def make_tokens(shape: Shape, seed: int, T: int, stream: int = 0,
                attempts: np.ndarray | None = None, sigma: float = 1.0) -> np.ndarray:
    """x [T, H] bf16 bits, row t drawn from its own stream (seed, stream, t, attempt[t])."""
    out = np.empty((T, shape.hidden), dtype=np.uint16)
    att = None
    if attempts is not None:
        att = np.ascontiguousarray(attempts, dtype=np.int32)
        assert att.shape == (T,)
    _L().k3s_fill_token_rows_bf16(_ptr(out), T, shape.hidden, seed, TX, stream,
                                  None if att is None else _ptr(att), 0.0, sigma)
    return out


def make_residual(shape: Shape, seed: int, T: int, stream: int = 0,
                  attempts: np.ndarray | None = None) -> np.ndarray:
    """Residual-stream rows h [T, H] fp32 as the decoder hands them to the
    RMSNorm in front of the MoE: N(0, 1) per element times a per-token scale
    2^u, u ~ N(1, 1) clipped to [-1, 4] (the pages print per-layer maxima of
    |h| from about 3 to 76), with four fixed channels ten times larger (the
    outlier channels of a residual stream). Row t comes from its own stream
    (seed, stream, t, attempts[t])."""
    H = shape.hidden
    att = None
    if attempts is not None:
        att = np.ascontiguousarray(attempts, dtype=np.int32)
        assert att.shape == (T,)
    rows = np.empty((T, H), dtype=np.float64)
    _L().k3s_fill_token_rows_f64(_ptr(rows), T, H, seed, TRESID, stream,
                                 None if att is None else _ptr(att), 0.0, 1.0)
    u = np.empty((T, 1), dtype=np.float64)
    _L().k3s_fill_token_rows_f64(_ptr(u), T, 1, seed, TRESID_SCALE, stream,
                                 None if att is None else _ptr(att), 1.0, 1.0)
    rows *= np.exp2(np.clip(u, -1.0, 4.0))
    rows[:, [3, H // 3, H // 2 + 1, H - 5]] *= 10.0
    return rows.astype(np.float32)


def dense_shape(hidden: int, dense_inter: int) -> "Shape":
    """The configuration of a dense feed-forward layer: no routed part."""
    return Shape(hidden=hidden, latent=0, n_experts=0, topk=0, moe_inter=0, shared_inter=dense_inter)


def make_dense_layer(shape: "Shape", seed: int, sigma: float = 0.02) -> dict:
    """Weights of a dense feed-forward layer: sh_w1/sh_w3 [F, H], sh_w2 [H, F]
    bf16 N(0, sigma), F = shape.shared_inter."""
    H, F = shape.hidden, shape.shared_inter
    return {"sh_w1": normal_bf16((F, H), key(seed, TD1), 0.0, sigma),
            "sh_w3": normal_bf16((F, H), key(seed, TD3), 0.0, sigma),
            "sh_w2": normal_bf16((H, F), key(seed, TD2), 0.0, sigma)}


def post_norm_gain(shape: Shape, seed: int, layer: int = 0) -> np.ndarray:
    """bf16 bits [H] of the RMSNorm gain in front of the MoE: 1 + N(0, 0.1)."""
    return normal_bf16((shape.hidden,), key(seed, TPOSTGAIN, layer), 1.0, 0.1)


def covering_tokens(shape: Shape, layer: dict, seed: int, T: int, a: float = 15.0,
                    stream: int = 1, attempts: np.ndarray | None = None) -> np.ndarray:
    """Tokens whose top-k sets tile the expert pool.

    x_t = N(0,1) + a * sum_{e in S_t} Wr_e / |Wr_e|^2 with S_t = {(k*t + j) mod E : j < k},
    so that the router logit of every e in S_t is about a, far above the others,
    and T*k >= E picks cover all E experts. The construction only places input
    vectors; it computes nothing of the layer.
    """
    H, E, k = shape.hidden, shape.n_experts, shape.topk
    out64 = np.empty((T, H), dtype=np.float64)
    att = None
    if attempts is not None:
        att = np.ascontiguousarray(attempts, dtype=np.int32)
    _L().k3s_fill_token_rows_f64(_ptr(out64), T, H, seed, TCOVER, stream,
                                 None if att is None else _ptr(att), 0.0, 1.0)
    W = bf16_bits_to_f32(layer["router_w"]).astype(np.float64)
    dirs = W / np.sum(W * W, axis=1, keepdims=True)
    for t in range(T):
        for j in range(k):
            out64[t] += a * dirs[(k * t + j) % E]
    return round_bf16(out64)


# Bias strength that gives the K3 prefill workload a Zipf(1.1) expert popularity
# (pick counts sorted by rank fall with slope -1.1 in log-log over ranks
# 1..256); written by tests/golden/calibrate_zipf.py into zipf_alpha.json.
K3_ZIPF_ALPHA = 0.059509


def zipf_bias(shape: Shape, seed: int, layer: int, alpha: float, s: float = 1.1) -> np.ndarray:
    """Per-expert score-correction bias that makes expert popularity Zipf-like:
    bias_e = alpha * ln((pi(e)+1)^-s) with pi a seeded permutation of the experts
    (pi(e) is e's popularity rank, 0 = most popular)."""
    E = shape.n_experts
    w = words(E, key(seed, TPERM, layer))
    rank = np.empty(E, dtype=np.int64)
    rank[np.argsort(w, kind="stable")] = np.arange(E)
    return (alpha * (-s) * np.log(rank.astype(np.float64) + 1.0)).astype(np.float32)


def with_bias(layer: dict, bias: np.ndarray) -> dict:
    d = dict(layer)
    d["router_bias"] = np.ascontiguousarray(bias, dtype=np.float32)
    return d


__all__ = ["Shape", "K3", "TINY", "WeightRecipe", "K3_RECIPE", "TINY_RECIPE", "make_layer",
           "make_residual", "post_norm_gain", "dense_shape", "make_dense_layer", "K3_DENSE",
           "make_tokens", "covering_tokens", "zipf_bias", "with_bias", "bf16_bits_to_f32",
           "round_bf16", "build", "key", "replace", "MXFP4_GROUP"]
