"""CPU oracle for the K3 LatentMoE layer (plain C99, fp64) and its loader.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may call it. The CUDA library never does and
shares nothing with it. The arithmetic lives in ``k3moe_oracle.c``; this
module compiles it with gcc (no fast-math, no FMA contraction) and marshals
numpy arrays through ctypes. `build(out=..., flags=SANITIZE_FLAGS)` makes an
AddressSanitizer/UBSan build of the same source, and K3MOE_ORACLE_LIB makes
the loader use such a build (tests/test_oracle_sanitized.py).

Parity status of each function is recorded where it is pinned (tests/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


_FLAGS = ["-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]
# an instrumented build of the same source: address and undefined-behaviour
# sanitizers, stopping at the first finding
SANITIZE_FLAGS = ["-O1", "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
                  "-fno-sanitize-recover=all"]


def build(force: bool = False, out: str | None = None, flags=("-O2",)) -> str:
    """Compiles the oracle to `out` (default: liboracle.so beside the source).
    K3MOE_ORACLE_LIB names an already built library to load instead."""
    if out is None and os.environ.get("K3MOE_ORACLE_LIB"):
        return os.environ["K3MOE_ORACLE_LIB"]
    out = out or _LIB_PATH
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    try:
        subprocess.check_call(["gcc", *flags, *_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


class _Cfg(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("latent", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("topk", ctypes.c_int), ("moe_inter", ctypes.c_int), ("shared_inter", ctypes.c_int),
                ("renorm", ctypes.c_int), ("rms_eps", ctypes.c_double),
                ("situ_b1", ctypes.c_double), ("situ_b2", ctypes.c_double),
                ("routed_scale", ctypes.c_double), ("topp", ctypes.c_double)]


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("router_w", "router_bias", "down_w", "up_w", "latent_gain", "sh_w1", "sh_w3",
                 "sh_w2", "w1p", "w1s", "w3p", "w3s", "w2p", "w2s")]


class _Trace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("ids", "w", "margin", "z", "acc", "nrm", "shared", "h")]


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        d, p, i = ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.orc_bf16.restype = d
        lib.orc_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_e2m1.restype = d
        lib.orc_e2m1.argtypes = [ctypes.c_uint]
        lib.orc_e8m0.restype = d
        lib.orc_e8m0.argtypes = [ctypes.c_uint]
        lib.orc_mxfp4_weight.restype = d
        lib.orc_mxfp4_weight.argtypes = [p, p, i]
        lib.orc_mxfp4_matvec.argtypes = [p, p, p, p, i, i]
        lib.orc_bf16_matvec.argtypes = [p, p, p, i, i]
        lib.orc_sigmoid.restype = d
        lib.orc_sigmoid.argtypes = [d]
        lib.orc_situ.restype = d
        lib.orc_situ.argtypes = [d, d, d, d]
        lib.orc_rmsnorm.argtypes = [p, p, p, i, d]
        lib.orc_router_token.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, d]
        lib.orc_permutation.argtypes = [p, i, i, i, p, p, p]
        lib.orc_layer_forward.argtypes = [p, p, p, i, p, i, p, p]
        lib.orc_route.argtypes = [p, p, p, i, p, p, p, p, p]
        lib.orc_chain_glue.argtypes = [p, p, i, i, d]
        lib.orc_dense_ffn.argtypes = [p, p, i, p, p, p, i, i, d, d]
        lib.orc_topp_cut.restype = i
        lib.orc_topp_cut.argtypes = [p, p, i, d, p]
        lib.orc_group_size.restype = i
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---- formats -----------------------------------------------------------------

def bf16(bits: int) -> float:
    return _L().orc_bf16(int(bits) & 0xFFFF)


def e2m1(nibble: int) -> float:
    return _L().orc_e2m1(int(nibble))


def e8m0(byte: int) -> float:
    return _L().orc_e8m0(int(byte))


def group_size() -> int:
    return _L().orc_group_size()


def mxfp4_weight(packed_row, scale_row, c: int) -> float:
    pr, sr = _c(packed_row, np.uint8), _c(scale_row, np.uint8)
    return _L().orc_mxfp4_weight(_p(pr), _p(sr), int(c))


def mxfp4_matvec(x, packed, scales, n_in: int) -> np.ndarray:
    packed, scales = _c(packed, np.uint8), _c(scales, np.uint8)
    rows = packed.shape[0]
    assert packed.shape[1] == (n_in + 1) // 2 and scales.shape == (rows, (n_in + 31) // 32)
    x = _c(x, np.float64)
    assert x.shape == (n_in,)
    y = np.empty(rows, np.float64)
    _L().orc_mxfp4_matvec(_p(y), _p(x), _p(packed), _p(scales), n_in, rows)
    return y


def bf16_matvec(x, W_bits) -> np.ndarray:
    W = _c(W_bits, np.uint16)
    out, n_in = W.shape
    x = _c(x, np.float64)
    y = np.empty(out, np.float64)
    _L().orc_bf16_matvec(_p(y), _p(x), _p(W), n_in, out)
    return y


# ---- elementwise ---------------------------------------------------------------

def sigmoid(v: float) -> float:
    return _L().orc_sigmoid(float(v))


def situ(g: float, u: float, b1: float = 4.0, b2: float = 25.0) -> float:
    return _L().orc_situ(float(g), float(u), float(b1), float(b2))


def rmsnorm(x, gain=None, eps: float = 1e-5) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty_like(x)
    g = None if gain is None else _c(gain, np.float64)
    _L().orc_rmsnorm(_p(out), _p(x), _p(g), x.size, float(eps))
    return out


def round_bf16(v) -> np.ndarray:
    """fp64 -> bf16 bit patterns, round to nearest with ties to even, overflow
    to infinity: the 8 significant bits of bf16 (7 stored), with the fp32
    exponent range and subnormals down to 2^-133. The value is rounded once,
    at its own unit in the last place."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)                                 # a = m * 2^e, m in [0.5, 1)
    ulp = np.maximum(e - 8, -133)                      # 2^(e-8): the last of 8 bits
    q = np.ldexp(np.round(np.ldexp(a, -ulp)), ulp)     # np.round: ties to even; exact
    with np.errstate(over="ignore"):
        mag = (q.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # q fits exactly
    return np.where(np.signbit(v), mag | np.uint16(0x8000), mag).astype(np.uint16)


def residual_input(h, gain_bits, eps: float = 1e-5) -> np.ndarray:
    """x = RMSNorm(h) * gain per token in fp64, the input the decoder hands to
    the MoE (kimi-k3-in-c README, Part II: post_norm then k3_moe; section 5
    k3_rmsnorm). h [T, H] (any float type), gain bf16 bits [H]."""
    h = np.asarray(h, dtype=np.float64)
    g = (np.asarray(gain_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.stack([rmsnorm(row, g, eps) for row in h])


# ---- router / permutation ------------------------------------------------------------

def router_token(x, Wr_bits, bias, k: int, renorm: int = 1, routed_scale: float = 1.0):
    """Returns (ids[k], w[k], sc[E], ch[E], margin) for one token (x in fp64)."""
    Wr = _c(Wr_bits, np.uint16)
    E, H = Wr.shape
    x = _c(x, np.float64)
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty(k, np.int32)
    w = np.empty(k, np.float64)
    sc = np.empty(E, np.float64)
    ch = np.empty(E, np.float64)
    m = np.empty(1, np.float64)
    _L().orc_router_token(_p(ids), _p(w), _p(sc), _p(ch), _p(m), _p(x), _p(Wr), _p(b),
                          H, E, k, int(renorm), float(routed_scale))
    return ids, w, sc, ch, float(m[0])


def topp_cut(ids, w, p: float):
    """The cumulative-weight cut of one token's picks (ids, w in selection
    order): returns (ids, w, kept, margin); dropped slots hold -1 and 0."""
    ids = np.array(ids, dtype=np.int32)
    w = np.array(w, dtype=np.float64)
    m = np.empty(1, np.float64)
    n = _L().orc_topp_cut(_p(ids), _p(w), ids.size, float(p), _p(m))
    return ids, w, int(n), float(m[0])


def permutation(ids, E: int):
    """(counts[E], offsets[E+1], perm[T*k]) of a [T, k] id matrix."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    _L().orc_permutation(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm


# ---- layer -----------------------------------------------------------------

def _cfg(shape) -> _Cfg:
    return _Cfg(shape.hidden, shape.latent, shape.n_experts, shape.topk, shape.moe_inter,
                shape.shared_inter, int(shape.renorm), float(shape.rms_eps),
                float(shape.situ_b1), float(shape.situ_b2), float(shape.routed_scale),
                float(getattr(shape, "topp", 0.0)))


_LAYER_KEYS = ("router_w", "router_bias", "down_w", "up_w", "latent_gain", "sh_w1", "sh_w3",
               "sh_w2", "w1p", "w1s", "w3p", "w3s", "w2p", "w2s")
_LAYER_DT = {"router_bias": np.float32, "w1p": np.uint8, "w1s": np.uint8, "w3p": np.uint8,
             "w3s": np.uint8, "w2p": np.uint8, "w2s": np.uint8}


def _layer(shape, layer: dict):
    H, L, E, I, S = shape.hidden, shape.latent, shape.n_experts, shape.moe_inter, shape.shared_inter
    want = {"router_w": (E, H), "router_bias": (E,), "down_w": (L, H), "up_w": (H, L),
            "latent_gain": (L,), "sh_w1": (S, H), "sh_w3": (S, H), "sh_w2": (H, S),
            "w1p": (E, I, L // 2), "w1s": (E, I, L // 32), "w3p": (E, I, L // 2),
            "w3s": (E, I, L // 32), "w2p": (E, L, I // 2), "w2s": (E, L, I // 32)}
    keep = {}
    ptrs = []
    for k in _LAYER_KEYS:
        a = layer.get(k)
        if a is None:
            if k in ("router_bias", "latent_gain"):
                ptrs.append(None)
                continue
            raise KeyError(k)
        a = _c(a, _LAYER_DT.get(k, np.uint16))
        assert a.shape == want[k], (k, a.shape, want[k])
        keep[k] = a
        ptrs.append(a.ctypes.data)
    return _Layer(*ptrs), keep


def route(shape, layer: dict, x_bits, want_scores: bool = False):
    """Router for all tokens: (ids[T,k], w[T,k], margin[T]) (+ sc, ch [T,E])."""
    x = _c(x_bits, np.uint16)
    T = x.shape[0]
    lw, keep = _layer(shape, layer)
    cfg = _cfg(shape)
    ids = np.empty((T, shape.topk), np.int32)
    w = np.empty((T, shape.topk), np.float64)
    margin = np.empty(T, np.float64)
    sc = ch = None
    if want_scores:
        sc = np.empty((T, shape.n_experts), np.float64)
        ch = np.empty((T, shape.n_experts), np.float64)
    _L().orc_route(ctypes.byref(cfg), ctypes.byref(lw), _p(x), T, _p(ids), _p(w), _p(margin),
                   _p(sc), _p(ch))
    del keep
    if want_scores:
        return ids, w, margin, sc, ch
    return ids, w, margin


def layer_forward(shape, layer: dict, x_bits, rows=None, trace: bool = False):
    """y [nrows, H] fp64 for tokens `rows` of x [T, H] (all tokens if rows is None).
    With trace=True also returns a dict of intermediates (ids, w, margin, z, acc,
    nrm, shared, h)."""
    x = _c(x_bits, np.uint16)
    T = x.shape[0]
    assert x.shape[1] == shape.hidden
    r = None if rows is None else _c(rows, np.int32)
    n = T if r is None else r.size
    if r is not None:
        assert r.min() >= 0 and r.max() < T
    lw, keep = _layer(shape, layer)
    cfg = _cfg(shape)
    y = np.empty((n, shape.hidden), np.float64)
    tr = None
    arrs = None
    if trace:
        K, L, I, S = shape.topk, shape.latent, shape.moe_inter, shape.shared_inter
        arrs = dict(ids=np.empty((n, K), np.int32), w=np.empty((n, K)), margin=np.empty(n),
                    z=np.empty((n, L)), acc=np.empty((n, L)), nrm=np.empty((n, L)),
                    shared=np.empty((n, S)), h=np.empty((n, K, I)))
        tr = _Trace(*[arrs[k].ctypes.data for k in ("ids", "w", "margin", "z", "acc", "nrm",
                                                    "shared", "h")])
    _L().orc_layer_forward(ctypes.byref(cfg), ctypes.byref(lw), _p(x), T, _p(r), n, _p(y),
                           ctypes.byref(tr) if tr is not None else None)
    del keep
    return (y, arrs) if trace else y


def dense_ffn(x_bits, w1_bits, w3_bits, w2_bits, b1: float = 4.0, b2: float = 25.0) -> np.ndarray:
    """The dense feed-forward layer: y = W2 . SiTU(W1 x, W3 x) per token, fp64.
    x [T, H], W1/W3 [F, H], W2 [H, F], all bf16 bits."""
    x = _c(x_bits, np.uint16)
    W1, W3, W2 = _c(w1_bits, np.uint16), _c(w3_bits, np.uint16), _c(w2_bits, np.uint16)
    T, H = x.shape
    F = W1.shape[0]
    assert W1.shape == (F, H) and W3.shape == (F, H) and W2.shape == (H, F)
    y = np.empty((T, H), np.float64)
    _L().orc_dense_ffn(_p(y), _p(x), T, _p(W1), _p(W3), _p(W2), H, F, float(b1), float(b2))
    return y


def chain_glue(y, eps: float = 1e-5) -> np.ndarray:
    """x_next = RMSNorm(y) per token with unit gain (fp64)."""
    y = _c(y, np.float64)
    T, H = y.shape
    out = np.empty_like(y)
    _L().orc_chain_glue(_p(out), _p(y), T, H, float(eps))
    return out
