"""Python binding of libk3moe (the Kimi K3 LatentMoE layer on GB300).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. The functions carry the C names of include/k3moe.h. Device pointers
may be given as integers or as torch tensors (their data_ptr is used); the
stream as an integer handle, a torch.cuda.Stream, or None (the legacy default
stream).

Loading fails loudly when libk3moe.so has not been built: there is no CPU or
PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libk3moe.so")

K3MOE_OK = 0
K3MOE_ERR_INVALID_ARG = -1
K3MOE_ERR_CONFIG = -2
K3MOE_ERR_SHAPE = -3
K3MOE_ERR_OOM = -4
K3MOE_ERR_BAD_SCALE = -5
K3MOE_ERR_NOT_LOADED = -6
K3MOE_ERR_CUDA = -7
K3MOE_ERR_TIMEOUT = -8
K3MOE_ERR_DEVICE = -9
K3MOE_ERR_GUARD = -10
K3MOE_HOST, K3MOE_DEVICE = 0, 1
K3MOE_T_Z, K3MOE_T_ACC, K3MOE_T_SHARED, K3MOE_T_LOGITS, K3MOE_T_X = 1, 2, 3, 4, 5

# Every symbol include/k3moe.h declares.
EXPORTS = ("k3moe_create", "k3moe_load_layer", "k3moe_forward", "k3moe_forward_chain",
           "k3moe_forward_host", "k3moe_get_routing", "k3moe_get_intermediate",
           "k3moe_sync_status", "k3moe_set_profiling", "k3moe_profile_read", "k3moe_destroy",
           "k3moe_strerror", "k3moe_abi_version", "k3moe_route_static", "k3moe_set_expert_path",
           "k3moe_set_expert_tier", "k3moe_get_tier_stats", "k3moe_load_post_norm",
           "k3moe_forward_residual", "k3moe_set_topp", "k3moe_tier_pin_layer",
           "k3moe_check_wait_timeout")
K3MOE_ROUTE_STATIC_MAX_LOGITS = 1 << 20
K3MOE_EXPERT_AUTO, K3MOE_EXPERT_GEMV, K3MOE_EXPERT_GEMM, K3MOE_EXPERT_MX = 0, 1, 2, 3


class K3MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


class k3moe_config(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("hidden", ctypes.c_int32),
                ("latent", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("moe_inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("max_layers", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("device", ctypes.c_int32),
                ("renorm", ctypes.c_int32), ("latent_norm", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("situ_b1", ctypes.c_float),
                ("situ_b2", ctypes.c_float), ("routed_scale", ctypes.c_float)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class k3moe_layer_weights(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("where", ctypes.c_int32),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("down_w", ctypes.c_void_p), ("up_w", ctypes.c_void_p),
                ("latent_gain", ctypes.c_void_p), ("shared_w1", ctypes.c_void_p),
                ("shared_w3", ctypes.c_void_p), ("shared_w2", ctypes.c_void_p),
                ("w1_packed", _PP), ("w1_scale", _PP), ("w3_packed", _PP), ("w3_scale", _PP),
                ("w2_packed", _PP), ("w2_scale", _PP)]


class k3moe_tier_stats(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_int32), ("slots", ctypes.c_int32),
                ("hits", ctypes.c_int64), ("misses", ctypes.c_int64),
                ("bytes_filled", ctypes.c_int64)]


class k3moe_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32),
                ("total_ms", ctypes.c_double)]


_lib = None


def lib():
    """The loaded libk3moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mxfp4_routed_expert_gb300.build` (no fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.k3moe_create.argtypes = [ctypes.POINTER(k3moe_config), ctypes.POINTER(vp)]
        L.k3moe_load_layer.argtypes = [vp, i, ctypes.POINTER(k3moe_layer_weights)]
        L.k3moe_forward.argtypes = [vp, i, vp, vp, i, vp]
        L.k3moe_forward_chain.argtypes = [vp, i, i, vp, vp, i, vp]
        L.k3moe_forward_host.argtypes = [vp, i, vp, vp, i, vp]
        L.k3moe_get_routing.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.k3moe_get_intermediate.argtypes = [vp, i, vp, sz, vp]
        L.k3moe_sync_status.argtypes = [vp]
        L.k3moe_set_profiling.argtypes = [vp, i]
        L.k3moe_set_expert_path.argtypes = [vp, i]
        L.k3moe_profile_read.argtypes = [vp, ctypes.POINTER(k3moe_kernel_stat), i,
                                         ctypes.POINTER(ctypes.c_int)]
        L.k3moe_destroy.argtypes = [vp]
        L.k3moe_destroy.restype = None
        L.k3moe_strerror.argtypes = [i]
        L.k3moe_strerror.restype = ctypes.c_char_p
        L.k3moe_abi_version.restype = i
        L.k3moe_route_static.argtypes = [vp, vp, vp, i, i, i, i, i, ctypes.c_float, vp, vp, vp]
        L.k3moe_set_expert_tier.argtypes = [vp, i]
        L.k3moe_load_post_norm.argtypes = [vp, i, vp, i]
        L.k3moe_set_topp.argtypes = [vp, ctypes.c_float]
        L.k3moe_tier_pin_layer.argtypes = [vp, i]
        L.k3moe_forward_residual.argtypes = [vp, i, vp, vp, i, vp]
        L.k3moe_get_tier_stats.argtypes = [vp, ctypes.POINTER(k3moe_tier_stats)]
        L.k3moe_check_wait_timeout.argtypes = [vp, vp]
        for n in EXPORTS:
            if n not in ("k3moe_destroy", "k3moe_strerror"):
                getattr(L, n).restype = i
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().k3moe_strerror(int(code)).decode()


def _addr(v) -> int:
    """Address of a dense, row-major buffer (a torch tensor or numpy array):
    the library reads every buffer in that layout, so a strided view is refused
    rather than read as if it were dense."""
    if hasattr(v, "data_ptr"):
        if not v.is_contiguous():
            raise ValueError("tensor is not contiguous (row-major); pass .contiguous()")
        return v.data_ptr()
    if isinstance(v, np.ndarray):
        if not v.flags["C_CONTIGUOUS"]:
            raise ValueError("array is not C-contiguous; pass np.ascontiguousarray(...)")
        return v.ctypes.data
    raise TypeError(f"cannot pass {type(v)} as a pointer")


def _ptr(v):
    if v is None:
        return None
    if isinstance(v, int):
        return ctypes.c_void_p(v)
    return ctypes.c_void_p(_addr(v))


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return ctypes.c_void_p(s)
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str) -> int:
    if rc != K3MOE_OK:
        raise K3MoEError(rc, what)
    return rc


def make_config(shape, max_layers: int = 1, max_tokens: int = 1, device: int = 0,
                latent_norm: int = 1) -> k3moe_config:
    """k3moe_config from a layer shape (any object with the K3Cfg field names)."""
    c = k3moe_config()
    c.struct_size = ctypes.sizeof(k3moe_config)
    c.hidden, c.latent, c.n_experts = shape.hidden, shape.latent, shape.n_experts
    c.topk, c.moe_inter, c.shared_inter = shape.topk, shape.moe_inter, shape.shared_inter
    c.max_layers, c.max_tokens, c.device = max_layers, max_tokens, device
    c.renorm, c.latent_norm = int(shape.renorm), int(latent_norm)
    c.rms_eps, c.situ_b1, c.situ_b2 = shape.rms_eps, shape.situ_b1, shape.situ_b2
    c.routed_scale = shape.routed_scale
    return c


def k3moe_create(cfg: k3moe_config) -> int:
    h = ctypes.c_void_p()
    _check(lib().k3moe_create(ctypes.byref(cfg), ctypes.byref(h)), "k3moe_create")
    return h.value


def k3moe_destroy(h: int) -> None:
    lib().k3moe_destroy(ctypes.c_void_p(h))


def layer_weights(tensors: dict, n_experts: int, where: int = K3MOE_HOST):
    """k3moe_layer_weights pointing into `tensors` (numpy arrays for HOST, torch
    CUDA tensors for DEVICE) in the checkpoint layout; expert arrays are
    [E, rows, cols] and are split into per-expert pointers. Returns the struct
    and the objects that must stay alive while it is used."""
    keep = []

    def addr(v):
        return None if v is None else _addr(v)

    def per_expert(v):
        base = addr(v)
        stride = (v.nbytes if isinstance(v, np.ndarray) else v.numel() * v.element_size()) // n_experts
        arr = (ctypes.c_void_p * n_experts)(*[base + e * stride for e in range(n_experts)])
        keep.append(arr)
        return ctypes.cast(arr, _PP)

    w = k3moe_layer_weights()
    w.struct_size = ctypes.sizeof(k3moe_layer_weights)
    w.where = where
    if n_experts == 0:   # dense feed-forward layer: the three matrices only
        w.shared_w1 = addr(tensors["sh_w1"])
        w.shared_w3 = addr(tensors["sh_w3"])
        w.shared_w2 = addr(tensors["sh_w2"])
        keep.append(tensors)
        return w, keep
    w.router_w = addr(tensors["router_w"])
    w.router_bias = addr(tensors.get("router_bias"))
    w.down_w = addr(tensors["down_w"])
    w.up_w = addr(tensors["up_w"])
    w.latent_gain = addr(tensors.get("latent_gain"))
    w.shared_w1 = addr(tensors["sh_w1"])
    w.shared_w3 = addr(tensors["sh_w3"])
    w.shared_w2 = addr(tensors["sh_w2"])
    w.w1_packed, w.w1_scale = per_expert(tensors["w1p"]), per_expert(tensors["w1s"])
    w.w3_packed, w.w3_scale = per_expert(tensors["w3p"]), per_expert(tensors["w3s"])
    w.w2_packed, w.w2_scale = per_expert(tensors["w2p"]), per_expert(tensors["w2s"])
    keep.append(tensors)
    return w, keep


def k3moe_load_layer(h: int, layer: int, weights: k3moe_layer_weights) -> int:
    return _check(lib().k3moe_load_layer(ctypes.c_void_p(h), layer, ctypes.byref(weights)),
                  "k3moe_load_layer")


def k3moe_forward(h: int, layer: int, x, y, T: int, stream=None) -> int:
    return _check(lib().k3moe_forward(ctypes.c_void_p(h), layer, _ptr(x), _ptr(y), T,
                                      _stream(stream)), "k3moe_forward")


def k3moe_load_post_norm(h: int, layer: int, gain, where: int = K3MOE_HOST) -> int:
    """The RMSNorm gain (bf16 [hidden]: a numpy uint16 array for HOST, a CUDA
    tensor for DEVICE) in front of the MoE, for k3moe_forward_residual."""
    return _check(lib().k3moe_load_post_norm(ctypes.c_void_p(h), layer, _ptr(gain), where),
                  "k3moe_load_post_norm")


def k3moe_forward_residual(h: int, layer: int, h_in, y, T: int, stream=None) -> int:
    """The layer on x = bf16(RMSNorm(h_in) * post-norm gain); h_in fp32 [T, hidden]."""
    return _check(lib().k3moe_forward_residual(ctypes.c_void_p(h), layer, _ptr(h_in), _ptr(y), T,
                                               _stream(stream)),
                  "k3moe_forward_residual")


def k3moe_forward_chain(h: int, first_layer: int, n_layers: int, x, y, T: int, stream=None) -> int:
    return _check(lib().k3moe_forward_chain(ctypes.c_void_p(h), first_layer, n_layers, _ptr(x),
                                            _ptr(y), T, _stream(stream)), "k3moe_forward_chain")


def k3moe_forward_host(h: int, layer: int, x_host, y_host, T: int, stream=None) -> int:
    """The layer on host buffers (x in, y out); returns once y is written. The
    per-token decode loop calls it once per token, so its marshalling is kept
    to the checks the library needs (dense buffers)."""
    rc = lib().k3moe_forward_host(h, layer, _addr(x_host), _addr(y_host), T,
                                  stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)
    return rc if rc == K3MOE_OK else _check(rc, "k3moe_forward_host")


def k3moe_get_routing(h: int, ids=None, w=None, counts=None, offsets=None, perm=None,
                      stream=None) -> int:
    return _check(lib().k3moe_get_routing(ctypes.c_void_p(h), _ptr(ids), _ptr(w), _ptr(counts),
                                          _ptr(offsets), _ptr(perm), _stream(stream)),
                  "k3moe_get_routing")


def k3moe_get_intermediate(h: int, which: int, dst, nbytes: int, stream=None) -> int:
    return _check(lib().k3moe_get_intermediate(ctypes.c_void_p(h), which, _ptr(dst), nbytes,
                                               _stream(stream)), "k3moe_get_intermediate")


def k3moe_sync_status(h: int) -> int:
    return lib().k3moe_sync_status(ctypes.c_void_p(h))


def k3moe_check_wait_timeout(h: int, stream=None) -> int:
    """Launch a kernel whose one bounded wait runs out: the next
    k3moe_sync_status returns K3MOE_ERR_TIMEOUT (about two seconds later)."""
    return _check(lib().k3moe_check_wait_timeout(ctypes.c_void_p(h), _stream(stream)),
                  "k3moe_check_wait_timeout")


def k3moe_set_profiling(h: int, enable: bool) -> int:
    return _check(lib().k3moe_set_profiling(ctypes.c_void_p(h), int(bool(enable))),
                  "k3moe_set_profiling")


def k3moe_set_expert_path(h: int, mode: int) -> int:
    """K3MOE_EXPERT_AUTO / _GEMV / _GEMM / _MX: which routed-expert kernels forwards use."""
    return _check(lib().k3moe_set_expert_path(ctypes.c_void_p(h), int(mode)),
                  "k3moe_set_expert_path")


def k3moe_set_topp(h: int, p: float) -> int:
    """Keep each token's picks up to cumulative weight p (0: all topk)."""
    return _check(lib().k3moe_set_topp(ctypes.c_void_p(h), float(p)), "k3moe_set_topp")


def k3moe_set_expert_tier(h: int, slots: int) -> int:
    """Host memory holds the routed experts of layers loaded afterwards; `slots`
    device slots cache them (0: off). Call before the first k3moe_load_layer."""
    return _check(lib().k3moe_set_expert_tier(ctypes.c_void_p(h), int(slots)),
                  "k3moe_set_expert_tier")


def k3moe_tier_pin_layer(h: int, layer: int) -> int:
    """Copy a loaded layer's experts into tier slots that eviction skips."""
    return _check(lib().k3moe_tier_pin_layer(ctypes.c_void_p(h), layer), "k3moe_tier_pin_layer")


def k3moe_get_tier_stats(h: int) -> dict:
    """Cumulative expert-tier counters: slots, hits, misses, bytes_filled."""
    st = k3moe_tier_stats()
    st.struct_size = ctypes.sizeof(k3moe_tier_stats)
    _check(lib().k3moe_get_tier_stats(ctypes.c_void_p(h), ctypes.byref(st)), "k3moe_get_tier_stats")
    return dict(slots=st.slots, hits=st.hits, misses=st.misses, bytes_filled=st.bytes_filled)


def k3moe_profile_read(h: int, max_entries: int = 32):
    """[(name, launches, total_ms)] since the last read."""
    arr = (k3moe_kernel_stat * max_entries)()
    n = ctypes.c_int(0)
    _check(lib().k3moe_profile_read(ctypes.c_void_p(h), arr, max_entries, ctypes.byref(n)),
           "k3moe_profile_read")
    return [(arr[i].name.decode(), arr[i].launches, arr[i].total_ms)
            for i in range(min(n.value, max_entries))]


def k3moe_abi_version() -> int:
    return lib().k3moe_abi_version()


def k3moe_route_static(x, router_w, router_bias, T: int, hidden: int, n_experts: int, topk: int,
                       renorm: int, routed_scale: float, ids, w, stream=None) -> int:
    """Router step without a handle or any allocation (see include/k3moe.h)."""
    return _check(lib().k3moe_route_static(_ptr(x), _ptr(router_w), _ptr(router_bias), T, hidden,
                                           n_experts, topk, renorm, float(routed_scale),
                                           _ptr(ids), _ptr(w), _stream(stream)),
                  "k3moe_route_static")
