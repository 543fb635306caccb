"""The C ABI library loads and exports every symbol include/k3moe.h declares,
and its host-side argument/config checks answer without touching a GPU
(CPU only; no compute call is made)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def km():
    from mxfp4_routed_expert_gb300 import build
    build.build()
    import mxfp4_routed_expert_gb300 as km
    return km


def declared():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    return sorted(set(re.findall(r"K3MOE_API\s+[\w\s\*]*?\b(k3moe_\w+)\s*\(", src)))


def test_header_declares_the_layer_calls():
    names = declared()
    for n in ("k3moe_create", "k3moe_load_layer", "k3moe_forward", "k3moe_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(km):
    names = declared()
    assert set(names) == set(km.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", km.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (k3moe_\w+)", out))
    assert set(names) <= exported
    lib = km.lib()
    for n in names:
        assert hasattr(lib, n)


def test_library_leaves_no_own_symbol_unresolved(km):
    """Every function of the library's own namespace is defined inside it: an
    internal helper left out of a translation unit would otherwise surface
    only when its first call tries to bind (no GPU needed to see it)."""
    out = subprocess.run(["nm", "-D", "--undefined-only", "-C", km.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    own = [ln for ln in out.splitlines() if "k3::" in ln or "k3moe" in ln]
    assert not own, own


def test_abi_version_and_strerror(km):
    assert km.k3moe_abi_version() == 1
    for code in range(0, -11, -1):
        assert km.strerror(code) != "unknown error"
    assert km.strerror(-99) == "unknown error"


def _cfg(km, **over):
    import k3synth
    c = km.make_config(k3synth.TINY, max_layers=1, max_tokens=8)
    for k, v in over.items():
        setattr(c, k, v)
    return c


def _create(km, cfg):
    h = ctypes.c_void_p()
    rc = km.lib().k3moe_create(ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(h))
    return rc, h.value


@pytest.mark.parametrize("field,value,code", [
    ("struct_size", 4, -2), ("hidden", 0, -2), ("latent", -64, -2), ("n_experts", 0, -2),
    ("topk", 0, -2), ("max_tokens", 0, -2), ("rms_eps", 0.0, -2), ("situ_b1", float("nan"), -2),
    ("routed_scale", -1.0, -2), ("renorm", 2, -2), ("latent_norm", -1, -2),
    ("hidden", 100, -3), ("topk", 33, -3), ("n_experts", 2048, -3), ("latent", 8192, -3), ("moe_inter", 8192, -3),
    ("situ_b1", 100.0, -3), ("max_layers", 0, -2), ("max_layers", 1025, -3)])
def test_create_refuses_bad_config(km, field, value, code):
    rc, h = _create(km, _cfg(km, **{field: value}))
    assert rc == code and not h


def test_null_arguments(km):
    lib = km.lib()
    rc, h = _create(km, None)
    assert rc == km.K3MOE_ERR_INVALID_ARG and not h
    assert lib.k3moe_create(ctypes.byref(_cfg(km)), None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_forward(None, 0, None, None, 1, None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_load_layer(None, 0, None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_forward_chain(None, 0, 1, None, None, 1, None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_forward_host(None, 0, None, None, 1, None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_get_routing(None, None, None, None, None, None, None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_get_intermediate(None, 1, None, 0, None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_sync_status(None) == km.K3MOE_ERR_INVALID_ARG
    assert lib.k3moe_set_profiling(None, 1) == km.K3MOE_ERR_INVALID_ARG
    lib.k3moe_destroy(None)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import mxfp4_routed_expert_gb300 as km
    monkeypatch.setattr(km, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(km, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        km.lib()


def test_binding_refuses_strided_buffers():
    """The library reads every buffer row-major and dense: the binding passes
    the address of a contiguous tensor or array (or a plain integer address)
    and refuses a strided view instead of handing over its first element."""
    import numpy as np
    import torch
    import mxfp4_routed_expert_gb300 as km
    t = torch.zeros((4, 8), dtype=torch.int16)
    a = np.zeros((4, 8), dtype=np.uint16)
    assert km._ptr(t).value == t.data_ptr()
    assert km._ptr(t[1:3]).value == t[1:3].data_ptr()          # a block of rows is dense
    assert km._ptr(a).value == a.ctypes.data
    assert km._ptr(1234).value == 1234 and km._ptr(None) is None
    for bad in (t[:, ::2], t.t(), a[:, 1:], a.T):
        with pytest.raises(ValueError):
            km._ptr(bad)
    with pytest.raises(TypeError):
        km._ptr([1, 2, 3])
    with pytest.raises(ValueError):                             # weights too
        km.layer_weights({"sh_w1": t.t(), "sh_w3": t, "sh_w2": t}, 0)
