"""Forward from the residual stream through the C ABI (GPU): the RMSNorm in
front of the MoE (kimi-k3-in-c README, Part II: the decoder layer's
post_norm, then k3_moe; section 5, k3_rmsnorm) made inside the layer's first
kernels (T <= 2) or by a first kernel (otherwise).

Two checks per case, as for the stacked layers' glue:
  - the input the GPU made, x = bf16(RMSNorm(h) * gain), against the oracle's
    fp64 norm: within one bf16 step everywhere and equal to its correctly
    rounded value almost everywhere (the GPU forms inv in fp64 like the pages,
    but multiplies in fp32);
  - the layer given the GPU's own x against the oracle (ids and permutation
    exact, y within the layer tolerance).
"""
import numpy as np
import pytest

import k3synth
import oracle
from _harness import Layer, assert_close, bf16_to_f64, check_routing, guarded_tokens

pytestmark = pytest.mark.gpu

MID = k3synth.Shape(hidden=1024, latent=512, n_experts=64, topk=8, moe_inter=512,
                    shared_inter=1024)
WIDE = k3synth.Shape(hidden=1024, latent=512, n_experts=128, topk=8, moe_inter=512,
                     shared_inter=1024)
SHAPES = {"tiny": k3synth.TINY, "mid": MID, "wide": WIDE}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


def residual_case(shape, seed, T):
    d = k3synth.make_layer(shape, seed, 0, k3synth.TINY_RECIPE)
    g = k3synth.post_norm_gain(shape, seed)
    eps = shape.rms_eps
    make = lambda att: oracle.round_bf16(   # noqa: E731
        oracle.residual_input(k3synth.make_residual(shape, seed, T, 0, att), g, eps))
    _, att = guarded_tokens(shape, d, seed, T, make=make)
    return d, g, k3synth.make_residual(shape, seed, T, 0, att)


@pytest.mark.parametrize("name,T", [("tiny", 1), ("mid", 1), ("mid", 2), ("mid", 5),
                                    ("wide", 2), ("wide", 40)])
def test_forward_residual(name, T):
    import mxfp4_routed_expert_gb300 as km
    shape = SHAPES[name]
    d, g, hres = residual_case(shape, 60 + T, T)
    lay = Layer(shape, [d], max_tokens=T)
    try:
        km.k3moe_load_post_norm(lay.h, 0, g)
        y = lay.forward_residual(hres)
        x_gpu = lay.layer_input(T)
        r = lay.routing(T)
    finally:
        lay.close()
    # the input: one bf16 step at most from the fp64 norm, mostly its rounding
    v = oracle.residual_input(hres, g, shape.rms_eps)
    xg = bf16_to_f64(x_gpu)
    step = np.ldexp(1.0, np.frexp(np.abs(v))[1] - 8)
    assert np.all(np.abs(xg - v) <= step), "made input off by more than one bf16 step"
    assert np.mean(x_gpu == oracle.round_bf16(v)) >= 0.999
    # the layer on the GPU's own input
    ref, tr = oracle.layer_forward(shape, d, x_gpu, trace=True)
    check_routing(r, shape, x_gpu, tr["ids"], tr["w"])
    assert_close(bf16_to_f64(y), ref)


def test_forward_residual_errors():
    import torch
    import mxfp4_routed_expert_gb300 as km
    d, g, hres = residual_case(MID, 70, 2)
    lay = Layer(MID, [d], max_tokens=4)
    try:
        hd = torch.from_numpy(hres).cuda()
        y = torch.empty((2, MID.hidden), dtype=torch.int16, device="cuda")
        with pytest.raises(km.K3MoEError) as ei:           # no post-norm gain yet
            km.k3moe_forward_residual(lay.h, 0, hd, y, 2)
        assert ei.value.code == km.K3MOE_ERR_NOT_LOADED
        km.k3moe_load_post_norm(lay.h, 0, g)
        flat = torch.zeros(2 * MID.hidden + 1, dtype=torch.float32, device="cuda")
        with pytest.raises(km.K3MoEError) as ei:           # h_in not 16-byte aligned
            km.k3moe_forward_residual(lay.h, 0, flat[1:].data_ptr(), y, 2)
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        x = torch.from_numpy(k3synth.make_tokens(MID, 70, 2).view(np.int16).copy()).cuda()
        km.k3moe_forward(lay.h, 0, x, y, 2)
        torch.cuda.synchronize()
        buf = torch.empty((2, MID.hidden), dtype=torch.int16, device="cuda")
        with pytest.raises(km.K3MoEError) as ei:           # the last forward took x as given
            km.k3moe_get_intermediate(lay.h, km.K3MOE_T_X, buf, buf.numel() * 2)
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        with pytest.raises(km.K3MoEError) as ei:
            km.k3moe_load_post_norm(lay.h, 1, g)            # no such layer
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
    finally:
        lay.close()
