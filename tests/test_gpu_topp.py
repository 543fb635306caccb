"""The cumulative-weight cut of the picks (the pages' K3_TOPP run-time option:
keep each token's picks up to cumulative weight p, renormalised) through the
C ABI against the oracle with the same cut: kept ids and permutation exact,
y within the layer tolerance. Test tokens pass the routing margin guard, which
with a cut also covers the distance of every cumulative weight from p."""
import dataclasses

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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


@pytest.mark.parametrize("shape,T,p,path", [(MID, 1, 0.6, None), (MID, 5, 0.4, None),
                                            (WIDE, 40, 0.6, "gemm"), (WIDE, 40, 0.6, "gemv"),
                                            (MID, 3, 1.0, None)])
def test_topp_matches_oracle(shape, T, p, path):
    import mxfp4_routed_expert_gb300 as km
    sh = dataclasses.replace(shape, topp=p)
    d = k3synth.make_layer(sh, 70, 0, k3synth.TINY_RECIPE)
    x, _ = guarded_tokens(sh, d, 70 + T, T)
    lay = Layer(sh, [d], max_tokens=T)
    try:
        km.k3moe_set_topp(lay.h, p)
        if path is not None:
            km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_GEMM if path == "gemm" else km.K3MOE_EXPERT_GEMV)
        y = lay.forward(x)
        r = lay.routing(T)
    finally:
        lay.close()
    ref, tr = oracle.layer_forward(sh, d, x, trace=True)
    check_routing(r, sh, x, tr["ids"], tr["w"])
    if p < 1.0:
        assert (r["ids"] < 0).any(), "the cut dropped nothing"
    assert_close(bf16_to_f64(y), ref)


def test_topp_argument_errors():
    import mxfp4_routed_expert_gb300 as km
    lay = Layer(MID, [None], max_tokens=2)
    try:
        for bad in (-0.1, 1.5, float("nan")):
            with pytest.raises(km.K3MoEError) as ei:
                km.k3moe_set_topp(lay.h, bad)
            assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        km.k3moe_set_topp(lay.h, 0.0)
    finally:
        lay.close()
