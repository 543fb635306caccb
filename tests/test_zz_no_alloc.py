"""k3moe_route_static: the router step for callers that may not allocate
device memory (its scratch is a fixed static device array).

Checked against the routing that k3moe_forward produces for the same tokens,
with the tolerances of the other parity tests (identical expert id sets,
weights to 1e-5), on two calls in a row with different tokens so that
leftovers of the first call in the shared scratch would show. This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import k3synth
from _harness import Layer, check_routing, guarded_tokens

MID = k3synth.Shape(hidden=1024, latent=512, n_experts=64, topk=8, moe_inter=512,
                    shared_inter=1024)


def test_route_static_refuses_oversize_without_touching_the_gpu():
    import mxfp4_routed_expert_gb300 as km
    from mxfp4_routed_expert_gb300 import build
    build.build()
    lib = km.lib()
    fake = ctypes.c_void_p(16)   # never dereferenced: the size check comes first
    T = km.K3MOE_ROUTE_STATIC_MAX_LOGITS // 896 + 1
    rc = lib.k3moe_route_static(fake, fake, None, T, 7168, 896, 16, 1, ctypes.c_float(1.0),
                                fake, fake, None)
    assert rc == km.K3MOE_ERR_SHAPE
    rc = lib.k3moe_route_static(None, fake, None, 1, 7168, 896, 16, 1, ctypes.c_float(1.0),
                                fake, fake, None)
    assert rc == km.K3MOE_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("shape,seed,T", [(MID, 11, 37), (k3synth.TINY, 12, 9)])
def test_route_static_matches_forward_routing(shape, seed, T):
    import torch
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(shape, seed, 0, k3synth.TINY_RECIPE)
    lay = Layer(shape, [d], max_tokens=T)
    wr = torch.from_numpy(d["router_w"].view(np.int16).copy()).cuda()
    bias = torch.from_numpy(d["router_bias"].copy()).cuda()
    try:
        for call, stream in enumerate((0, 1)):
            x, _ = guarded_tokens(shape, d, seed, T, stream=stream)
            lay.forward(x)
            ref = lay.routing(T)
            xd = torch.from_numpy(x.view(np.int16).copy()).cuda()
            ids = torch.full((T, shape.topk), -1, dtype=torch.int32, device="cuda")
            w = torch.full((T, shape.topk), -1.0, dtype=torch.float32, device="cuda")
            km.k3moe_route_static(xd, wr, bias, T, shape.hidden, shape.n_experts, shape.topk,
                                  shape.renorm, shape.routed_scale, ids, w)
            torch.cuda.synchronize()
            got = dict(ref)
            got["ids"], got["w"] = ids.cpu().numpy(), w.cpu().numpy()
            # same id sets and weights as the forward's routing (which the oracle pins)
            check_routing(got, shape, x, ref["ids"], ref["w"])
            # and the same selection order
            np.testing.assert_array_equal(got["ids"], ref["ids"])
    finally:
        lay.close()
