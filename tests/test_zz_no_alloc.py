"""k3moe_route_static: the router step for callers that may not allocate
device memory (its scratch is a fixed static device array).

Checked against the oracle's router: identical expert id sets, weights to
1e-5, and the selection order wherever two picked scores are more than the
margin guard apart. Each case makes two calls in a row with different tokens,
so that leftovers of the first call in the shared scratch would show; the K3
case (896 experts, hidden 7168) runs at the largest T the array holds. This
file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import k3synth
import oracle
from _harness import MARGIN_TAU, check_ids_and_weights, guarded_tokens, router_only_layer

MID = k3synth.Shape(hidden=1024, latent=512, n_experts=64, topk=8, moe_inter=512,
                    shared_inter=1024)


def _lib():
    import mxfp4_routed_expert_gb300 as km
    from mxfp4_routed_expert_gb300 import build
    build.build()
    return km, km.lib()


def test_route_static_refuses_oversize_without_touching_the_gpu():
    km, lib = _lib()
    fake = ctypes.c_void_p(16)   # never dereferenced: the size check comes first
    T = km.K3MOE_ROUTE_STATIC_MAX_LOGITS // 896 + 1
    rc = lib.k3moe_route_static(fake, fake, None, T, 7168, 896, 16, 1, ctypes.c_float(1.0),
                                fake, fake, None)
    assert rc == km.K3MOE_ERR_SHAPE
    rc = lib.k3moe_route_static(None, fake, None, 1, 7168, 896, 16, 1, ctypes.c_float(1.0),
                                fake, fake, None)
    assert rc == km.K3MOE_ERR_INVALID_ARG


def test_route_static_refuses_unaligned_inputs_without_touching_the_gpu():
    """x and Wr are read in 16-byte chunks: a pointer off a 16-byte boundary is
    refused before any device call (the fake addresses are never used)."""
    km, lib = _lib()
    ok, off = ctypes.c_void_p(256), ctypes.c_void_p(256 + 2)
    for x, wr in ((off, ok), (ok, off)):
        rc = lib.k3moe_route_static(x, wr, None, 1, 7168, 896, 16, 1, ctypes.c_float(1.0),
                                    ok, ok, None)
        assert rc == km.K3MOE_ERR_INVALID_ARG


def _order_agrees(ids_gpu, ids_ref, ch, tau):
    """Within each token, picks whose selection scores differ by more than tau
    come in the oracle's order (descending score)."""
    for t in range(ids_gpu.shape[0]):
        pos = {int(e): j for j, e in enumerate(ids_gpu[t])}
        ref = [int(e) for e in ids_ref[t]]
        for a in range(len(ref)):
            for b in range(a + 1, len(ref)):
                if ch[t, ref[a]] - ch[t, ref[b]] > tau:
                    assert pos[ref[a]] < pos[ref[b]], (t, ref[a], ref[b])


@pytest.mark.gpu
@pytest.mark.parametrize("shape,seed,T", [(k3synth.TINY, 12, 9), (MID, 11, 37),
                                          (k3synth.K3, 13, 1170)])
def test_route_static_matches_oracle(shape, seed, T):
    import torch
    km, _ = _lib()
    assert T * shape.n_experts <= km.K3MOE_ROUTE_STATIC_MAX_LOGITS
    router = k3synth.make_router(shape, seed, 0, k3synth.TINY_RECIPE)
    rshape, d = router_only_layer(shape, router)
    wr = torch.from_numpy(router["router_w"].view(np.int16).copy()).cuda()
    bias = torch.from_numpy(router["router_bias"].copy()).cuda()
    for stream in (0, 1):
        x, _ = guarded_tokens(rshape, d, seed, T, stream=stream)
        ids_ref, w_ref, _, _, ch = oracle.route(rshape, d, x, want_scores=True)
        xd = torch.from_numpy(x.view(np.int16).copy()).cuda()
        ids = torch.full((T, shape.topk), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, shape.topk), -1.0, dtype=torch.float32, device="cuda")
        km.k3moe_route_static(xd, wr, bias, T, shape.hidden, shape.n_experts, shape.topk,
                              shape.renorm, shape.routed_scale, ids, w)
        torch.cuda.synchronize()
        ids_g, w_g = ids.cpu().numpy(), w.cpu().numpy()
        check_ids_and_weights(ids_g, w_g, ids_ref, w_ref)
        _order_agrees(ids_g, ids_ref, ch, MARGIN_TAU)


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["flat", "cut"])
def test_route_static_exact_ties(case):
    """Zero router weights: every score is sigmoid(0) = 0.5 exactly and every
    selection key 0.5 + bias, so experts tie in groups (the bias cases of
    tests/test_gpu_router_ties.py). The picks must be the larger keys first
    and the lower ids among equal keys, in that order, with equal weights."""
    import torch
    from test_gpu_router_ties import expected_ids, tie_bias
    km, _ = _lib()
    shape, T = MID, 5
    bias_np = tie_bias(shape.n_experts, case)
    wr = torch.zeros((shape.n_experts, shape.hidden), dtype=torch.int16, device="cuda")
    bias = torch.from_numpy(bias_np).cuda()
    x = torch.from_numpy(k3synth.make_tokens(shape, 5, T, stream=4).view(np.int16).copy()).cuda()
    ids = torch.full((T, shape.topk), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, shape.topk), -1.0, dtype=torch.float32, device="cuda")
    km.k3moe_route_static(x, wr, bias, T, shape.hidden, shape.n_experts, shape.topk,
                          shape.renorm, shape.routed_scale, ids, w)
    torch.cuda.synchronize()
    want = expected_ids(bias_np, shape.topk)
    ids_g, w_g = ids.cpu().numpy(), w.cpu().numpy()
    for t in range(T):
        np.testing.assert_array_equal(ids_g[t], want, err_msg=f"token {t}")
    np.testing.assert_allclose(w_g, shape.routed_scale / shape.topk, rtol=1e-6)
