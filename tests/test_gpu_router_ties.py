"""Exact ties in the router selection, on the GPU paths (through the C ABI).

With every router weight zero, every logit is exactly 0 and every score
sigmoid(0) = 0.5, so a selection key is 0.5 + bias exactly, in the kernels'
fp32 as in the oracle's fp64, for the bias values used here (0, 0.25, 0.5).
Whole groups of experts then tie. The rule (kimi-k3-in-c README, Part II
section 9, k3_router: the top k taken as repeated strict maxima) takes the
larger keys first and, among equal keys, the lower expert ids. The expected
selection is written out here from that rule alone, and the GPU's ids must
equal it in order, besides matching the oracle (ids, permutation, weights)
and y within the layer's tolerance. The weights come out exactly equal
(0.5 / (k 0.5) each, times the routed scale).

The cases cover ties that all fall inside the selection and ties that
straddle its end, at T = 1 (the router epilogue writes the permutation
itself), at a decode batch on the GEMVs and at batches on both grouped GEMMs.
Since every token routes alike, each chosen expert gets all T tokens (several
n-tiles at T = 64 and 200).
"""
import numpy as np
import pytest

import k3synth
import oracle
from _harness import Layer, assert_close, bf16_to_f64, check_routing
from test_gpu_parity import MID, WIDE, _mode


@pytest.fixture(scope="module")
def _built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


def tie_bias(E, case):
    """Bias with exact ties: 'flat' (every key equal) or 'cut' (three experts
    at 0.5, ten at 0.25 across the ids, the rest 0, so the 0.25 group straddles
    the end of a top-8)."""
    b = np.zeros(E, np.float32)
    if case == "cut":
        b[[40, 9, 33]] = 0.5
        b[[5, 50, 17, 61, 2, 30, 44, 12, 58, 21]] = 0.25
    return b


def expected_ids(bias, k):
    """The first k experts by (0.5 + bias descending, id ascending)."""
    keys = 0.5 + bias.astype(np.float64)
    order = sorted(range(len(bias)), key=lambda e: (-keys[e], e))
    return np.asarray(order[:k], np.int32)


@pytest.mark.gpu
@pytest.mark.parametrize("shape,T,path", [("mid", 1, None), ("mid", 5, None), ("wide", 1, None),
                                          ("wide", 64, None), ("wide", 64, "gemm"),
                                          ("wide", 200, "mx")])
@pytest.mark.parametrize("case", ["flat", "cut"])
def test_router_exact_ties(_built, shape, T, path, case):
    import mxfp4_routed_expert_gb300 as km
    sh = {"mid": MID, "wide": WIDE}[shape]
    d = dict(k3synth.make_layer(sh, 31, 0, k3synth.TINY_RECIPE))
    d["router_w"] = np.zeros_like(d["router_w"])
    bias = tie_bias(sh.n_experts, case)
    d = k3synth.with_bias(d, bias)
    x = k3synth.make_tokens(sh, 31, T, stream=3)
    lay = Layer(sh, [d], max_tokens=T)
    try:
        if path is not None:
            km.k3moe_set_expert_path(lay.h, _mode(path))
        y = lay.forward(x)
        r = lay.routing(T)
    finally:
        lay.close()
    want = expected_ids(bias, sh.topk)
    for t in range(T):
        np.testing.assert_array_equal(r["ids"][t], want, err_msg=f"token {t}")
    np.testing.assert_allclose(r["w"], 1.0 / sh.topk * sh.routed_scale, rtol=1e-6)
    ref, tr = oracle.layer_forward(sh, d, x, trace=True)
    np.testing.assert_array_equal(np.asarray(tr["ids"]), np.broadcast_to(want, (T, sh.topk)))
    check_routing(r, sh, x, tr["ids"], tr["w"])
    assert_close(bf16_to_f64(y), ref, f"y with tied selection keys ({case}, T={T})")


def test_tie_fixture_expectations():
    """The expected selections of the two cases, by hand (CPU)."""
    np.testing.assert_array_equal(expected_ids(tie_bias(64, "flat"), 8), np.arange(8))
    np.testing.assert_array_equal(expected_ids(tie_bias(64, "cut"), 8), [9, 33, 40, 2, 5, 12, 17, 21])
