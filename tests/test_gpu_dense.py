"""The dense feed-forward layer (the model's layer 0: y = W2 . SiTU(W1 x,
W3 x), width dense_inter; a configuration with no routed part) through the C
ABI against the oracle's dense_ffn: normwise max relative error <= 2e-2 and
cosine >= 0.9995, as for the MoE layer. Decode batches run two tokens per pass
of the TMA-fed kernels, T >= 16 the tcgen05 GEMMs; both at the K3 width
(hidden 7168, dense_inter 33792) and at a small one."""
import numpy as np
import pytest

import k3synth
import oracle
from _harness import Layer, assert_close, bf16_to_f64

pytestmark = pytest.mark.gpu

SMALL = k3synth.dense_shape(1024, 4096)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def k3dense():
    return k3synth.make_dense_layer(k3synth.K3_DENSE, 3)


def run_dense(shape, d, T, seed, residual=False):
    import mxfp4_routed_expert_gb300 as km
    lay = Layer(shape, [d], max_tokens=T)
    try:
        if residual:
            g = k3synth.post_norm_gain(shape, seed)
            km.k3moe_load_post_norm(lay.h, 0, g)
            hres = k3synth.make_residual(shape, seed, T)
            y = lay.forward_residual(hres)
            x = lay.layer_input(T)
            v = oracle.residual_input(hres, g, shape.rms_eps)
            step = np.ldexp(1.0, np.frexp(np.abs(v))[1] - 8)
            assert np.all(np.abs(bf16_to_f64(x) - v) <= step)
        else:
            x = k3synth.make_tokens(shape, seed, T)
            y = lay.forward(x)
    finally:
        lay.close()
    ref = oracle.dense_ffn(x, d["sh_w1"], d["sh_w3"], d["sh_w2"], shape.situ_b1, shape.situ_b2)
    return assert_close(bf16_to_f64(y), ref)


@pytest.mark.parametrize("T", [1, 2, 3, 7, 16, 40, 200, 256, 300, 600])
def test_dense_small(T):
    run_dense(SMALL, k3synth.make_dense_layer(SMALL, 11), T, 11 + T)


# dense_inter 4160 = 32.5 row tiles of 128, hidden 1152 = 9 (the last pair of
# the down projection's paired tiles has its second tile past the matrix):
# the GEMM epilogues write partial row runs
RAGGED = k3synth.dense_shape(1152, 4160)


@pytest.mark.parametrize("T", [200, 300, 600])
def test_dense_ragged_rows(T):
    run_dense(RAGGED, k3synth.make_dense_layer(RAGGED, 13), T, 50 + T)


@pytest.mark.parametrize("T", [1, 2, 5, 20])
def test_dense_k3_width(k3dense, T):
    run_dense(k3synth.K3_DENSE, k3dense, T, 30 + T)


@pytest.mark.parametrize("T", [1, 20])
def test_dense_from_residual(T):
    run_dense(SMALL, k3synth.make_dense_layer(SMALL, 12), T, 40 + T, residual=True)


def test_dense_config_errors():
    import mxfp4_routed_expert_gb300 as km
    lay = Layer(SMALL, [None], max_tokens=4)
    try:
        with pytest.raises(km.K3MoEError) as ei:       # no routed experts to cache
            km.k3moe_set_expert_tier(lay.h, 16)
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
    finally:
        lay.close()
    bad = k3synth.Shape(hidden=1024, latent=0, n_experts=0, topk=8, moe_inter=0,
                        shared_inter=4096)              # a routed field set: not dense, not valid
    with pytest.raises(km.K3MoEError) as ei:
        km.k3moe_create(km.make_config(bad))
    assert ei.value.code == km.K3MOE_ERR_CONFIG


def test_dense_through_host_buffers():
    """k3moe_forward_host on the dense layer: pinned host x and y."""
    import torch
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_dense_layer(SMALL, 13)
    x = k3synth.make_tokens(SMALL, 13, 3)
    lay = Layer(SMALL, [d], max_tokens=3)
    try:
        xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
        yh = torch.empty((3, SMALL.hidden), dtype=torch.int16).pin_memory()
        km.k3moe_forward_host(lay.h, 0, xh, yh, 3)
        y = yh.numpy().view(np.uint16)
    finally:
        lay.close()
    ref = oracle.dense_ffn(x, d["sh_w1"], d["sh_w3"], d["sh_w2"], SMALL.situ_b1, SMALL.situ_b2)
    assert_close(bf16_to_f64(y), ref)
