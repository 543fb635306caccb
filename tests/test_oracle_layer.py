"""Whole-layer pins for the oracle on the tiny LatentMoE layer (CPU only).

The pages print no worked numeric example of a full layer, so the layer is
pinned by a second, structurally different route and by invariants of the
method (kimi-k3-in-c README section 9, k3_moe; colibri "Stable LatentMoE"):
  - a dense fp64 route: every expert dequantised to a dense matrix, every
    expert run on every token, combined through a dense gate matrix that is
    zero off the top-k (library matmul/einsum, scipy expit, numpy lexsort);
  - token permutation equivariance and expert relabelling invariance;
  - with every expert scale set to 255 only the shared experts remain, and
    they act on the original x, unweighted;
  - without the latent norm the routed part is linear in routed_scale; with
    it (eps = 0) the output does not depend on routed_scale, because the norm
    is taken on the aggregate.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

import k3synth
import oracle

SH = k3synth.TINY
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return k3synth.bf16_bits_to_f32(bits).astype(np.float64)


def decode_experts(packed, scales):
    with open(os.path.join(GOLD, "mxfp4_format.json")) as f:
        lut = np.array(json.load(f)["e2m1_lut"])
    E, R, C2 = packed.shape
    v = np.empty((E, R, 2 * C2))
    v[..., 0::2] = lut[packed & 15]
    v[..., 1::2] = lut[packed >> 4]
    s = np.where(scales == 255, 0.0, np.ldexp(1.0, scales.astype(np.int64) - 127))
    return v * np.repeat(s, 32, axis=2)


def situ_np(g, u, b1, b2):
    return b1 * np.tanh(g / b1) * expit(g) * b2 * np.tanh(u / b2)


def dense_route(shape, d, x_bits):
    X = f64(x_bits)
    T, E, K = X.shape[0], shape.n_experts, shape.topk
    sc = expit(X @ f64(d["router_w"]).T)
    ch = sc + d["router_bias"].astype(np.float64)[None, :]
    G = np.zeros((T, E))
    for t in range(T):
        sel = np.lexsort((np.arange(E), -ch[t]))[:K]
        w = sc[t, sel]
        if shape.renorm and w.sum() > 0:
            w = w / w.sum()
        G[t, sel] = w * shape.routed_scale
    Z = X @ f64(d["down_w"]).T
    W1 = decode_experts(d["w1p"], d["w1s"])
    W3 = decode_experts(d["w3p"], d["w3s"])
    W2 = decode_experts(d["w2p"], d["w2s"])
    A = situ_np(np.einsum("tl,eil->tei", Z, W1), np.einsum("tl,eil->tei", Z, W3),
                shape.situ_b1, shape.situ_b2)
    O = np.einsum("tei,eli->tel", A, W2)
    acc = np.einsum("te,tel->tl", G, O)
    if d.get("latent_gain") is not None:
        ms = np.mean(acc * acc, axis=1, keepdims=True)
        acc = acc / np.sqrt(ms + shape.rms_eps) * f64(d["latent_gain"])[None, :]
    S = situ_np(X @ f64(d["sh_w1"]).T, X @ f64(d["sh_w3"]).T, shape.situ_b1, shape.situ_b2)
    return acc @ f64(d["up_w"]).T + S @ f64(d["sh_w2"]).T, G


@pytest.fixture(scope="module")
def tiny():
    d = k3synth.make_layer(SH, 0, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(SH, 0, 4)
    return d, x


def relerr(a, b):
    return np.abs(a - b).max() / np.abs(b).max()


def test_dense_route_matches(tiny):
    d, x = tiny
    y, tr = oracle.layer_forward(SH, d, x, trace=True)
    ref, G = dense_route(SH, d, x)
    assert relerr(y, ref) < 1e-12
    for t in range(x.shape[0]):
        np.testing.assert_array_equal(np.sort(tr["ids"][t]), np.sort(np.nonzero(G[t])[0]))
        np.testing.assert_allclose(tr["w"][t], G[t, tr["ids"][t]], rtol=1e-14)
    assert np.abs(tr["h"]).max() <= SH.situ_b1 * SH.situ_b2


def test_dense_route_more_tokens_and_experts():
    shape = k3synth.replace(SH, n_experts=48, topk=6)
    d = k3synth.make_layer(shape, 1, 2, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 1, 33)
    assert relerr(oracle.layer_forward(shape, d, x), dense_route(shape, d, x)[0]) < 1e-12


def test_row_subset_and_token_permutation(tiny):
    d, x = tiny
    y = oracle.layer_forward(SH, d, x)
    perm = np.array([2, 0, 3, 1])
    np.testing.assert_array_equal(oracle.layer_forward(SH, d, x[perm]), y[perm])
    np.testing.assert_array_equal(oracle.layer_forward(SH, d, x, rows=[3, 1]), y[[3, 1]])


def test_expert_relabelling(tiny):
    d, x = tiny
    y, tr = oracle.layer_forward(SH, d, x, trace=True)
    pi = np.roll(np.arange(SH.n_experts), 5)[::-1].copy()     # new slot i holds old expert pi[i]
    d2 = dict(d)
    for k in ("router_w", "router_bias", "w1p", "w1s", "w3p", "w3s", "w2p", "w2s"):
        d2[k] = np.ascontiguousarray(d[k][pi])
    y2, tr2 = oracle.layer_forward(SH, d2, x, trace=True)
    np.testing.assert_allclose(y2, y, rtol=0, atol=1e-14 * np.abs(y).max())
    np.testing.assert_array_equal(pi[tr2["ids"]], tr["ids"])


def test_shared_experts_only(tiny):
    d, x = tiny
    d2 = dict(d)
    for k in ("w1s", "w3s", "w2s"):
        d2[k] = np.full_like(d[k], 255)           # every routed group decodes to 0
    y = oracle.layer_forward(SH, d2, x)
    X = f64(x)
    S = situ_np(X @ f64(d["sh_w1"]).T, X @ f64(d["sh_w3"]).T, SH.situ_b1, SH.situ_b2)
    np.testing.assert_allclose(y, S @ f64(d["sh_w2"]).T, rtol=1e-13, atol=1e-15)


def test_routed_part_linear_without_norm_and_scale_free_with_norm(tiny):
    d, x = tiny
    no_norm = dict(d)
    no_norm["latent_gain"] = None
    base = dict(d)
    for k in ("w1s", "w3s", "w2s"):
        base[k] = np.full_like(d[k], 255)
    shared = oracle.layer_forward(SH, base, x)
    y1 = oracle.layer_forward(SH, no_norm, x)
    y3 = oracle.layer_forward(k3synth.replace(SH, routed_scale=3.0), no_norm, x)
    np.testing.assert_allclose(y3 - shared, 3.0 * (y1 - shared), rtol=1e-12,
                               atol=1e-13 * np.abs(y1 - shared).max())
    s0 = k3synth.replace(SH, rms_eps=0.0)
    a = oracle.layer_forward(s0, d, x)
    b = oracle.layer_forward(k3synth.replace(s0, routed_scale=3.0), d, x)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13 * np.abs(a).max())


def test_trace_consistency(tiny):
    d, x = tiny
    _, tr = oracle.layer_forward(SH, d, x, trace=True)
    gain = f64(d["latent_gain"])
    for t in range(x.shape[0]):
        np.testing.assert_allclose(tr["nrm"][t], oracle.rmsnorm(tr["acc"][t], gain, SH.rms_eps),
                                   rtol=1e-15)
        np.testing.assert_allclose(tr["z"][t], f64(d["down_w"]) @ f64(x[t]), rtol=1e-12,
                                   atol=1e-15)


def test_chain_glue_unit_gain():
    y = k3synth.normal_f64((3, 64), k3synth.key(12, 1))
    out = oracle.chain_glue(y, 1e-5)
    for t in range(3):
        np.testing.assert_allclose(out[t], y[t] / np.sqrt(np.mean(y[t] ** 2) + 1e-5), rtol=1e-14)
