"""Pins of the oracle's dense feed-forward layer (the model's layer 0,
y = W2 . SiTU(W1 x, W3 x); kimi-k3-in-c README Part II, K3Cfg
"first_dense"/"dense_inter", in the SiTU-GLU form of section 9).

- By hand: a two-wide input and a one-wide hidden layer, every product exact.
- Against the layer: a LatentMoE layer whose up projection is zero reduces to
  its shared experts, which are a dense feed-forward layer of width S on the
  same x; the two oracle functions must agree to the bit.
"""
import math

import numpy as np

import k3synth
import oracle


def bf16(v):
    return int(np.float32(v).view(np.uint32) >> 16)


def test_dense_ffn_by_hand():
    # W1 = [[0.5, -1]], W3 = [[2, 0.25]], W2 = [[3], [-0.5]], x = [1, 2]
    W1 = np.array([[bf16(0.5), bf16(-1.0)]], np.uint16)
    W3 = np.array([[bf16(2.0), bf16(0.25)]], np.uint16)
    W2 = np.array([[bf16(3.0)], [bf16(-0.5)]], np.uint16)
    x = np.array([[bf16(1.0), bf16(2.0)]], np.uint16)
    g, u = 0.5 - 2.0, 2.0 + 0.5
    s = 4.0 * math.tanh(g / 4.0) / (1.0 + math.exp(-g)) * 25.0 * math.tanh(u / 25.0)
    y = oracle.dense_ffn(x, W1, W3, W2)
    np.testing.assert_allclose(y, [[3.0 * s, -0.5 * s]], rtol=1e-15)


def test_dense_ffn_is_the_layer_shared_part():
    sh = k3synth.TINY
    d = dict(k3synth.make_layer(sh, 5, 0, k3synth.TINY_RECIPE))
    d["up_w"] = np.zeros_like(d["up_w"])
    x = k3synth.make_tokens(sh, 5, 6)
    y_layer = oracle.layer_forward(sh, d, x)
    y_dense = oracle.dense_ffn(x, d["sh_w1"], d["sh_w3"], d["sh_w2"], sh.situ_b1, sh.situ_b2)
    assert np.array_equal(y_layer, y_dense)


def test_dense_ffn_tokens_are_independent():
    sh = k3synth.dense_shape(64, 96)
    d = k3synth.make_dense_layer(sh, 9)
    x = k3synth.make_tokens(sh, 9, 5)
    y = oracle.dense_ffn(x, d["sh_w1"], d["sh_w3"], d["sh_w2"])
    for t in range(5):
        yt = oracle.dense_ffn(x[t:t + 1], d["sh_w1"], d["sh_w3"], d["sh_w2"])
        assert np.array_equal(yt[0], y[t])
