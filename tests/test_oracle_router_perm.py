"""Pins for the oracle's router and token->expert permutation (CPU only).

Router (kimi-k3-in-c README section 9, k3_router; colibri "Stable LatentMoE"):
a hand-built fixture whose selections are derived by hand below (the bias
changes the picks or their order on 5 of 6 tokens, while the weights stay the
renormalised UNBIASED sigmoid, from scipy's expit), exact ties going to the
lower expert id, renormalised weights summing to 1, routed_scale, and the
page's own selection procedure (repeated strict-'>' maximum) re-run as brute
force on random tokens. Permutation: the canonical (expert, token, slot)
order equals a stable library sort of the flat id list.
"""
import numpy as np
import pytest
from scipy.special import expit

import k3synth
import oracle

ONE = 0x3F80  # bf16 bit patterns of small exact values
BF = {1.0: 0x3F80, -1.0: 0xBF80, 0.5: 0x3F00, 2.0: 0x4000, -2.0: 0xC000, 4.0: 0x4080,
      0.0: 0x0000}


def _bf(vals):
    return np.array([BF[v] for v in vals], np.uint16)


# 4 experts over a 2-wide input; bias only on experts 2 and 3.
WR = np.stack([_bf([1.0, 0.0]), _bf([0.0, 1.0]), _bf([0.5, 0.5]), _bf([-1.0, 0.0])])
BIAS = np.array([0.0, 0.0, 0.3, 0.6], np.float32)

# token -> (expected ids with bias, expected ids without bias), top-2, derived by
# hand from logits = Wr x, sc = sigmoid(logit), ch = sc + bias.
CASES = [
    ((2.0, 0.0), [2, 0], [0, 2]),   # logits  2, 0, 1,-2: same pair, order flipped
    ((0.0, 2.0), [3, 2], [1, 2]),   # logits  0, 2, 1, 0: bias swaps in expert 3
    ((-2.0, 0.0), [3, 2], [3, 1]),  # logits -2, 0,-1, 2
    ((0.0, 0.0), [3, 2], [0, 1]),   # all logits 0: unbiased is a 4-way tie -> 0, 1
    ((4.0, 4.0), [2, 0], [0, 1]),   # experts 0 and 1 tie exactly -> lower id first
    ((1.0, -1.0), [3, 2], [0, 2]),  # logits 1,-1, 0,-1
]


@pytest.mark.parametrize("x,with_bias,without_bias", CASES)
def test_router_fixture_bias_selects_only(x, with_bias, without_bias):
    xv = np.array(x, np.float64)
    logits = np.array([xv @ np.array([1.0, 0.0]), xv @ np.array([0.0, 1.0]),
                       xv @ np.array([0.5, 0.5]), xv @ np.array([-1.0, 0.0])])
    sc = expit(logits)

    ids, w, sc_o, ch_o, margin = oracle.router_token(xv, WR, BIAS, 2)
    assert list(ids) == with_bias
    np.testing.assert_allclose(sc_o, sc, rtol=1e-15)
    np.testing.assert_allclose(ch_o, sc + BIAS.astype(np.float64), rtol=1e-15)
    # the weights are the UNBIASED scores of the winners, renormalised
    np.testing.assert_allclose(w, sc[with_bias] / sc[with_bias].sum(), rtol=1e-15)
    assert margin >= 0.0

    ids0, w0, _, _, _ = oracle.router_token(xv, WR, None, 2)
    assert list(ids0) == without_bias
    np.testing.assert_allclose(w0, sc[without_bias] / sc[without_bias].sum(), rtol=1e-15)


def test_bias_changes_picks_on_five_of_six_tokens():
    changed = sum(1 for _, a, b in CASES if a != b)
    assert changed == 6 and sum(1 for _, a, b in CASES if set(a) != set(b)) == 5


def test_exact_ties_go_to_lower_id():
    E, H = 9, 3
    W = np.tile(_bf([1.0, 0.5, 0.0]), (E, 1))          # identical rows -> identical scores
    ids, w, _, _, margin = oracle.router_token(np.array([1.0, 1.0, 1.0]), W, None, 4)
    assert list(ids) == [0, 1, 2, 3]
    assert margin == 0.0
    np.testing.assert_allclose(w, 0.25, rtol=1e-15)


def _page_selection(ch, k):
    """The README's procedure: k passes, each taking the untaken expert with the
    largest selection score (strict '>', so the first of equal scores wins)."""
    taken = np.zeros(ch.size, bool)
    out = []
    for _ in range(k):
        best = -1
        for e in range(ch.size):
            if not taken[e] and (best < 0 or ch[e] > ch[best]):
                best = e
        taken[best] = True
        out.append(best)
    return out


def test_sort_equals_repeated_max_and_weights_sum_to_one():
    shape = k3synth.replace(k3synth.TINY, n_experts=64, topk=6, hidden=96)
    layer = k3synth.make_layer(shape, 3, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 3, 40)
    ids, w, margin, sc, ch = oracle.route(shape, layer, x, want_scores=True)
    for t in range(40):
        assert list(ids[t]) == _page_selection(ch[t], shape.topk)
        assert abs(w[t].sum() - 1.0) < 1e-15
        np.testing.assert_allclose(w[t], sc[t, ids[t]] / sc[t, ids[t]].sum(), rtol=1e-15)
        srt = np.sort(ch[t])[::-1]
        assert margin[t] == srt[shape.topk - 1] - srt[shape.topk]
    # logits against the library matmul
    xf = k3synth.bf16_bits_to_f32(x).astype(np.float64)
    Wf = k3synth.bf16_bits_to_f32(layer["router_w"]).astype(np.float64)
    np.testing.assert_allclose(sc, expit(xf @ Wf.T), rtol=1e-13)


def test_routed_scale_and_no_renorm():
    shape = k3synth.replace(k3synth.TINY, routed_scale=2.5)
    layer = k3synth.make_layer(shape, 4, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 4, 5)
    _, w, _ = oracle.route(shape, layer, x)
    np.testing.assert_allclose(w.sum(1), 2.5, rtol=1e-15)
    shape0 = k3synth.replace(k3synth.TINY, renorm=0)
    ids, w0, _, sc, _ = oracle.route(shape0, layer, x, want_scores=True)
    np.testing.assert_array_equal(w0, np.take_along_axis(sc, ids.astype(np.int64), 1))


def test_all_experts_when_k_equals_E():
    shape = k3synth.replace(k3synth.TINY, n_experts=8, topk=8)
    layer = k3synth.make_layer(shape, 5, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 5, 3)
    ids, w, margin = oracle.route(shape, layer, x)
    for t in range(3):
        assert sorted(ids[t]) == list(range(8))
    assert np.all(np.isinf(margin))


def test_permutation_is_stable_sort_of_flat_ids():
    rng_ids = (k3synth.words(200 * 5, k3synth.key(6, 1)) % 17).astype(np.int32)
    ids = rng_ids.reshape(200, 5)
    counts, offsets, perm = oracle.permutation(ids, 17)
    flat = ids.ravel()
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=17))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))


def test_permutation_of_router_ids():
    shape = k3synth.TINY
    layer = k3synth.make_layer(shape, 0, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 0, 13)
    ids, _, _ = oracle.route(shape, layer, x)
    counts, offsets, perm = oracle.permutation(ids, shape.n_experts)
    assert offsets[-1] == 13 * shape.topk
    assert sorted(perm) == list(range(13 * shape.topk))
    for e in range(shape.n_experts):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(ids.ravel()[seg] == e)
        assert np.all(np.diff(seg // shape.topk) > 0)      # tokens ascending, each once


# ---- the cumulative-weight cut of the picks (the pages' K3_TOPP option) ----------------

def test_topp_cut_by_hand():
    # selection order ids [7, 3, 9, 1], weights 1/2, 1/4, 1/8, 1/8 (exact in binary);
    # weight order 7, 3, then 1 before 9 (equal weights: lower id first)
    ids, w = [7, 3, 9, 1], [0.5, 0.25, 0.125, 0.125]
    i2, w2, m, _ = oracle.topp_cut(ids, w, 0.75)      # before: 0, 1/2, 3/4 (not < 3/4)
    assert m == 2 and i2.tolist() == [7, 3, -1, -1]
    np.testing.assert_allclose(w2, [2 / 3, 1 / 3, 0, 0], rtol=1e-15)
    i3, w3, m3, _ = oracle.topp_cut(ids, w, 0.76)     # 3/4 < 0.76: expert 1 stays too
    assert m3 == 3 and i3.tolist() == [7, 3, 1, -1]
    np.testing.assert_allclose(w3, [0.5 / 0.875, 0.25 / 0.875, 0.125 / 0.875, 0], rtol=1e-15)


def test_topp_cut_ties_go_to_lower_ids_and_first_pick_stays():
    i2, w2, m, _ = oracle.topp_cut([5, 2, 8, 4], [0.25] * 4, 0.5)   # order 2, 4, 5, 8
    assert m == 2 and i2.tolist() == [2, 4, -1, -1]
    np.testing.assert_allclose(w2, [0.5, 0.5, 0, 0], rtol=1e-15)
    i1, w1, m1, _ = oracle.topp_cut([5, 2, 8, 4], [0.1, 0.4, 0.3, 0.2], 1e-9)
    assert m1 == 1 and i1.tolist() == [2, -1, -1, -1]
    np.testing.assert_allclose(w1, [1.0, 0, 0, 0], rtol=1e-15)        # scaled back to the total


def test_topp_cut_one_keeps_all_but_a_zero_tail_and_reports_its_margin():
    i, w, m, mg = oracle.topp_cut([1, 2, 3], [0.6, 0.4, 0.0], 1.0)   # before 1.0 is not < 1.0
    assert m == 2 and i.tolist() == [1, 2, -1]
    np.testing.assert_allclose(w, [0.6, 0.4, 0.0], rtol=1e-15)
    assert mg == 0.0
    _, _, _, mg2 = oracle.topp_cut([7, 3, 9, 1], [0.5, 0.25, 0.125, 0.125], 0.7)
    np.testing.assert_allclose(mg2, 0.05, rtol=1e-12)                   # |3/4 - 0.7|
