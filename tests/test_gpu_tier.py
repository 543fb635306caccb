"""Expert tier through the C ABI (GPU): routed experts held in pinned host
memory and cached in device slots.

Every forward through the tier is checked against the fp64 oracle (ids and
permutation exact, y within the layer tolerance), so an expert read from a
wrong or stale slot fails at once. The tier's hit/miss counters are checked
against the cache policy written out on the host (kimi-k3-in-c README,
Part II section 12, "An LRU cache for the experts": a free slot first, else
the one used longest ago; here ties go to the lower slot, the slots a forward
hits are never its victims, and a forward's misses take its victims in
ascending expert order).
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


def expert_bytes(s):
    I, L, G = s.moe_inter, s.latent, 32
    return 2 * (I * L // 2 + I * L // G) + (L * I // 2 + L * I // G) + 2 * I + L


class LruModel:
    """The slot policy on the host: which (layer, expert) each slot holds and
    the stamp of the forward that last used it (0: never)."""

    def __init__(self, slots, rebase=None):
        self.key = [None] * slots
        self.used = [0] * slots
        self.stamp = 0
        self.hits = 0
        self.misses = 0
        self.rebase = rebase   # (at, keep) of the stamp shift, or None: never
        self.rebases = 0
        self.log = []          # (layer, touched) of every forward

    PIN = 1 << 40   # a pinned slot's stamp: above every forward's

    def forward(self, layer, touched, pin=False):
        if self.rebase and self.stamp >= self.rebase[0]:
            # the last `keep` stamps keep their order, older used slots tie at 1
            shift = self.stamp - self.rebase[1]
            self.used = [u if u in (0, self.PIN) else max(u - shift, 1) for u in self.used]
            self.stamp -= shift
            self.rebases += 1
        self.log.append((layer, tuple(int(e) for e in touched)))
        self.stamp += 1
        where = {k: s for s, k in enumerate(self.key) if k is not None}
        miss = []
        for e in sorted(touched):
            s = where.get((layer, int(e)))
            if s is None:
                miss.append(int(e))
            else:
                if pin:
                    self.used[s] = self.PIN
                elif self.used[s] != self.PIN:
                    self.used[s] = self.stamp
                self.hits += 1
        cand = sorted((self.used[s], s) for s in range(len(self.key)) if self.used[s] < self.stamp)
        assert len(cand) >= len(miss)
        victims = sorted(s for _, s in cand[:len(miss)])
        for e, s in zip(miss, victims):
            self.key[s] = (layer, e)
            self.used[s] = self.PIN if pin else self.stamp
        self.misses += len(miss)


def run_sequence(shape, layers, slots, steps, expert_path=None, max_tokens=64, rebase=None):
    """Forwards (layer, T, seed) through one tiered handle, each against the
    oracle; returns the handle's counters and the model's. rebase: (at, keep)
    given to the handle through K3MOE_TIER_REBASE."""
    import os
    import mxfp4_routed_expert_gb300 as km
    from mxfp4_routed_expert_gb300.tier_trace import replay, trace_from_counts
    if rebase:
        os.environ["K3MOE_TIER_REBASE"] = f"{rebase[0]},{rebase[1]}"
    try:
        lay = Layer(shape, layers, max_tokens=max_tokens, tier_slots=slots)
    finally:
        os.environ.pop("K3MOE_TIER_REBASE", None)
    model = LruModel(slots, rebase)
    trace = []
    try:
        if expert_path is not None:
            km.k3moe_set_expert_path(lay.h, expert_path)
        for layer, T, seed in steps:
            d = layers[layer]
            x, _ = guarded_tokens(shape, d, seed, T)
            y = lay.forward(x, layer=layer)
            r = lay.routing(T)
            ref, tr = oracle.layer_forward(shape, d, x, trace=True)
            check_routing(r, shape, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref, f"y (layer {layer}, T={T})")
            model.forward(layer, np.nonzero(r["counts"])[0])
            trace.append(trace_from_counts(layer, r["counts"]))
        st = km.k3moe_get_tier_stats(lay.h)
    finally:
        lay.close()
    if not rebase:   # the shipped sizing tool replays the same trace to the same counters
        rp = replay(trace, slots, "tier", expert_bytes=expert_bytes(shape))
        assert (rp["hits"], rp["misses"], rp["bytes_copied"]) == (st["hits"], st["misses"], st["bytes_filled"])
    return st, model


def test_tier_decode_sequence_matches_oracle_and_policy():
    """Three layers share E slots (one layer's worth) over single-token and
    3-token forwards (the GEMV path): hits on repeated tokens, free slots taken
    first, then least-recently-used eviction across layers."""
    layers = [k3synth.make_layer(MID, 20 + i, 0, k3synth.TINY_RECIPE) for i in range(3)]
    steps = [(0, 1, 0), (1, 1, 1), (0, 1, 0), (2, 3, 2), (1, 1, 1), (0, 3, 3), (2, 1, 4),
             (2, 1, 4), (1, 3, 5), (0, 1, 0), (2, 3, 6), (1, 1, 7)]
    st, model = run_sequence(MID, layers, MID.n_experts, steps)
    assert st["slots"] == MID.n_experts
    assert model.hits > 0 and model.misses > MID.n_experts   # both hits and evictions happened
    assert (st["hits"], st["misses"]) == (model.hits, model.misses)
    assert st["bytes_filled"] == model.misses * expert_bytes(MID)


def test_tier_stamp_rebase_keeps_the_policy():
    """The slots' 32-bit stamps are shifted down once the count reaches a
    limit; with the limit at 4 and 2 stamps kept (a shift every second
    forward, older slots tied at 1 and taken lower slot first) the handle's
    counters follow the policy with the same shifts and every forward still
    matches the oracle."""
    layers = [k3synth.make_layer(MID, 20 + i, 0, k3synth.TINY_RECIPE) for i in range(3)]
    steps = [(0, 1, 0), (1, 1, 1), (0, 1, 0), (2, 3, 2), (1, 1, 1), (0, 3, 3), (2, 1, 4),
             (2, 1, 4), (1, 3, 5), (0, 1, 0), (2, 3, 6), (1, 1, 7), (0, 3, 3), (1, 3, 5)]
    slots = MID.n_experts + 8
    st, model = run_sequence(MID, layers, slots, steps, rebase=(4, 2))
    assert model.rebases >= 5
    assert (st["hits"], st["misses"]) == (model.hits, model.misses)
    # the tie at 1 changes a victim here: without the shifts the counters differ
    plain = LruModel(slots)
    for layer, touched in model.log:
        plain.forward(layer, touched)
    assert (plain.hits, plain.misses) != (model.hits, model.misses)


def test_tier_rebase_setting_checked(monkeypatch):
    import mxfp4_routed_expert_gb300 as km
    lay = Layer(MID, [None], max_tokens=4)
    try:
        for bad in ("2,2", "3,0", "5", "x,y", "4294967295,2"):
            monkeypatch.setenv("K3MOE_TIER_REBASE", bad)
            with pytest.raises(km.K3MoEError) as ei:
                km.k3moe_set_expert_tier(lay.h, MID.n_experts)
            assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        monkeypatch.setenv("K3MOE_TIER_REBASE", "4,2")
        km.k3moe_set_expert_tier(lay.h, MID.n_experts)
        assert km.k3moe_get_tier_stats(lay.h)["slots"] == MID.n_experts
    finally:
        lay.close()


@pytest.mark.parametrize("path", ["gemm", "gemv"])
def test_tier_batches_evict_whole_layers(path):
    """T = 40 on 128 experts touches most of them: with 128 slots every switch
    of layer evicts most of the other layer's experts. Both expert paths."""
    import mxfp4_routed_expert_gb300 as km
    layers = [k3synth.make_layer(WIDE, 30 + i, 0, k3synth.TINY_RECIPE) for i in range(2)]
    steps = [(0, 40, 0), (1, 40, 1), (0, 40, 0), (0, 17, 2), (1, 40, 3), (1, 40, 3)]
    mode = km.K3MOE_EXPERT_GEMM if path == "gemm" else km.K3MOE_EXPERT_GEMV
    st, model = run_sequence(WIDE, layers, WIDE.n_experts, steps, expert_path=mode)
    assert (st["hits"], st["misses"]) == (model.hits, model.misses)
    assert st["bytes_filled"] == model.misses * expert_bytes(WIDE)


def test_tier_with_room_for_every_layer_only_misses_once():
    """Slots for both layers: after the first forward of each layer nothing is
    evicted, so repeating the same tokens only hits."""
    layers = [k3synth.make_layer(MID, 40 + i, 0, k3synth.TINY_RECIPE) for i in range(2)]
    steps = [(0, 5, 0), (1, 5, 1), (0, 5, 0), (1, 5, 1), (0, 5, 0)]
    st, model = run_sequence(MID, layers, 2 * MID.n_experts, steps)
    assert (st["hits"], st["misses"]) == (model.hits, model.misses)
    # each (layer, expert) was copied in once and never evicted
    assert st["misses"] == sum(k is not None for k in model.key)
    assert st["hits"] > 0


def test_tier_reload_forgets_the_old_experts():
    """Reloading a tiered layer with other weights frees its slots: the next
    forward misses every touched expert and matches the new weights."""
    import mxfp4_routed_expert_gb300 as km
    d0 = k3synth.make_layer(MID, 50, 0, k3synth.TINY_RECIPE)
    d1 = k3synth.make_layer(MID, 51, 0, k3synth.TINY_RECIPE)
    lay = Layer(MID, [d0], max_tokens=8, tier_slots=MID.n_experts)
    try:
        x, _ = guarded_tokens(MID, d0, 3, 4)
        lay.forward(x)
        before = km.k3moe_get_tier_stats(lay.h)
        lay.load(0, d1)
        x1, _ = guarded_tokens(MID, d1, 3, 4)
        y = lay.forward(x1)
        r = lay.routing(4)
        after = km.k3moe_get_tier_stats(lay.h)
    finally:
        lay.close()
    ref, tr = oracle.layer_forward(MID, d1, x1, trace=True)
    check_routing(r, MID, x1, tr["ids"], tr["w"])
    assert_close(bf16_to_f64(y), ref)
    assert after["hits"] == before["hits"]
    assert after["misses"] - before["misses"] == int(np.count_nonzero(r["counts"]))


def test_tier_argument_errors():
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(MID, 52, 0, k3synth.TINY_RECIPE)
    lay = Layer(MID, [None], max_tokens=4)
    try:
        assert km.k3moe_get_tier_stats(lay.h) == dict(slots=0, hits=0, misses=0, bytes_filled=0)
        for bad in (MID.n_experts - 1, -1, 16385):
            with pytest.raises(km.K3MoEError) as ei:
                km.k3moe_set_expert_tier(lay.h, bad)
            assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        km.k3moe_set_expert_tier(lay.h, MID.n_experts)
        km.k3moe_set_expert_tier(lay.h, 0)                 # off again before any load
        km.k3moe_set_expert_tier(lay.h, MID.n_experts + 3)
        lay.load(0, d)
        with pytest.raises(km.K3MoEError) as ei:            # too late: a layer is loaded
            km.k3moe_set_expert_tier(lay.h, MID.n_experts)
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        assert km.k3moe_get_tier_stats(lay.h)["slots"] == MID.n_experts + 3
    finally:
        lay.close()


def test_tier_with_the_topp_cut():
    """The cut drops picks before the tier plans: only kept experts are
    copied in, and the counters follow the policy on the kept sets."""
    import dataclasses
    import mxfp4_routed_expert_gb300 as km
    sh = dataclasses.replace(MID, topp=0.5)
    layers = [k3synth.make_layer(sh, 80 + i, 0, k3synth.TINY_RECIPE) for i in range(2)]
    lay = Layer(sh, layers, max_tokens=8, tier_slots=sh.n_experts)
    model = LruModel(sh.n_experts)
    try:
        km.k3moe_set_topp(lay.h, 0.5)
        for layer, T, seed in [(0, 5, 1), (1, 5, 2), (0, 5, 1), (1, 1, 3)]:
            d = layers[layer]
            x, _ = guarded_tokens(sh, d, seed, T)
            y = lay.forward(x, layer=layer)
            r = lay.routing(T)
            ref, tr = oracle.layer_forward(sh, d, x, trace=True)
            check_routing(r, sh, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref)
            assert int(np.count_nonzero(r["counts"])) <= T * sh.topk
            model.forward(layer, np.nonzero(r["counts"])[0])
        st = km.k3moe_get_tier_stats(lay.h)
    finally:
        lay.close()
    assert (st["hits"], st["misses"]) == (model.hits, model.misses)


def test_tier_with_the_residual_forward():
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(MID, 85, 0, k3synth.TINY_RECIPE)
    g = k3synth.post_norm_gain(MID, 85)
    make = lambda att: oracle.round_bf16(   # noqa: E731
        oracle.residual_input(k3synth.make_residual(MID, 85, 1, 0, att), g, MID.rms_eps))
    _, att = guarded_tokens(MID, d, 85, 1, make=make)
    hres = k3synth.make_residual(MID, 85, 1, 0, att)
    lay = Layer(MID, [d], max_tokens=1, tier_slots=MID.n_experts)
    try:
        km.k3moe_load_post_norm(lay.h, 0, g)
        y = lay.forward_residual(hres)
        x_gpu = lay.layer_input(1)
        r = lay.routing(1)
        st = km.k3moe_get_tier_stats(lay.h)
    finally:
        lay.close()
    ref, tr = oracle.layer_forward(MID, d, x_gpu, trace=True)
    check_routing(r, MID, x_gpu, tr["ids"], tr["w"])
    assert_close(bf16_to_f64(y), ref)
    assert st["misses"] == MID.topk and st["hits"] == 0


def test_tier_chain_matches_the_resident_chain():
    """Two stacked layers through k3moe_forward_chain on a tiered handle (one
    layer's worth of slots) give the resident handle's output."""
    layers = [k3synth.make_layer(k3synth.TINY, 86, i, k3synth.TINY_RECIPE) for i in range(2)]
    x, _ = guarded_tokens(k3synth.TINY, layers[0], 86, 8)
    ys = []
    for slots in (0, k3synth.TINY.n_experts):
        lay = Layer(k3synth.TINY, layers, max_tokens=8, tier_slots=slots)
        try:
            ys.append(bf16_to_f64(lay.forward(x, layer=0, chain=2)))
            ys.append(bf16_to_f64(lay.forward(x, layer=0, chain=2)))   # again: now from the slots
        finally:
            lay.close()
    for y in ys[1:]:
        assert_close(y, ys[0], "tiered chain vs resident chain", rel=2e-3, cos=0.99999)


def test_tier_pinned_layer_only_hits():
    """A pinned layer's experts are copied in once and never evicted: its
    forwards only hit while two other layers churn through the other slots."""
    import mxfp4_routed_expert_gb300 as km
    E = MID.n_experts
    layers = [k3synth.make_layer(MID, 90 + i, 0, k3synth.TINY_RECIPE) for i in range(3)]
    lay = Layer(MID, layers, max_tokens=8, tier_slots=3 * E)
    model = LruModel(3 * E)
    try:
        km.k3moe_tier_pin_layer(lay.h, 0)
        km.k3moe_tier_pin_layer(lay.h, 0)       # again: nothing happens
        model.forward(0, range(E), pin=True)
        assert km.k3moe_get_tier_stats(lay.h)["misses"] == E
        for layer, T, seed in [(1, 8, 1), (0, 8, 2), (2, 8, 3), (1, 8, 4), (0, 8, 5), (2, 8, 6)]:
            d = layers[layer]
            x, _ = guarded_tokens(MID, d, seed, T)
            before = km.k3moe_get_tier_stats(lay.h)["misses"]
            y = lay.forward(x, layer=layer)
            r = lay.routing(T)
            ref, tr = oracle.layer_forward(MID, d, x, trace=True)
            check_routing(r, MID, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref)
            if layer == 0:
                assert km.k3moe_get_tier_stats(lay.h)["misses"] == before
            model.forward(layer, np.nonzero(r["counts"])[0])
        st = km.k3moe_get_tier_stats(lay.h)
    finally:
        lay.close()
    assert (st["hits"], st["misses"]) == (model.hits, model.misses)


def test_tier_pin_needs_room():
    import mxfp4_routed_expert_gb300 as km
    E = MID.n_experts
    d = k3synth.make_layer(MID, 95, 0, k3synth.TINY_RECIPE)
    lay = Layer(MID, [d], max_tokens=4, tier_slots=2 * E - 1)   # the first pin needs 2E
    try:
        with pytest.raises(km.K3MoEError) as ei:   # a pin leaves fewer than E slots to the rest
            km.k3moe_tier_pin_layer(lay.h, 0)
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
    finally:
        lay.close()

