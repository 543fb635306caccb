"""CUDA path vs the fp64 oracle, through the C ABI (GPU).

Ids and the permutation must match exactly (inputs pass the routing margin
guard); y, z, the latent aggregate and the shared-expert activations must be
within normwise max relative error 2e-2 and cosine >= 0.9995.
"""
import numpy as np
import pytest

import k3synth
import oracle
from _harness import (Layer, assert_close, bf16_to_f64, check_routing, guarded_tokens)

pytestmark = pytest.mark.gpu

MID = k3synth.Shape(hidden=1024, latent=512, n_experts=64, topk=8, moe_inter=512,
                    shared_inter=1024)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


def run_case(shape, recipe, seed, T, stream=0, check_intermediates=True, expert_path=None,
             d=None):
    import mxfp4_routed_expert_gb300 as km
    if d is None:
        d = k3synth.make_layer(shape, seed, 0, recipe)
    x, _ = guarded_tokens(shape, d, seed, T, stream)
    lay = Layer(shape, [d], max_tokens=T)
    try:
        if expert_path is not None:
            km.k3moe_set_expert_path(lay.h, expert_path)
        y = lay.forward(x)
        r = lay.routing(T)
        z = lay.intermediate(km.K3MOE_T_Z, T, shape.latent)
        acc = lay.intermediate(km.K3MOE_T_ACC, T, shape.latent)
        sh = lay.intermediate(km.K3MOE_T_SHARED, T, shape.shared_inter)
    finally:
        lay.close()
    ref, tr = oracle.layer_forward(shape, d, x, trace=True)
    check_routing(r, shape, x, tr["ids"], tr["w"])
    if check_intermediates:
        assert_close(z, tr["z"], "z", rel=1e-4, cos=0.9999999)
        assert_close(sh, tr["shared"], "shared SiTU", rel=1e-3, cos=0.99999)
        assert_close(acc, tr["acc"], "latent aggregate")
    return assert_close(bf16_to_f64(y), ref)


@pytest.mark.parametrize("T", [4, 1, 2, 3, 37])
def test_tiny(T):
    run_case(k3synth.TINY, k3synth.TINY_RECIPE, 0, T)


@pytest.mark.parametrize("T", [1, 5, 33])
def test_mid_shape(T):
    run_case(MID, k3synth.TINY_RECIPE, 1, T)


# 128 experts: every weight matrix has at least 128 rows, so T >= 16 runs the
# dense projections on the tcgen05 tensor-core GEMMs (T <= 128 with split-K)
WIDE = k3synth.Shape(hidden=1024, latent=512, n_experts=128, topk=8, moe_inter=512,
                     shared_inter=1024)


@pytest.mark.parametrize("T", [16, 37, 100, 300, 600, 1030])
def test_tensor_core_dense_path(T):
    """From 512 tokens router+down and up+shared-down take two m-tiles per CTA
    (WIDE: 5 router+down m-tiles, so the last pair's second tile lies past the
    matrix and reads zeros)."""
    run_case(WIDE, k3synth.TINY_RECIPE, 6, T)


# Row counts that are not multiples of the 128-row tiles: 130 experts (a
# router tile of 2 rows, whose fp32 logit rows of 520 bytes are not 16-byte
# multiples, and router+down partial sums of 706 rows that are not either),
# latent 576, shared 1088, hidden 1152 (9 row tiles, so the last pair of
# paired tiles has its second tile past the matrix); T = 40 and 200 split K
RAGGED = k3synth.Shape(hidden=1152, latent=576, n_experts=130, topk=8, moe_inter=512,
                       shared_inter=1088)


@pytest.mark.parametrize("T", [40, 200, 300, 600])
def test_tensor_core_dense_ragged_rows(T):
    run_case(RAGGED, k3synth.TINY_RECIPE, 8, T)


def _mode(path):
    import mxfp4_routed_expert_gb300 as km
    return {"gemm": km.K3MOE_EXPERT_GEMM, "gemv": km.K3MOE_EXPERT_GEMV, "mx": km.K3MOE_EXPERT_MX}[path]


@pytest.mark.parametrize("T,path", [(16, "gemm"), (37, "gemv"), (300, "gemv"), (20, "gemm"), (16, "mx"),
                                    (300, "mx")])
def test_expert_paths(T, path):
    """The routed-expert paths against the oracle: the per-pair GEMVs, the
    grouped tcgen05 GEMM and its block-scaled form (T=16 with topk 8 is the
    grouped GEMMs' smallest batch, 128 pairs)."""
    run_case(WIDE, k3synth.TINY_RECIPE, 6, T, expert_path=_mode(path))


@pytest.mark.parametrize("E,k,T,path", [(16, 16, 1, None), (16, 16, 5, None), (16, 16, 16, "mx"),
                                        (16, 16, 16, "gemm"), (32, 1, 1, None), (32, 1, 3, None),
                                        (32, 1, 130, "mx"), (32, 1, 130, "gemm")])
def test_degenerate_topk(E, k, T, path):
    """The degenerate selections: every expert picked (k = E, so the weights
    are all experts' renormalised scores and every expert holds every token)
    and a single pick (k = 1, weight 1 after renormalisation). T = 1 writes
    the permutation in the router epilogue, small batches run the GEMVs, and
    128 pairs and more the grouped GEMMs."""
    sh = k3synth.Shape(hidden=256, latent=128, n_experts=E, topk=k, moe_inter=128, shared_inter=256)
    run_case(sh, k3synth.TINY_RECIPE, 14, T, expert_path=_mode(path) if path else None)


@pytest.mark.parametrize("T,path", [(1, None), (5, None), (40, None), (40, "mx"), (40, "gemm")])
def test_max_routing_shape(T, path):
    """The largest routing the library accepts: 1024 experts, top-32 (the
    router keeps 32 scores per lane; the permutation's histogram and placement
    warps then stage 32-token chunks of 32 ids and weights each beside 1024
    counters)."""
    sh = k3synth.Shape(hidden=256, latent=128, n_experts=1024, topk=32, moe_inter=128, shared_inter=256)
    run_case(sh, k3synth.TINY_RECIPE, 15, T, expert_path=_mode(path) if path else None)


@pytest.mark.parametrize("shape,T", [("tiny", 1), ("tiny", 4), ("mid", 1), ("mid", 5), ("wide", 1),
                                     ("wide", 7), ("wide", 15)])
def test_block_scaled_small_batches(shape, T):
    """The block-scaled grouped GEMM below its whole-item range (fewer than
    128 pairs): every item's K range is split, W2 parts add into the latent
    aggregate like whole items and W1/W3 parts meet in a partial-sum buffer
    whose last arrival applies SiTU. 4 to 120 pairs, one to several pairs per
    expert, against the oracle."""
    sh = {"tiny": k3synth.TINY, "mid": MID, "wide": WIDE}[shape]
    run_case(sh, k3synth.TINY_RECIPE, 9, T, expert_path=_mode("mx"))


@pytest.mark.parametrize("path", ["gemm", "gemv", "mx"])
def test_expert_gemm_multi_tile(path):
    """Four experts forced into every token's selection (+10 router bias): each
    holds all 300 tokens, five n-tiles of the grouped GEMM (2400 pairs on 128
    experts take 64-pair tiles: 4 x 64 + 44)."""
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(WIDE, 8, 0, k3synth.TINY_RECIPE)
    bias = np.asarray(d["router_bias"], np.float32).copy()
    bias[[3, 40, 77, 127]] += 10.0
    d = k3synth.with_bias(d, bias)
    run_case(WIDE, k3synth.TINY_RECIPE, 8, 300, expert_path=_mode(path), d=d)


@pytest.mark.parametrize("T,path", [(40, "gemm"), (64, "gemm"), (40, "mx"), (64, "mx")])
def test_expert_gemm_narrow_ntiles(T, path):
    """At most four pairs per expert on average (T*8 <= 4*128) selects 32-pair
    n-tiles; four experts forced into every selection then hold T pairs each,
    two n-tiles (32 + 8 at T=40, 32 + 32 at T=64)."""
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(WIDE, 10, 0, k3synth.TINY_RECIPE)
    bias = np.asarray(d["router_bias"], np.float32).copy()
    bias[[5, 50, 90, 126]] += 10.0
    d = k3synth.with_bias(d, bias)
    run_case(WIDE, k3synth.TINY_RECIPE, 10, T, expert_path=_mode(path), d=d)


# latent 384: three 128-row m-tiles of W2, which the grouped GEMM runs one per
# item with the k-stage split across its two MMA issuers (no m-tile pairing)
ODD_LATENT = k3synth.Shape(hidden=1024, latent=384, n_experts=128, topk=8, moe_inter=512,
                           shared_inter=1024)


@pytest.mark.parametrize("T,path", [(48, "gemm"), (200, "gemm"), (48, "mx"), (200, "mx")])
def test_expert_gemm_unpaired_w2(T, path):
    """The unpaired W2 mode at 32-pair (T=48) and 64-pair (T=200) n-tiles."""
    run_case(ODD_LATENT, k3synth.TINY_RECIPE, 11, T, expert_path=_mode(path))


@pytest.mark.parametrize("hot,path", [(False, "gemm"), (True, "gemm"), (False, "mx"), (True, "mx")])
def test_expert_gemm_wide_ntiles(hot, path):
    """T=1100 on the 128-expert shape: 8800 pairs, at least 64 per expert on
    average, so the grouped GEMM cuts 128-pair n-tiles. With four experts forced
    into every selection each of them holds 1100 pairs (nine n-tiles)."""
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(WIDE, 9, 0, k3synth.TINY_RECIPE)
    if hot:
        bias = np.asarray(d["router_bias"], np.float32).copy()
        bias[[0, 31, 64, 100]] += 10.0
        d = k3synth.with_bias(d, bias)
    run_case(WIDE, k3synth.TINY_RECIPE, 9, 1100, expert_path=_mode(path), d=d,
             check_intermediates=not hot)


def test_expert_path_selection_and_errors():
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(WIDE, 6, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(WIDE, 6, 37)
    lay = Layer(WIDE, [d], max_tokens=37)
    try:
        with pytest.raises(km.K3MoEError) as ei:
            km.k3moe_set_expert_path(lay.h, 7)
        assert ei.value.code == km.K3MOE_ERR_INVALID_ARG
        km.k3moe_set_profiling(lay.h, True)
        lay.forward(x)                                   # auto: 296 pairs -> grouped GEMM
        auto = {s[0] for s in km.k3moe_profile_read(lay.h)}
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_GEMV)
        lay.forward(x)
        gemv = {s[0] for s in km.k3moe_profile_read(lay.h)}
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_GEMM)
        lay.forward(x[:8])                               # 64 pairs: below one n-tile -> GEMVs
        small = {s[0] for s in km.k3moe_profile_read(lay.h)}
        km.k3moe_set_profiling(lay.h, False)
    finally:
        lay.close()
    gemm_names = {"expert_tiles", "gather_latent", "expert_w13_gemm", "expert_w2_gemm"}
    gemv_names = {"expert_w13_gemv", "expert_w2_gemv"}
    assert gemm_names <= auto and not (gemv_names & auto)
    assert gemv_names <= gemv and not (gemm_names & gemv)
    assert gemv_names <= small and not (gemm_names & small)
    tiny = Layer(k3synth.TINY, [None], max_tokens=4)     # 16 pairs at most: no grouped GEMM
    try:
        with pytest.raises(km.K3MoEError) as ei:
            km.k3moe_set_expert_path(tiny.h, km.K3MOE_EXPERT_GEMM)
        assert ei.value.code == km.K3MOE_ERR_SHAPE
    finally:
        tiny.close()


def test_mid_shape_no_bias_no_renorm():
    shape = k3synth.replace(MID, renorm=0, routed_scale=0.5)
    run_case(shape, k3synth.replace(k3synth.TINY_RECIPE, zero_bias=True), 2, 9)


def test_bad_scale_rejected_and_layer_stays_unloaded():
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(k3synth.TINY, 0, 0, k3synth.TINY_RECIPE)
    d["w2s"] = d["w2s"].copy()
    d["w2s"][7, 3, 1] = 255
    lay = Layer(k3synth.TINY, [None], max_tokens=4)
    try:
        with pytest.raises(km.K3MoEError) as ei:
            lay.load(0, d)
        assert ei.value.code == km.K3MOE_ERR_BAD_SCALE
        with pytest.raises(km.K3MoEError) as ei:
            lay.forward(k3synth.make_tokens(k3synth.TINY, 0, 4))
        assert ei.value.code == km.K3MOE_ERR_NOT_LOADED
    finally:
        lay.close()


def test_forward_argument_errors():
    import torch
    import mxfp4_routed_expert_gb300 as km
    d = k3synth.make_layer(k3synth.TINY, 0, 0, k3synth.TINY_RECIPE)
    lay = Layer(k3synth.TINY, [d], max_tokens=4)
    try:
        x = torch.zeros((8, 256), dtype=torch.int16, device="cuda")
        y = torch.zeros_like(x)
        xo = x.data_ptr() + 2            # inside x, not on a 16-byte boundary
        for args, code in [((1, x, y, 4), km.K3MOE_ERR_INVALID_ARG),     # layer out of range
                           ((0, x, y, 5), km.K3MOE_ERR_INVALID_ARG),     # T > max_tokens
                           ((0, x, y, 0), km.K3MOE_ERR_INVALID_ARG),     # T = 0
                           ((0, x, x, 4), km.K3MOE_ERR_INVALID_ARG),     # x and y overlap
                           ((0, xo, y, 4), km.K3MOE_ERR_INVALID_ARG),    # x unaligned
                           ((0, x, y.data_ptr() + 8, 4), km.K3MOE_ERR_INVALID_ARG)]:  # y unaligned
            with pytest.raises(km.K3MoEError) as ei:
                km.k3moe_forward(lay.h, *args)
            assert ei.value.code == code
        assert km.k3moe_sync_status(lay.h) == 0
    finally:
        lay.close()


def test_device_wait_timeout_is_reported_and_the_handle_stays_usable():
    """A kernel whose one bounded wait can never be satisfied latches the
    time-out (after about two seconds) instead of hanging: k3moe_sync_status
    returns it once, then the same handle runs a forward that matches the
    oracle."""
    import time
    import mxfp4_routed_expert_gb300 as km
    shape = k3synth.TINY
    d = k3synth.make_layer(shape, 7, 0, k3synth.TINY_RECIPE)
    x, _ = guarded_tokens(shape, d, 7, 4)
    lay = Layer(shape, [d], max_tokens=4)
    try:
        assert km.k3moe_sync_status(lay.h) == 0
        t0 = time.monotonic()
        km.k3moe_check_wait_timeout(lay.h)
        assert km.k3moe_sync_status(lay.h) == km.K3MOE_ERR_TIMEOUT
        assert 1.5 < time.monotonic() - t0 < 60
        assert km.k3moe_sync_status(lay.h) == 0          # read once, then cleared
        y = lay.forward(x)
        assert km.k3moe_sync_status(lay.h) == 0
    finally:
        lay.close()
    assert_close(bf16_to_f64(y), oracle.layer_forward(shape, d, x))


def test_oversized_requests_refused_before_allocating(monkeypatch):
    """With the device-memory budget below what a request needs (its bytes
    plus the margin), create and load return K3MOE_ERR_OOM with nothing
    allocated: the handle stays as it was, the layer stays unloaded, and the
    same load goes through once the budget is lifted."""
    import mxfp4_routed_expert_gb300 as km
    shape = k3synth.TINY
    d = k3synth.make_layer(shape, 8, 0, k3synth.TINY_RECIPE)
    x, _ = guarded_tokens(shape, d, 8, 4)
    monkeypatch.setenv("K3MOE_DEVICE_BUDGET_MB", "1")       # below the workspace margin
    with pytest.raises(km.K3MoEError) as ei:
        Layer(shape, [None], max_tokens=4)
    assert ei.value.code == km.K3MOE_ERR_OOM
    monkeypatch.setenv("K3MOE_DEVICE_BUDGET_MB", "128")     # the workspace fits, a layer does not
    lay = Layer(shape, [None], max_tokens=4)
    try:
        with pytest.raises(km.K3MoEError) as ei:
            lay.load(0, d)
        assert ei.value.code == km.K3MOE_ERR_OOM
        with pytest.raises(km.K3MoEError) as ei:
            km.k3moe_set_expert_tier(lay.h, shape.n_experts)
        assert ei.value.code == km.K3MOE_ERR_OOM
        assert km.k3moe_get_tier_stats(lay.h)["slots"] == 0
        import torch
        xd = torch.zeros((4, shape.hidden), dtype=torch.int16, device="cuda")
        with pytest.raises(km.K3MoEError) as ei:
            km.k3moe_forward(lay.h, 0, xd, torch.zeros_like(xd), 4)
        assert ei.value.code == km.K3MOE_ERR_NOT_LOADED
        monkeypatch.delenv("K3MOE_DEVICE_BUDGET_MB")
        lay.load(0, d)
        y = lay.forward(x)
    finally:
        lay.close()
    assert_close(bf16_to_f64(y), oracle.layer_forward(shape, d, x))


def test_forward_host_matches_device_forward():
    import mxfp4_routed_expert_gb300 as km
    shape = k3synth.TINY
    d = k3synth.make_layer(shape, 3, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 3, 6)
    lay = Layer(shape, [d], max_tokens=6)
    try:
        y_dev = lay.forward(x)
        y_host = np.empty_like(x)
        km.k3moe_forward_host(lay.h, 0, x, y_host, 6)
    finally:
        lay.close()
    # the w2 scatter-add uses fp32 atomics, whose order varies between runs: an
    # output may differ by one bf16 unit in the last place, and an output that
    # cancels to near zero by more than one unit of its own, so the two runs
    # are compared on the output's scale (as the host-buffer tests below do)
    a, b = bf16_to_f64(y_host), bf16_to_f64(y_dev)
    assert np.max(np.abs(a - b)) <= np.max(np.abs(b)) * 2.0 ** -7


@pytest.mark.parametrize("shape_T", [("mid", 1), ("mid", 2), ("wide", 37)])
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_buffers(shape_T, pinned):
    """Host buffers at one or two tokens (decode GEMVs) and at 37 (tensor-core
    GEMMs): a pinned y is written in place by the layer's last kernel, a
    pageable one is copied back; both match the device forward."""
    import torch
    import mxfp4_routed_expert_gb300 as km
    name, T = shape_T
    shape = {"mid": MID, "wide": WIDE}[name]
    d = k3synth.make_layer(shape, 15, 0, k3synth.TINY_RECIPE)
    x, _ = guarded_tokens(shape, d, 15, T)
    lay = Layer(shape, [d], max_tokens=T)
    try:
        y_dev = lay.forward(x)
        if pinned:
            xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
            yh = torch.full((T, shape.hidden), -1, dtype=torch.int16).pin_memory()
            km.k3moe_forward_host(lay.h, 0, xh, yh, T)
            y_host = yh.numpy().view(np.uint16)
        else:
            y_host = np.empty_like(x)
            km.k3moe_forward_host(lay.h, 0, x, y_host, T)
        assert km.k3moe_sync_status(lay.h) == 0
    finally:
        lay.close()
    # the fp32 atomics of the expert scatter-add vary their order between runs:
    # the two outputs agree to a bf16 unit of the output's scale
    a, b = bf16_to_f64(y_host), bf16_to_f64(y_dev)
    assert np.max(np.abs(a - b)) <= np.max(np.abs(b)) * 2.0 ** -7
    assert_close(a, oracle.layer_forward(shape, d, x), f"host buffers T={T}")


def test_routing_is_deterministic_and_profiling_lists_kernels():
    import mxfp4_routed_expert_gb300 as km
    shape = MID
    d = k3synth.make_layer(shape, 4, 0, k3synth.TINY_RECIPE)
    x = k3synth.make_tokens(shape, 4, 20)
    lay = Layer(shape, [d], max_tokens=20)
    try:
        km.k3moe_set_profiling(lay.h, True)
        lay.forward(x)
        a = lay.routing(20)
        lay.forward(x)
        b = lay.routing(20)
        stats = km.k3moe_profile_read(lay.h)
        km.k3moe_set_profiling(lay.h, False)
    finally:
        lay.close()
    for k in ("ids", "counts", "offsets", "perm"):
        np.testing.assert_array_equal(a[k], b[k])
    names = {s[0] for s in stats}
    # T=20 (160 pairs): dense GEMVs (64 experts < 128 rows), grouped expert GEMM
    assert {"router_down_gemv", "shared_gate_up_gemv", "route_topk", "perm_count", "perm_scan",
            "perm_place", "expert_tiles",
            "gather_latent", "expert_w13_gemm", "expert_w2_gemm", "norm_up_shared_gemv"} <= names
    assert all(s[1] == 2 and s[2] > 0 for s in stats)


def test_chain_two_layers_tiny():
    shape = k3synth.TINY
    d0 = k3synth.make_layer(shape, 5, 0, k3synth.TINY_RECIPE)
    d1 = k3synth.make_layer(shape, 5, 1, k3synth.TINY_RECIPE)
    x, _ = guarded_tokens(shape, d0, 5, 8)
    lay = Layer(shape, [d0, d1], max_tokens=8)
    try:
        y = lay.forward(x, layer=0, chain=2)
        y0 = lay.forward(x, layer=0)
    finally:
        lay.close()
    ref0 = oracle.layer_forward(shape, d0, x)
    assert_close(bf16_to_f64(y0), ref0, "layer 0")
    # layer 1 is checked against the oracle given the GPU's own layer-1 input
    x1 = k3synth.round_bf16(oracle.chain_glue(bf16_to_f64(y0), shape.rms_eps))
    _, _, margin = oracle.route(shape, d1, x1)
    ref1 = oracle.layer_forward(shape, d1, x1)
    ok = margin > 1e-5          # tokens whose layer-1 routing is not a near-tie
    assert ok.sum() >= 6
    assert_close(bf16_to_f64(y)[ok], ref1[ok], "layer 1 of the chain")


# ---------------------------------------------------------------------------
# K3-shape layer (about 16 GB on the device)

@pytest.fixture(scope="module")
def k3layer():
    d = k3synth.make_layer(k3synth.K3, 0, 0, k3synth.K3_RECIPE)
    lay = Layer(k3synth.K3, [d], max_tokens=4096)
    yield d, lay
    lay.close()


def test_k3_decode_T1(k3layer):
    d, lay = k3layer
    shape = k3synth.K3
    pool, _ = guarded_tokens(shape, d, 0, 64, stream=7)
    for t in (0, 13, 63):
        x = pool[t:t + 1]
        y = lay.forward(x)
        r = lay.routing(1)
        ref, tr = oracle.layer_forward(shape, d, x, trace=True)
        check_routing(r, shape, x, tr["ids"], tr["w"])
        assert_close(bf16_to_f64(y), ref, f"K3 T=1 token {t}")


def test_k3_decode_T1_block_scaled(k3layer):
    """K3 T=1 on the block-scaled grouped GEMM with split K ranges (16 pairs,
    W1/W3 in 4 parts and W2 in 6 per item)."""
    import mxfp4_routed_expert_gb300 as km
    d, lay = k3layer
    shape = k3synth.K3
    pool, _ = guarded_tokens(shape, d, 0, 64, stream=7)
    try:
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_MX)
        for t in (0, 13, 63):
            x = pool[t:t + 1]
            y = lay.forward(x)
            r = lay.routing(1)
            acc = lay.intermediate(km.K3MOE_T_ACC, 1, shape.latent)
            ref, tr = oracle.layer_forward(shape, d, x, trace=True)
            check_routing(r, shape, x, tr["ids"], tr["w"])
            assert_close(acc, tr["acc"], f"K3 T=1 token {t} latent aggregate")
            assert_close(bf16_to_f64(y), ref, f"K3 T=1 token {t}")
    finally:
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_AUTO)


@pytest.mark.parametrize("T", [2, 5, 8, 16])
def test_k3_decode_batches(k3layer, T):
    """K3 width at the batch sizes between one token and T=64: T=2 runs the
    TMA-fed dense GEMVs, 3 <= T <= 15 the register GEMVs, T=16 the smallest
    tensor-core batch (split-K dense GEMMs; 256 pairs, so the automatic expert
    path is the grouped GEMM, and the per-pair GEMVs are checked on the same
    tokens)."""
    import mxfp4_routed_expert_gb300 as km
    d, lay = k3layer
    shape = k3synth.K3
    x, _ = guarded_tokens(shape, d, 0, T, stream=20 + T)
    ref, tr = oracle.layer_forward(shape, d, x, trace=True)
    # the block-scaled grouped GEMM at every batch (K ranges split below 128 pairs)
    modes = ((km.K3MOE_EXPERT_AUTO, km.K3MOE_EXPERT_GEMV, km.K3MOE_EXPERT_MX) if T >= 16
             else (km.K3MOE_EXPERT_AUTO, km.K3MOE_EXPERT_MX))
    try:
        for mode in modes:
            km.k3moe_set_expert_path(lay.h, mode)
            y = lay.forward(x)
            r = lay.routing(T)
            check_routing(r, shape, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref, f"K3 T={T}, expert path {mode}")
    finally:
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_AUTO)


def test_k3_residual_T1(k3layer):
    """The RMSNorm in front of the MoE fused into the decode kernels at K3 size
    (hidden 7168: 14 float4 per consumer thread per token)."""
    import mxfp4_routed_expert_gb300 as km
    d, lay = k3layer
    shape = k3synth.K3
    g = k3synth.post_norm_gain(shape, 1)
    make = lambda att: oracle.round_bf16(   # noqa: E731
        oracle.residual_input(k3synth.make_residual(shape, 1, 1, 0, att), g, shape.rms_eps))
    _, att = guarded_tokens(shape, d, 1, 1, make=make)
    hres = k3synth.make_residual(shape, 1, 1, 0, att)
    km.k3moe_load_post_norm(lay.h, 0, g)
    y = lay.forward_residual(hres)
    x_gpu = lay.layer_input(1)
    r = lay.routing(1)
    v = oracle.residual_input(hres, g, shape.rms_eps)
    step = np.ldexp(1.0, np.frexp(np.abs(v))[1] - 8)
    assert np.all(np.abs(bf16_to_f64(x_gpu) - v) <= step)
    ref, tr = oracle.layer_forward(shape, d, x_gpu, trace=True)
    check_routing(r, shape, x_gpu, tr["ids"], tr["w"])
    assert_close(bf16_to_f64(y), ref, "K3 T=1 from the residual")


def test_k3_tier_T1(k3layer):
    """The expert tier at K3 size: the layer's 15.7 GB of experts in pinned host
    memory, 896 device slots. The first forward of a token copies its 16
    experts in, the second finds them resident; both match the oracle."""
    import mxfp4_routed_expert_gb300 as km
    d, _ = k3layer
    shape = k3synth.K3
    pool, _ = guarded_tokens(shape, d, 0, 64, stream=7)
    x = pool[5:6]
    ref, tr = oracle.layer_forward(shape, d, x, trace=True)
    tl = Layer(shape, [d], max_tokens=1, tier_slots=shape.n_experts)
    try:
        for want in ((0, 16), (16, 16)):
            y = tl.forward(x)
            r = tl.routing(1)
            check_routing(r, shape, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref, "K3 T=1 through the tier")
            st = km.k3moe_get_tier_stats(tl.h)
            assert (st["hits"], st["misses"]) == want
    finally:
        tl.close()


def test_k3_T64_covering(k3layer):
    """Every expert touched, on the grouped GEMM (auto) and its block-scaled form."""
    import mxfp4_routed_expert_gb300 as km
    d, lay = k3layer
    shape = k3synth.K3
    d0 = k3synth.with_bias(d, np.zeros(shape.n_experts, np.float32))
    lay.load(0, d0)
    try:
        x, _ = guarded_tokens(shape, d0, 0, 64,
                              make=lambda att: k3synth.covering_tokens(shape, d0, 0, 64,
                                                                       attempts=att))
        ref, tr = oracle.layer_forward(shape, d0, x, trace=True)
        for mode in (km.K3MOE_EXPERT_AUTO, km.K3MOE_EXPERT_MX):
            km.k3moe_set_expert_path(lay.h, mode)
            y = lay.forward(x)
            r = lay.routing(64)
            assert (r["counts"] > 0).sum() == shape.n_experts       # every expert touched
            check_routing(r, shape, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref, f"K3 T=64 covering, expert path {mode}")
    finally:
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_AUTO)
        lay.load(0, d)


def test_k3_T64_random(k3layer):
    """Both routed-expert paths (auto picks the grouped GEMM at T=64)."""
    import mxfp4_routed_expert_gb300 as km
    d, lay = k3layer
    shape = k3synth.K3
    x, _ = guarded_tokens(shape, d, 0, 64, stream=9)
    ref, tr = oracle.layer_forward(shape, d, x, trace=True)
    try:
        for mode in (km.K3MOE_EXPERT_AUTO, km.K3MOE_EXPERT_GEMV, km.K3MOE_EXPERT_MX):
            km.k3moe_set_expert_path(lay.h, mode)
            y = lay.forward(x)
            r = lay.routing(64)
            check_routing(r, shape, x, tr["ids"], tr["w"])
            assert_close(bf16_to_f64(y), ref, f"K3 T=64 random, expert path {mode}")
    finally:
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_AUTO)


def test_k3_T4096_zipf_prefill(k3layer):
    """Prefill: 4096 tokens, Zipf(1.1) expert popularity through the router
    bias. Ids and the permutation are checked on every token; y against the
    oracle on every 16th token, on every token of the 4 least-picked experts
    (ragged n-tiles) and on 32 tokens of each of the 4 most-picked ones (many
    n-tiles). Both grouped GEMMs: the f16 one (auto) and the block-scaled one."""
    import mxfp4_routed_expert_gb300 as km
    d, lay = k3layer
    shape = k3synth.K3
    dz = k3synth.with_bias(d, k3synth.zipf_bias(shape, 0, 0, k3synth.K3_ZIPF_ALPHA))
    lay.load(0, dz)
    try:
        T = 4096
        x, _ = guarded_tokens(shape, dz, 0, T, stream=11)
        y = lay.forward(x)
        r = lay.routing(T)
        ids, w, _ = oracle.route(shape, dz, x)
        check_routing(r, shape, x, ids, w)
        counts = np.bincount(ids.ravel(), minlength=shape.n_experts)
        used = np.flatnonzero(counts)
        cold = used[np.argsort(counts[used], kind="stable")[:4]]
        hot = np.argsort(-counts, kind="stable")[:4]
        rows = set(range(0, T, 16))
        for e in cold:
            rows.update(np.flatnonzero((ids == e).any(1)).tolist())
        for e in hot:
            rows.update(np.flatnonzero((ids == e).any(1))[:32].tolist())
        rows = np.array(sorted(rows), dtype=np.int32)
        ref = oracle.layer_forward(shape, dz, x, rows=rows)
        assert_close(bf16_to_f64(y)[rows], ref, f"K3 T=4096 Zipf ({rows.size} sampled rows)")
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_MX)
        y = lay.forward(x)
        check_routing(lay.routing(T), shape, x, ids, w)
        assert_close(bf16_to_f64(y)[rows], ref, f"K3 T=4096 Zipf, block-scaled ({rows.size} sampled rows)")
    finally:
        km.k3moe_set_expert_path(lay.h, km.K3MOE_EXPERT_AUTO)
        lay.load(0, d)


def test_k3_chain_two_layers_T256():
    """Two stacked K3-shape layers at T=256 (the chain workload's batch): layer 0
    against the oracle, layer 1 against the oracle given the GPU's own layer-1
    input (RMSNorm of layer 0's output), both on 32 sampled tokens."""
    shape = k3synth.K3
    d0 = k3synth.make_layer(shape, 3, 0, k3synth.K3_RECIPE)
    d1 = k3synth.make_layer(shape, 3, 1, k3synth.K3_RECIPE)
    T = 256
    x, _ = guarded_tokens(shape, d0, 3, T, stream=13)
    lay = Layer(shape, [d0, d1], max_tokens=T)
    try:
        y = lay.forward(x, layer=0, chain=2)
        y0 = lay.forward(x, layer=0)
    finally:
        lay.close()
    rows = np.arange(0, T, 8, dtype=np.int32)
    assert_close(bf16_to_f64(y0)[rows], oracle.layer_forward(shape, d0, x, rows=rows), "K3 chain layer 0")
    x1 = k3synth.round_bf16(oracle.chain_glue(bf16_to_f64(y0), shape.rms_eps))
    _, _, margin = oracle.route(shape, d1, x1)
    ok = np.flatnonzero(margin > 1e-5)
    sel = ok[:: max(1, ok.size // 32)][:32].astype(np.int32)
    assert sel.size >= 24
    ref1 = oracle.layer_forward(shape, d1, x1, rows=sel)
    assert_close(bf16_to_f64(y)[sel], ref1, "K3 chain layer 1")
