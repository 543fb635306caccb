"""Host-side figures of bench.py (CPU only): the algorithmic bytes behind the
roofline fractions, checked against the byte census of the expert format
printed on the pages (tests/golden/mxfp4_format.json: 17,547,264 bytes per
expert, kimi-k3-in-c README Part II section 4) and the K3 layer's shapes."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import k3synth  # noqa: E402

K3 = k3synth.K3


def census():
    with open(os.path.join(ROOT, "tests", "golden", "mxfp4_format.json")) as f:
        return json.load(f)["bytes_per_expert"]


def test_k3_shape_is_the_pages_layer():
    assert (K3.hidden, K3.latent, K3.n_experts, K3.topk, K3.moe_inter, K3.shared_inter) == \
        (7168, 3584, 896, 16, 3072, 6144)


def test_layer_bytes_at_decode():
    # bf16 router [E, H], down [L, H], up [H, L], two shared experts fused:
    # gate and up [S, H] each, down [H, S]
    dense = 2 * (896 * 7168 + 3584 * 7168 + 7168 * 3584 + 3 * 6144 * 7168)
    assert dense == 379_846_656
    assert bench.layer_bytes(K3, 1, 16) == dense + 16 * census() + 2 * 2 * 7168
    assert bench.layer_bytes(K3, 64, 896) == dense + 896 * census() + 64 * 4 * 7168
    # the dense feed-forward layer reads its three matrices
    D = k3synth.K3_DENSE
    assert bench.layer_bytes(D, 1, 0) == 2 * 3 * D.shared_inter * D.hidden + 4 * D.hidden


def test_expert_kernels_read_the_census_per_touched_expert():
    """The W1/W3 and W2 kernels of one forward read, between them, every
    touched expert's packed nibbles and scales once (the census figure), plus
    activations that do not depend on the number of experts touched."""
    for T, touched in ((1, 16), (64, 896), (4096, 896)):
        for path in ("gemv", "gemm"):
            a = bench.kernel_model(K3, T, touched)
            b = bench.kernel_model(K3, T, touched - 1)
            d13 = a[f"expert_w13_{path}"][0] - b[f"expert_w13_{path}"][0]
            d2 = a[f"expert_w2_{path}"][0] - b[f"expert_w2_{path}"][0]
            assert d13 + d2 == census()
            assert d13 == 2 * census() // 3   # W1 and W3 are two of the three equal matrices


def test_flops_per_token():
    """1.437 GFLOP per token at K3: 16 pairs of three [3072 x 3584] expert
    matmuls plus the bf16 projections, 2 flops per multiply-add."""
    m = bench.kernel_model(K3, 1, 16)
    routed = m["expert_w13_gemm"][1] + m["expert_w2_gemm"][1]
    dense = m["router_down_gemm"][1] + m["shared_gate_up_gemm"][1] + m["up_shared_gemm"][1]
    assert routed == 16 * 3 * 2 * 3072 * 3584
    assert dense == 379_846_656   # 2 flops per bf16 weight (2 bytes) read once
    assert abs((routed + dense) / 1e9 - 1.437) < 5e-4
