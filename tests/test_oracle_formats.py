"""Pins for the oracle's MXFP4 / bf16 decoding (CPU only).

What is pinned, and by what (kimi-k3-in-c README, Part II section 4; colibri
docs/kimi_k3.md "Weights"):
  - the E2M1 table printed on the page (golden file);
  - hand-packed bytes with known decoded pairs (low nibble = even column);
  - the ue8m0 rule (127 is the identity, +1 doubles, 255 zeroes the group);
  - a swapped-nibble fixture whose statistics match but whose positions differ;
  - one-hot rows recover each decoded weight exactly;
  - the byte census of one expert printed on the page;
  - bf16 widening against torch's own bfloat16 -> float32 conversion.
"""
import json
import math
import os

import numpy as np
import pytest

import k3synth
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_e2m1_table_matches_page():
    lut = _gold("mxfp4_format.json")["e2m1_lut"]
    for n in range(16):
        v = oracle.e2m1(n)
        assert v == lut[n]
        # bit 3 is the sign, including the negative zero at nibble 8
        assert math.copysign(1.0, v) == (-1.0 if n & 8 else 1.0)


def test_group_size_matches_page():
    assert oracle.group_size() == _gold("mxfp4_format.json")["group_size"]


def test_e8m0_rule():
    assert oracle.e8m0(127) == 1.0
    assert oracle.e8m0(128) == 2.0
    assert oracle.e8m0(126) == 0.5
    assert oracle.e8m0(0) == math.ldexp(1.0, -127)
    assert oracle.e8m0(254) == math.ldexp(1.0, 127)
    assert oracle.e8m0(255) == 0.0
    for b in range(255):
        assert oracle.e8m0(b) == math.ldexp(1.0, b - 127)


@pytest.mark.parametrize("byte,pair", [(0x21, (0.5, 1.0)), (0x8F, (-6.0, -0.0)),
                                       (0x70, (0.0, 6.0)), (0xF7, (6.0, -6.0)),
                                       (0x3C, (-2.0, 1.5))])
def test_hand_packed_bytes(byte, pair):
    row = np.array([byte] + [0] * 15, np.uint8)
    sc = np.array([127], np.uint8)
    even, odd = oracle.mxfp4_weight(row, sc, 0), oracle.mxfp4_weight(row, sc, 1)
    assert (even, odd) == pair
    assert math.copysign(1.0, even) == math.copysign(1.0, pair[0])
    assert math.copysign(1.0, odd) == math.copysign(1.0, pair[1])
    # scale 128 doubles, 126 halves, both exactly
    assert oracle.mxfp4_weight(row, np.array([128], np.uint8), 0) == 2 * pair[0]
    assert oracle.mxfp4_weight(row, np.array([126], np.uint8), 1) == 0.5 * pair[1]


def test_swapped_nibble_fixture():
    """Same multiset of weights, different positions: only the correct nibble
    order reproduces the dot products (the README's swapped-nibble warning)."""
    packed = np.array([[0x71, 0x2A, 0x06, 0xD3] + [0] * 12], np.uint8)  # 32 columns
    sc = np.array([[127]], np.uint8)
    lut = _gold("mxfp4_format.json")["e2m1_lut"]
    right = np.zeros(32)
    swapped = np.zeros(32)
    for i, b in enumerate(packed[0]):
        right[2 * i], right[2 * i + 1] = lut[b & 15], lut[b >> 4]
        swapped[2 * i], swapped[2 * i + 1] = lut[b >> 4], lut[b & 15]
    assert sorted(right) == sorted(swapped)          # identical statistics
    x = np.arange(1, 33, dtype=np.float64)           # position-sensitive probe
    y = oracle.mxfp4_matvec(x, packed, sc, 32)
    assert y[0] == pytest.approx(float(right @ x), abs=0)
    assert y[0] != float(swapped @ x)


def _numpy_decode(packed, scales, n_in):
    """Independent vectorised decode of the documented layout (table lookup per
    nibble, low nibble -> even column, one power-of-two scale per 32 columns)."""
    lut = np.array(_gold("mxfp4_format.json")["e2m1_lut"])
    rows = packed.shape[0]
    vals = np.empty((rows, packed.shape[1] * 2))
    vals[:, 0::2] = lut[packed & 15]
    vals[:, 1::2] = lut[packed >> 4]
    vals = vals[:, :n_in]
    s = np.where(scales == 255, 0.0, np.ldexp(1.0, scales.astype(np.int64) - 127))
    return vals * np.repeat(s, 32, axis=1)[:, :n_in]


def test_one_hot_rows_recover_weights():
    rows, n_in = 8, 96
    packed = k3synth.uniform_bytes((rows, n_in // 2), k3synth.key(7, 1))
    scales = k3synth.uniform_u8((rows, n_in // 32), k3synth.key(7, 2), 110, 140)
    dense = _numpy_decode(packed, scales, n_in)
    for c in range(n_in):
        x = np.zeros(n_in)
        x[c] = 1.0
        y = oracle.mxfp4_matvec(x, packed, scales, n_in)
        np.testing.assert_array_equal(y, dense[:, c])
        for r in range(rows):
            assert oracle.mxfp4_weight(packed[r], scales[r], c) == dense[r, c]


def test_matvec_equals_dense_decode():
    rows, n_in = 16, 3584
    packed = k3synth.uniform_bytes((rows, n_in // 2), k3synth.key(8, 1))
    scales = k3synth.uniform_u8((rows, n_in // 32), k3synth.key(8, 2), 117, 123)
    x = k3synth.normal_f64((n_in,), k3synth.key(8, 3))
    y = oracle.mxfp4_matvec(x, packed, scales, n_in)
    ref = _numpy_decode(packed, scales, n_in) @ x
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_scale_255_zeroes_only_its_group():
    rows, n_in = 4, 128
    packed = k3synth.uniform_bytes((rows, n_in // 2), k3synth.key(9, 1))
    scales = np.full((rows, 4), 127, np.uint8)
    x = k3synth.normal_f64((n_in,), k3synth.key(9, 2))
    full = oracle.mxfp4_matvec(x, packed, scales, n_in)
    scales2 = scales.copy()
    scales2[:, 2] = 255
    cut = oracle.mxfp4_matvec(x, packed, scales2, n_in)
    xg = x.copy()
    xg[64:96] = 0.0
    np.testing.assert_allclose(cut, oracle.mxfp4_matvec(xg, packed, scales, n_in), rtol=0, atol=1e-15)
    assert not np.allclose(cut, full)


def test_scale_zero_is_two_to_minus_127():
    packed = np.array([[0x22] * 16], np.uint8)   # 1.0 everywhere
    x = np.ones(32)
    y = oracle.mxfp4_matvec(x, packed, np.array([[0]], np.uint8), 32)
    assert y[0] == 32 * math.ldexp(1.0, -127)


def test_odd_length_tail():
    """A short last group (35 columns) is handled, the last column being the
    low nibble of the last byte (the README writes this case although the
    checkpoint never hits it)."""
    n_in = 35
    packed = np.zeros((1, 18), np.uint8)
    packed[0, 17] = 0x57                               # column 34 = low nibble 7 -> 6.0
    scales = np.array([[127, 129]], np.uint8)          # column 34 is in group 1
    x = np.zeros(n_in)
    x[34] = 1.0
    assert oracle.mxfp4_matvec(x, packed, scales, n_in)[0] == 6.0 * 4
    assert oracle.mxfp4_weight(packed[0], scales[0], 34) == 24.0


def test_expert_census_matches_page():
    g = _gold("mxfp4_format.json")
    K3 = k3synth.K3
    params = 3 * K3.latent * K3.moe_inter
    assert params == g["params_per_expert"]
    assert K3.expert_bytes == g["bytes_per_expert"]
    assert K3.expert_bytes == params * g["bytes_per_weight"]
    ex = g["example_tensor"]
    assert ex["packed_cols"] == K3.latent // 2 and ex["scale_cols"] == K3.latent // 32
    assert ex["logical_width"] == K3.latent


def test_bf16_widening_matches_torch():
    torch = pytest.importorskip("torch")
    bits = k3synth.uniform_bytes((4096,), k3synth.key(10, 1)).view(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]            # finite values
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16(int(b)) for b in bits])
    np.testing.assert_array_equal(got, ref.astype(np.float64))


def test_bf16_matvec_equals_library_matmul():
    W = k3synth.normal_bf16((64, 300), k3synth.key(11, 1), 0.0, 0.02)
    x = k3synth.normal_f64((300,), k3synth.key(11, 2))
    Wf = k3synth.bf16_bits_to_f32(W).astype(np.float64)
    np.testing.assert_allclose(oracle.bf16_matvec(x, W), Wf @ x, rtol=1e-13, atol=1e-15)
