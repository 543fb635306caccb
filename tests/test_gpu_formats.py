"""MXFP4 scale-byte edge cases through the C ABI, on every routed-expert path.

The format (kimi-k3-in-c README, Part II section 4) gives a weight the value
v * 2^(s - 127) for its group's ue8m0 byte s: byte 0 is 2^-127 (a subnormal
in fp32), 127 the identity, 254 is 2^127; 255 is refused at load. The layer
here (the 128-expert WIDE shape) forces four experts into every token's
selection, each carrying one kind of edge:

  - every row of W1, W3 and W2 at scale byte 0 (an expert whose output is
    about 2^-127 of a normal one);
  - groups cycling through bytes 1, 127, 120 and 0 in W1/W3 (127: weights up
    to 6, so the gate saturates SiTU) and 118, 1, 0, 120 in W2;
  - the first group of every row at byte 254 over all-zero nibbles (+0 and -0),
    the others at normal bytes: the group adds exactly zero, and must neither
    overflow nor push the row's real groups out of range;
  - rows whose groups alternate between bytes 124 and 94, thirty binades
    apart.

Bytes 0 and 1 put a group 2^-127 / 2^-126 below the identity, far under what
a layer output can show next to normal groups, so their part of the check is
that they decode to finite values and leave the other groups exact. Ids and
the permutation must match the oracle exactly, y and the latent aggregate
within the layer's tolerances, on the per-pair GEMVs, the f16 grouped GEMM
and the block-scaled grouped GEMM alike.
"""
import numpy as np
import pytest

import k3synth
from test_gpu_parity import WIDE, _mode, run_case

SPECIAL = (3, 40, 77, 120)


@pytest.fixture(scope="module")
def built():
    from mxfp4_routed_expert_gb300 import build
    build.build()


def _cycle(shape, pattern):
    """A scale array [E, rows, G] whose groups cycle through `pattern`."""
    return np.resize(np.asarray(pattern, np.uint8), shape)


def edge_layer(seed):
    d = dict(k3synth.make_layer(WIDE, seed, 0, k3synth.TINY_RECIPE))
    for k in ("w1p", "w1s", "w3p", "w3s", "w2p", "w2s"):
        d[k] = d[k].copy()
    e0, e1, e2, e3 = SPECIAL
    # every row at byte 0
    for k in ("w1s", "w3s", "w2s"):
        d[k][e0] = 0
    # cycling small, identity and zero bytes
    d["w1s"][e1] = _cycle(d["w1s"][e1].shape, [1, 127, 120, 0])
    d["w3s"][e1] = _cycle(d["w3s"][e1].shape, [1, 127, 120, 0])
    d["w2s"][e1] = _cycle(d["w2s"][e1].shape, [118, 1, 0, 120])
    # byte 254 on a group of zero nibbles at the start of every row
    for p, sk in (("w1p", "w1s"), ("w3p", "w3s"), ("w2p", "w2s")):
        d[sk][e2][:, 0] = 254
        d[p][e2][:, :16] &= 0x88          # keep the signs: +0 and -0
    # thirty binades between neighbouring groups
    for k in ("w1s", "w3s", "w2s"):
        d[k][e3] = _cycle(d[k][e3].shape, [124, 94])
    bias = np.asarray(d["router_bias"], np.float32).copy()
    bias[list(SPECIAL)] += 10.0
    return k3synth.with_bias(d, bias)


@pytest.mark.gpu
@pytest.mark.parametrize("path,T", [("gemv", 48), ("gemm", 48), ("mx", 48), ("mx", 8)])
def test_scale_edges_every_path(built, path, T):
    """T = 8 (64 pairs) runs the block-scaled kernel with split K ranges."""
    d = edge_layer(21)
    run_case(WIDE, k3synth.TINY_RECIPE, 21, T, expert_path=_mode(path), d=d)


def test_edge_layer_has_the_edges():
    """The fixture carries what the docstring says (CPU check of the bytes)."""
    d = edge_layer(21)
    e0, e1, e2, e3 = SPECIAL
    assert not d["w1s"][e0].any() and not d["w2s"][e0].any()
    assert set(np.unique(d["w1s"][e1])) == {0, 1, 120, 127}
    assert (d["w2s"][e2][:, 0] == 254).all() and not (d["w2p"][e2][:, :16] & 0x77).any()
    assert set(np.unique(d["w3s"][e3])) == {94, 124}
