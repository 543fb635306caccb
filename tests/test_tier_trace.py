"""The host-side replay of a routing trace for sizing the expert tier
(kimi-k3-in-c README, Part II section 13): the tier's own policy and the
offline optimum (Belady), checked on CPU against facts that hold for any
correct replay."""
import random

import numpy as np
import pytest

from mxfp4_routed_expert_gb300.tier_trace import replay, trace_from_counts


def random_trace(seed, n_fwd=60, layers=3, E=40, per=6):
    r = random.Random(seed)
    return [(r.randrange(layers), r.sample(range(E), per)) for _ in range(n_fwd)]


def test_trace_from_counts():
    assert trace_from_counts(2, np.array([0, 3, 0, 1, 0])) == (2, (1, 3))


def test_by_hand_tier_policy():
    # 4 slots: forward 1 puts (0,1), (0,2) in slots 0, 1; forward 2 takes the
    # never-used 2, 3 and the oldest slot 0 (evicting (0,1)); forward 3 hits
    # (0,2) in slot 1 and puts (0,1) back into slot 0, the oldest left
    tr = [(0, [1, 2]), (1, [1, 2, 3]), (0, [1, 2])]
    st = replay(tr, 4, "tier", expert_bytes=10)
    assert (st["hits"], st["misses"], st["compulsory"], st["bytes_copied"]) == (1, 6, 5, 60)


@pytest.mark.parametrize("policy", ["tier", "belady"])
def test_room_for_everything_misses_only_once(policy):
    tr = random_trace(1)
    distinct = len({(l, e) for l, ex in tr for e in ex})
    st = replay(tr, distinct + 3, policy)
    assert st["misses"] == st["compulsory"] == distinct


@pytest.mark.parametrize("seed", range(8))
def test_belady_is_a_ceiling(seed):
    tr = random_trace(seed)
    for slots in (6, 10, 25, 60):
        assert replay(tr, slots, "belady")["hits"] >= replay(tr, slots, "tier")["hits"]


def test_cyclic_scan_defeats_lru_but_not_the_optimum():
    # four layers, the same 8 experts each, visited in a cycle: 32 keys, 16 slots
    tr = [(l, range(8)) for _ in range(10) for l in range(4)]
    assert replay(tr, 16, "tier")["hits"] == 0
    assert replay(tr, 16, "belady")["hits"] > 0


def test_a_forward_must_fit():
    with pytest.raises(ValueError):
        replay([(0, range(9))], 8)


def test_pinned_layer_never_misses_and_survives_the_scan():
    # the cyclic scan again, with layer 0 pinned: its requests all hit
    tr = [(l, range(8)) for _ in range(10) for l in range(4)]
    st = replay(tr, 24, "tier", pin=[(0, range(8))])
    assert st["pin_copies"] == 8
    assert st["hits"] >= 10 * 8          # every visit of layer 0
    plain = replay(tr, 24, "tier")
    assert st["hits"] > plain["hits"]


def test_pins_must_leave_room():
    with pytest.raises(ValueError):
        replay([(1, range(8))], 12, "tier", pin=[(0, range(8))])

