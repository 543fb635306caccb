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



def test_trace_files_and_command_line(tmp_path, capsys):
    """A trace saved as JSON lines or recorded as per-forward counts in an
    .npz reads back unchanged, and the command line prints the replay of
    both policies per slot count (pins included)."""
    import json
    from mxfp4_routed_expert_gb300 import tier_trace as tt
    tr = [(l, tuple(sorted(ex))) for l, ex in random_trace(7, n_fwd=30, layers=2, E=24, per=5)]
    p = tmp_path / "t.jsonl"
    tt.save_trace(str(p), tr)
    assert tt.load_trace(str(p)) == tr
    counts = np.zeros((len(tr), 24), np.int32)
    for i, (_, ex) in enumerate(tr):
        counts[i, list(ex)] = 3
    q = tmp_path / "t.npz"
    np.savez(q, layers=np.array([l for l, _ in tr]), counts=counts)
    assert tt.load_trace(str(q)) == tr
    q2 = tmp_path / "trace.bin"                    # any name: the reader looks at the bytes
    tt.save_counts(str(q2), [l for l, _ in tr], counts)
    assert tt.load_trace(str(q2)) == tr
    with pytest.raises(ValueError):
        tt.save_counts(str(q2), [0, 1], counts)
    assert tt.main([str(p), "--slots", "8,24", "--expert-bytes", "10", "--json"]) == 0
    rows = [json.loads(line) for line in capsys.readouterr().out.splitlines()]
    assert [(r["slots"], r["policy"]) for r in rows] == [(8, "tier"), (8, "belady"), (24, "tier"),
                                                         (24, "belady")]
    for r in rows:
        ref = replay(tr, r["slots"], r["policy"], expert_bytes=10)
        assert (r["hits"], r["misses"], r["bytes_copied"]) == (ref["hits"], ref["misses"],
                                                               ref["bytes_copied"])
    # pinning layer 0 (all of its experts seen in the trace) on 48 slots: its
    # forwards never miss, so every miss is one of layer 1's
    assert tt.main([str(p), "--slots", "48", "--pin", "0", "--json"]) == 0
    r = json.loads(capsys.readouterr().out.splitlines()[0])
    seen0 = {e for l, ex in tr if l == 0 for e in ex}
    assert r["pin_copies"] == len(seen0)
    assert r["misses"] == len({e for l, ex in tr if l == 1 for e in ex})
    # too few slots for one forward: reported on its row, not raised
    assert tt.main([str(p), "--slots", "3"]) == 0
    assert "more experts than there are slots" in capsys.readouterr().out
    bad = tmp_path / "bad.jsonl"
    bad.write_text('{"layer": 0}\n')
    with pytest.raises(ValueError):
        tt.load_trace(str(bad))


def brute_force_min_misses(trace, slots):
    """The fewest misses any eviction choice reaches: every forward's experts
    must be resident together; on a miss with the slots full, any resident
    expert not used by this forward may go (all subsets tried)."""
    from functools import lru_cache
    from itertools import combinations
    tr = [frozenset((l, e) for e in ex) for l, ex in trace]

    @lru_cache(maxsize=None)
    def best(i, resident):
        if i == len(tr):
            return 0
        need = tr[i]
        miss = need - resident
        over = len(resident) + len(miss) - slots
        if over <= 0:
            return len(miss) + best(i + 1, resident | need)
        out = None
        for gone in combinations(sorted(resident - need), over):
            v = best(i + 1, (resident - frozenset(gone)) | need)
            out = v if out is None else min(out, v)
        return len(miss) + out

    return best(0, frozenset())


@pytest.mark.parametrize("seed", range(12))
def test_belady_is_the_optimum_on_small_traces(seed):
    """On traces small enough to search exhaustively, the offline policy's
    misses equal the fewest any policy can reach, and the tier's are never
    fewer."""
    r = random.Random(100 + seed)
    E, layers, per, slots = 5, 2, r.choice([1, 2, 3]), r.choice([3, 4, 5])
    tr = [(r.randrange(layers), r.sample(range(E), per)) for _ in range(9)]
    opt = brute_force_min_misses(tr, slots)
    assert replay(tr, slots, "belady")["misses"] == opt
    assert replay(tr, slots, "tier")["misses"] >= opt
