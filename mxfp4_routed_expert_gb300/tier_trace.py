"""Sizing the expert tier from a recorded routing trace (host-side utility).

Routing does not depend on the cache, so one run can record every forward's
(layer, touched experts) and the trace can be replayed at any number of slots
(kimi-k3-in-c README, Part II section 13, "How big should that cache be? Ask
the trace"). This module replays such a trace under

- "tier":   the policy of `k3moe_set_expert_tier`: per forward, the touched
            experts already resident are hits; the others take, in ascending
            expert order, the slots not used by this forward with the oldest
            last use (never-used slots first; equal ages: the lower slot);
- "belady": the offline optimum at forward granularity: a miss evicts the
            resident expert, not used by this forward, whose next use lies
            furthest ahead (a ceiling for any policy, not a policy).

A trace is a list of (layer, experts) pairs in forward order; it can be built
from each forward's expert counts (`k3moe_get_routing`) with
`trace_from_counts`, and stored with `save_trace` as JSON lines (one
`[layer, [experts...]]` per forward) or, with `save_counts`, as an .npz
archive of `layers` [n] and `counts` [n, E] (`bench.py --dump-trace`).

Command line (the pages' "ask the trace" for a slot count):

    python -m mxfp4_routed_expert_gb300.tier_trace TRACE --slots 896,1792,2688
        [--expert-bytes 17561856] [--pin 0,1] [--json]

prints, per slot count and policy, the hit rate, the misses, the compulsory
misses and the bytes the misses copy; `--pin` pins whole layers (every expert
of each listed layer seen in the trace) first.
"""
from __future__ import annotations

import argparse
import json
import sys
from collections import defaultdict, deque

import numpy as np


def trace_from_counts(layer: int, counts) -> tuple:
    """(layer, touched experts) of one forward from its per-expert pair counts."""
    return int(layer), tuple(int(e) for e in np.flatnonzero(np.asarray(counts) > 0))


def replay(trace, slots: int, policy: str = "tier", expert_bytes: int = 0, pin=()) -> dict:
    """Hits, misses and bytes copied when `trace` runs on `slots` slots.

    Every forward's experts must fit at once (slots >= the most experts any one
    forward touches), as the tier requires. compulsory = the distinct
    (layer, expert) keys: the misses no policy can avoid. `pin`: (layer,
    experts) entries placed before the trace in slots no eviction takes (the
    pages' pinned slots, `k3moe_tier_pin_layer`); their copies are counted in
    `pin_copies`, not in the misses."""
    if policy not in ("tier", "belady"):
        raise ValueError(f"unknown policy {policy!r}")
    trace = [(int(layer), tuple(sorted(set(int(e) for e in ex)))) for layer, ex in trace]
    if any(len(ex) > slots for _, ex in trace):
        raise ValueError("a forward touches more experts than there are slots")
    nxt = defaultdict(deque)   # key -> forward indices where it is used
    for i, (layer, ex) in enumerate(trace):
        for e in ex:
            nxt[(layer, e)].append(i)
    key = [None] * slots       # slot -> (layer, expert) or None
    used = [0] * slots         # slot -> stamp of its last forward (0: never)
    where = {}                 # (layer, expert) -> slot
    hits = misses = 0
    PIN = float("inf")         # a pinned slot: never below a forward's stamp
    pin_keys = sorted({(int(l), int(e)) for l, ex in pin for e in ex})
    if len(pin_keys) > slots:
        raise ValueError("more pinned experts than slots")
    for s_, k in enumerate(pin_keys):
        key[s_], used[s_], where[k] = k, PIN, s_
    for i, (layer, ex) in enumerate(trace):
        stamp = i + 1
        miss = []
        for e in ex:
            k = (layer, e)
            nxt[k].popleft()
            if k in where:
                if used[where[k]] != PIN:
                    used[where[k]] = stamp
                hits += 1
            else:
                miss.append(k)
        free = [s for s in range(slots) if used[s] < stamp]
        if len(free) < len(miss):
            raise ValueError("a forward's misses do not fit beside the pinned slots")
        if policy == "tier":
            chosen = sorted(sorted(free, key=lambda s: (used[s], s))[:len(miss)])
        else:   # furthest next use first; never used again counts as infinitely far
            def far(s):
                k = key[s]
                if k is None:
                    return (2, 0, s)
                return (1, nxt[k][0] if nxt[k] else 1 << 60, -s)
            chosen = sorted(sorted(free, key=far, reverse=True)[:len(miss)])
        for k, s in zip(miss, chosen):
            if key[s] is not None:
                del where[key[s]]
            key[s] = k
            where[k] = s
            used[s] = stamp
        misses += len(miss)
    total = hits + misses
    return {"slots": slots, "policy": policy, "hits": hits, "misses": misses,
            "hit_rate": hits / total if total else 0.0, "compulsory": len(nxt),
            "bytes_copied": misses * int(expert_bytes), "pin_copies": len(pin_keys)}


def save_trace(path: str, trace) -> None:
    """Writes a trace as JSON lines, one [layer, [experts...]] per forward."""
    with open(path, "w") as f:
        for layer, ex in trace:
            f.write(json.dumps([int(layer), [int(e) for e in ex]]) + "\n")


def save_counts(path: str, layers, counts) -> None:
    """Writes per-forward expert counts (as `k3moe_get_routing` returns them)
    and each forward's layer as an .npz trace."""
    layers, counts = np.asarray(layers, np.int32), np.asarray(counts, np.int32)
    if counts.ndim != 2 or layers.shape != (counts.shape[0],):
        raise ValueError("layers [n] and counts [n, E] expected")
    with open(path, "wb") as f:   # a file object: np.savez adds no suffix
        np.savez(f, layers=layers, counts=counts)


def load_trace(path: str) -> list:
    """Reads a trace written by `save_trace`, or an .npz of `layers` [n] and
    per-forward expert `counts` [n, E]."""
    with open(path, "rb") as f:
        is_npz = f.read(2) == b"PK"   # a zip archive
    if is_npz:
        z = np.load(path)
        layers, counts = np.asarray(z["layers"]), np.asarray(z["counts"])
        if counts.ndim != 2 or layers.shape != (counts.shape[0],):
            raise ValueError("an .npz trace holds layers [n] and counts [n, E]")
        return [trace_from_counts(l, c) for l, c in zip(layers, counts)]
    out = []
    with open(path) as f:
        for i, line in enumerate(f):
            if not line.strip():
                continue
            rec = json.loads(line)
            if (not isinstance(rec, list) or len(rec) != 2 or not isinstance(rec[1], list)):
                raise ValueError(f"line {i + 1}: expected [layer, [experts...]]")
            out.append((int(rec[0]), tuple(int(e) for e in rec[1])))
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(prog="python -m mxfp4_routed_expert_gb300.tier_trace",
                                 description="Replay a routing trace at several expert-tier sizes.")
    ap.add_argument("trace", help="JSON lines of [layer, [experts]] or an .npz of layers, counts")
    ap.add_argument("--slots", required=True, help="comma-separated slot counts")
    ap.add_argument("--expert-bytes", type=int, default=0, help="bytes of one expert (copied per miss)")
    ap.add_argument("--pin", default="", help="comma-separated layers to pin before the trace")
    ap.add_argument("--json", action="store_true", help="one JSON object per line instead of a table")
    a = ap.parse_args(argv)
    trace = load_trace(a.trace)
    slots = [int(v) for v in a.slots.split(",") if v.strip()]
    pin_layers = {int(v) for v in a.pin.split(",") if v.strip()}
    seen = defaultdict(set)
    for layer, ex in trace:
        seen[layer].update(ex)
    pin = [(l, sorted(seen[l])) for l in sorted(pin_layers)]
    rows = []
    for n in slots:
        for policy in ("tier", "belady"):
            try:
                rows.append(replay(trace, n, policy, expert_bytes=a.expert_bytes, pin=pin))
            except ValueError as e:
                rows.append({"slots": n, "policy": policy, "error": str(e)})
    for r in rows:
        if a.json:
            print(json.dumps(r))
        elif "error" in r:
            print(f"{r['slots']:>7} {r['policy']:>7}  {r['error']}")
        else:
            print(f"{r['slots']:>7} {r['policy']:>7}  hit rate {r['hit_rate']:.4f}  misses {r['misses']}"
                  f"  compulsory {r['compulsory']}  copied {r['bytes_copied'] / 1e9:.3f} GB")
    return 0


if __name__ == "__main__":
    sys.exit(main())
