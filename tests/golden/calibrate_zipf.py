"""Writes zipf_alpha.json: the strength of the per-expert router bias that
gives the K3 prefill workload (T = 4096) a Zipf(1.1) expert popularity.

bias_e = alpha * ln((pi(e) + 1)^-1.1) with pi a seeded permutation
(k3synth.zipf_bias). For a given alpha, 1024 seeded tokens are routed by the
oracle and the expert pick counts are sorted; alpha is bisected until the
least-squares slope of ln(count) against ln(rank) over ranks 1..256 is -1.1.
Uses only the generator and the oracle. Run: python tests/golden/calibrate_zipf.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import k3synth  # noqa: E402
import oracle  # noqa: E402

SEED, LAYER, STREAM, T, TARGET = 0, 0, 11, 1024, -1.1


def slope(alpha, router, x):
    shape = k3synth.K3
    lay = dict(router)
    lay["router_bias"] = k3synth.zipf_bias(shape, SEED, LAYER, alpha)
    # only the router tensors matter for route(); placeholders fill the rest
    ids, _, _ = route_only(shape, lay, x)
    counts = np.sort(np.bincount(ids.ravel(), minlength=shape.n_experts))[::-1].astype(float)
    r = np.arange(1, 257)
    c = np.maximum(counts[:256], 0.5)
    return float(np.polyfit(np.log(r), np.log(c), 1)[0]), counts


def route_only(shape, router, x):
    E, H, L, I, S = shape.n_experts, shape.hidden, shape.latent, shape.moe_inter, shape.shared_inter
    d = {k: v for k, v in router.items()}
    # route() reads only the router weights and bias; the other tensors are
    # required by the marshalling layer, so tiny stand-ins with the right
    # shapes are passed as zero-stride views
    z16 = np.zeros(1, np.uint16)
    z8 = np.zeros(1, np.uint8)
    def view(a, shp):
        return np.lib.stride_tricks.as_strided(a, shape=shp, strides=(0,) * len(shp))
    d.update(down_w=view(z16, (L, H)), up_w=view(z16, (H, L)), latent_gain=view(z16, (L,)),
             sh_w1=view(z16, (S, H)), sh_w3=view(z16, (S, H)), sh_w2=view(z16, (H, S)),
             w1p=view(z8, (E, I, L // 2)), w1s=view(z8, (E, I, L // 32)),
             w3p=view(z8, (E, I, L // 2)), w3s=view(z8, (E, I, L // 32)),
             w2p=view(z8, (E, L, I // 2)), w2s=view(z8, (E, L, I // 32)))
    return oracle.route(shape, d, x)


def main():
    shape = k3synth.K3
    router = k3synth.make_router(shape, SEED, LAYER)
    x = k3synth.make_tokens(shape, SEED, T, stream=STREAM)
    lo, hi = 0.0, 2.0
    for _ in range(14):
        mid = 0.5 * (lo + hi)
        s, _ = slope(mid, router, x)
        if s > TARGET:      # not steep enough: stronger bias
            lo = mid
        else:
            hi = mid
    alpha = 0.5 * (lo + hi)
    s, counts = slope(alpha, router, x)
    out = {"alpha": round(alpha, 6), "slope": round(s, 4), "tokens": T, "seed": SEED,
           "token_stream": STREAM, "hottest": int(counts[0]), "median": float(np.median(counts)),
           "touched": int((counts > 0).sum()),
           "source": "written by tests/golden/calibrate_zipf.py (generator + oracle router only)"}
    with open(os.path.join(HERE, "zipf_alpha.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
