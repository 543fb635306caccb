"""Accuracy of the routed experts' activation formats at K3 size, measured
against the fp64 oracle on the CPU.

The block-scaled tensor-core MMA (kind::mxf8f6f4) multiplies the stored e2m1
weights with 8-bit activations, so z (the latent, input of W1/W3) and h (the
SiTU output, input of W2) must be rounded to an 8-bit format first. This
script measures what each candidate rounding does to the layer's output y,
with the metrics of the parity tests (normwise max relative error and
cosine against the oracle's y):

  exact  - no rounding (the recomposition below must then equal the oracle's
           own layer to rounding noise; the script checks that first)
  f16    - the tensor-core path as built: z scaled by a per-token power of two
           into [32, 64) and rounded to f16, h rounded to f16
  mx     - MXFP8: per 32 consecutive elements one ue8m0 scale (the smallest
           power of two that brings the group's largest magnitude to <= 448)
           and e4m3 elements, round to nearest even
  hilo   - two MXFP8 terms: hi = mx(v), and lo = the residual v - hi in e4m3
           with a scale 2^-4 times hi's (the residual's largest scaled value
           is 16, half the e4m3 spacing of the top binade [256, 448], so it
           reaches at most 256): the rounding the tensor-core path applies

Combinations measured, written (z format for W1, z format for W3) / h
format, with one z format meaning both: exact/exact, f16/f16, mx/mx,
hilo/hilo, f16/mx (8-bit h only), mx/f16 (8-bit z only), and the per-matrix
splits (mx,hilo)/mx and (hilo,mx)/mx (SiTU saturates in the gate, so W1's
rounding may matter less than W3's).

The layer is recomposed from the oracle's own routines: z, the routing and
the shared-expert activations come from its trace; the expert products are
oracle.mxfp4_matvec on the rounded activations, SiTU is oracle.situ, the
latent norm oracle.rmsnorm and the projections back up oracle.bf16_matvec.
The only arithmetic written here is the rounding under study and the
weighted sum of the experts' outputs.

Workloads: K3 T = 64 with every expert touched (the covering construction,
zero bias) and K3 T = 4096 with Zipf(1.1) popularity on every 16th token,
each with the margin guard of the parity tests. One K3 layer is generated in
host memory (16 GB). Run:

    python tests/study_activation_formats.py [--threads N] [--rows-4096 N]
        [--out tests/golden/activation_formats.json]
"""
import argparse
import json
import os
import sys
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import k3synth  # noqa: E402
import oracle  # noqa: E402
from _harness import cosine, guarded_tokens, relerr  # noqa: E402

E4M3_MAX = 448.0
GROUP = 32


def round_e4m3(v):
    """fp64 -> nearest e4m3 value (3 mantissa bits, exponent bias 7, normals
    from 2^-6, subnormal step 2^-9, largest 448), ties to even. Inputs must
    already lie within [-448, 448]."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    assert np.all(a <= E4M3_MAX)
    _, e = np.frexp(a)                           # a = m 2^e, m in [0.5, 1)
    ulp = np.where(a >= 2.0 ** -6, e - 4, -9)    # 2^(e-1-3) for normals
    return np.copysign(np.ldexp(np.round(np.ldexp(a, -ulp)), ulp), v)


def q_mx(v):
    """MXFP8 (e4m3 elements, one power-of-two scale per 32 along the last
    axis) rounding of v, returned as the fp64 values it represents."""
    v = np.asarray(v, np.float64)
    shp = v.shape
    g = v.reshape(-1, shp[-1] // GROUP, GROUP)
    amax = np.abs(g).max(axis=-1, keepdims=True)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / E4M3_MAX)), 0.0)
    # log2 rounding: make sure amax * 2^-ex <= 448 exactly, and no smaller
    ex = np.where(np.ldexp(amax, -ex.astype(np.int64)) > E4M3_MAX, ex + 1, ex)
    ex = np.clip(ex, -127, 127).astype(np.int64)
    q = round_e4m3(np.ldexp(g, -ex))
    return np.ldexp(q, ex).reshape(shp)


def mx_exponents(v):
    """Per-group scale exponent of q_mx, broadcast back to v's shape."""
    v = np.asarray(v, np.float64)
    g = v.reshape(-1, v.shape[-1] // GROUP, GROUP)
    amax = np.abs(g).max(axis=-1, keepdims=True)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / E4M3_MAX)), 0.0)
    ex = np.where(np.ldexp(amax, -ex.astype(np.int64)) > E4M3_MAX, ex + 1, ex)
    ex = np.clip(ex, -127, 127).astype(np.int64)
    return np.broadcast_to(ex, g.shape).reshape(v.shape)


def q_hilo(v):
    v = np.asarray(v, np.float64)
    hi = q_mx(v)
    el = np.maximum(mx_exponents(v) - 4, -127)
    return hi + np.ldexp(round_e4m3(np.ldexp(v - hi, -el)), el)


def q_f16_z(v):
    """Per token (row) a power of two that brings the row maximum into
    [32, 64), then f16 round to nearest even (the built path's z16)."""
    v = np.asarray(v, np.float64)
    m = np.abs(v).max(axis=-1, keepdims=True)
    ex = np.where(m > 0, np.frexp(np.where(m > 0, m, 1.0))[1] - 1 - 5, 0)
    return np.ldexp(np.ldexp(v, -ex).astype(np.float16).astype(np.float64), ex)


def q_f16(v):
    return np.asarray(v, np.float64).astype(np.float16).astype(np.float64)


QZ = {"exact": lambda v: np.asarray(v, np.float64), "f16": q_f16_z, "mx": q_mx, "hilo": q_hilo}
QH = {"exact": lambda v: np.asarray(v, np.float64), "f16": q_f16, "mx": q_mx, "hilo": q_hilo}
# (z format for W1, z format for W3, h format)
COMBOS = [("exact", "exact", "exact"), ("f16", "f16", "f16"), ("mx", "mx", "mx"),
          ("hilo", "hilo", "hilo"), ("f16", "f16", "mx"), ("mx", "mx", "f16"),
          ("mx", "hilo", "mx"), ("hilo", "mx", "mx")]


def combo_name(c):
    z = c[0] if c[0] == c[1] else f"({c[0]},{c[1]})"
    return f"{z}/{c[2]}"


def study(shape, d, x, rows, threads):
    """y [len(rows), H] for every combination, and the oracle's own y."""
    L, I, K = shape.latent, shape.moe_inter, shape.topk
    y_ref, tr = oracle.layer_forward(shape, d, x, rows=rows, trace=True)
    n = rows.size
    zfmts = sorted({c[0] for c in COMBOS} | {c[1] for c in COMBOS})
    situ = np.vectorize(lambda g, u: oracle.situ(g, u, shape.situ_b1, shape.situ_b2))

    def one_pair(r, j):
        e = int(tr["ids"][r, j])
        zq = {zf: QZ[zf](tr["z"][r][None, :])[0] for zf in zfmts}
        g = {zf: oracle.mxfp4_matvec(zq[zf], d["w1p"][e], d["w1s"][e], L)
             for zf in {c[0] for c in COMBOS}}
        u = {zf: oracle.mxfp4_matvec(zq[zf], d["w3p"][e], d["w3s"][e], L)
             for zf in {c[1] for c in COMBOS}}
        out = {}
        for c in COMBOS:
            h = situ(g[c[0]], u[c[1]])
            hq = QH[c[2]](h[None, :])[0]
            out[c] = oracle.mxfp4_matvec(hq, d["w2p"][e], d["w2s"][e], I)
        return r, j, out

    acc = {c: np.zeros((n, L)) for c in COMBOS}
    jobs = [(r, j) for r in range(n) for j in range(K) if tr["ids"][r, j] >= 0]
    with ThreadPoolExecutor(threads) as ex:
        for r, j, out in ex.map(lambda a: one_pair(*a), jobs):
            for c, o in out.items():
                acc[c][r] += tr["w"][r, j] * o
    gain = k3synth.bf16_bits_to_f32(d["latent_gain"]).astype(np.float64)
    ys = {}
    for c in COMBOS:
        y = np.empty((n, shape.hidden))
        for r in range(n):
            nrm = oracle.rmsnorm(acc[c][r], gain, shape.rms_eps)
            y[r] = oracle.bf16_matvec(nrm, d["up_w"]) + oracle.bf16_matvec(tr["shared"][r], d["sh_w2"])
        ys[c] = (y, acc[c])
    return y_ref, tr, ys


def report(name, y_ref, tr, ys):
    res = {}
    for c, (y, acc) in ys.items():
        key = combo_name(c)
        cos_tok = [cosine(y[r], y_ref[r]) for r in range(y.shape[0])]
        res[key] = {"y_relerr": relerr(y, y_ref), "y_cosine": cosine(y, y_ref),
                    "y_min_token_cosine": float(min(cos_tok)),
                    "acc_relerr": relerr(acc, tr["acc"]), "acc_cosine": cosine(acc, tr["acc"])}
        print(f"{name:>14} {key:>10}  y relerr {res[key]['y_relerr']:.3e}  cos {res[key]['y_cosine']:.6f}"
              f"  (min token {res[key]['y_min_token_cosine']:.5f})  acc relerr {res[key]['acc_relerr']:.3e}"
              f"  cos {res[key]['acc_cosine']:.6f}", flush=True)
    assert res["exact/exact"]["y_relerr"] < 1e-12, "recomposition differs from the oracle's layer"
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--threads", type=int, default=os.cpu_count())
    ap.add_argument("--rows-4096", type=int, default=256,
                    help="tokens of the T=4096 workload measured (every 4096/N-th)")
    ap.add_argument("--out", default=None)
    a = ap.parse_args()
    shape = k3synth.K3
    t0 = time.time()
    d = k3synth.make_layer(shape, 0, 0, k3synth.K3_RECIPE)
    print(f"layer generated in {time.time() - t0:.0f} s", flush=True)
    results = {}

    d0 = k3synth.with_bias(d, np.zeros(shape.n_experts, np.float32))
    x, _ = guarded_tokens(shape, d0, 0, 64,
                          make=lambda att: k3synth.covering_tokens(shape, d0, 0, 64, attempts=att))
    rows = np.arange(64, dtype=np.int32)
    results["k3_t64_covering"] = report("T=64 covering", *study(shape, d0, x, rows, a.threads))

    dz = k3synth.with_bias(d, k3synth.zipf_bias(shape, 0, 0, k3synth.K3_ZIPF_ALPHA))
    x, _ = guarded_tokens(shape, dz, 0, 4096, stream=11)
    rows = np.arange(0, 4096, 4096 // a.rows_4096, dtype=np.int32)
    results["k3_t4096_zipf"] = report("T=4096 Zipf", *study(shape, dz, x, rows, a.threads))
    results["tokens"] = {"k3_t64_covering": 64, "k3_t4096_zipf": int(rows.size)}
    print(f"done in {time.time() - t0:.0f} s")
    if a.out:
        with open(a.out, "w") as f:
            json.dump(results, f, indent=1, sort_keys=True)
            f.write("\n")


if __name__ == "__main__":
    main()
