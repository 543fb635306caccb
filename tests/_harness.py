"""Shared test helpers: seeded layers and tokens, the routing margin guard,
the parity metrics, and thin wrappers that move numpy inputs through the
C ABI with torch-allocated device memory.

Tolerances of the layer: expert ids and the permutation bit-exact;
floating-point outputs within normwise max relative error 2e-2
(max_i |y_i - y*_i| / max_i |y*_i|, the pages' "relative to max|ref|" logit
metric) and cosine similarity >= 0.9995 against the fp64 oracle.
"""
from __future__ import annotations

import numpy as np

import k3synth
import oracle

REL_TOL = 2e-2
COS_TOL = 0.9995
MARGIN_TAU = 1e-4        # routing near-tie guard on the 16th-vs-17th selection score


def relerr(y, ref):
    return float(np.abs(np.asarray(y, np.float64) - ref).max() / max(np.abs(ref).max(), 1e-300))


def cosine(y, ref):
    a = np.asarray(y, np.float64).ravel()
    b = np.asarray(ref, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def assert_close(y, ref, what="y", rel=REL_TOL, cos=COS_TOL):
    r, c = relerr(y, ref), cosine(y, ref)
    assert r <= rel and c >= cos, f"{what}: relerr {r:.3e} (<= {rel}), cosine {c:.6f} (>= {cos})"
    return r, c


def guarded_tokens(shape, layer, seed, T, stream=0, tau=MARGIN_TAU, make=None, max_rounds=50):
    """Tokens whose oracle routing margin (k-th minus (k+1)-th selection score)
    is at least tau: tokens below it are redrawn from their next attempt
    stream. The guard uses only the oracle's router; the generator only
    supplies numbers."""
    att = np.zeros(T, np.int32)
    make = make or (lambda attempts: k3synth.make_tokens(shape, seed, T, stream, attempts))
    x = make(att)
    for _ in range(max_rounds):
        _, _, margin = oracle.route(shape, layer, x)
        bad = margin < tau
        if not bad.any():
            return x, att
        att[bad] += 1
        x = make(att)
    raise RuntimeError("margin guard did not converge")


def router_only_layer(shape, router: dict):
    """(shape, layer) for oracle.route from the router tensors alone: the route
    reads only router_w and router_bias, so the other tensors are zeros of a
    layer whose latent, expert and shared widths are 32 (a few hundred KB
    instead of the full layer)."""
    small = k3synth.replace(shape, latent=32, moe_inter=32, shared_inter=32)
    H, L, E, I, S = small.hidden, small.latent, small.n_experts, small.moe_inter, small.shared_inter
    z16 = lambda *s: np.zeros(s, np.uint16)   # noqa: E731
    z8 = lambda *s: np.zeros(s, np.uint8)     # noqa: E731
    d = {"router_w": router["router_w"], "router_bias": router["router_bias"],
         "down_w": z16(L, H), "up_w": z16(H, L), "latent_gain": z16(L), "sh_w1": z16(S, H),
         "sh_w3": z16(S, H), "sh_w2": z16(H, S), "w1p": z8(E, I, L // 2), "w1s": z8(E, I, L // 32),
         "w3p": z8(E, I, L // 2), "w3s": z8(E, I, L // 32), "w2p": z8(E, L, I // 2),
         "w2s": z8(E, L, I // 32)}
    return small, d


def ids_match(ids_gpu, ids_ref):
    """Per-token id SETS must match exactly (slot order inside a token is by
    selection score and is compared separately where scores are well apart)."""
    a = np.sort(np.asarray(ids_gpu), axis=1)
    b = np.sort(np.asarray(ids_ref), axis=1)
    return np.array_equal(a, b)


# ---- device side (imported lazily: CPU-only tests never touch CUDA) ---------------

class Layer:
    """One library handle with layers loaded from numpy tensors."""

    def __init__(self, shape, layers: list, max_tokens: int, device: int = 0,
                 latent_norm: int = 1, tier_slots: int = 0):
        import torch  # noqa: F401
        import mxfp4_routed_expert_gb300 as km
        self.km = km
        self.shape = shape
        cfg = km.make_config(shape, max_layers=len(layers), max_tokens=max_tokens, device=device,
                             latent_norm=latent_norm)
        self.h = km.k3moe_create(cfg)
        if tier_slots:
            km.k3moe_set_expert_tier(self.h, tier_slots)
        for i, d in enumerate(layers):
            if d is not None:
                self.load(i, d)

    def load(self, i, d):
        w, keep = self.km.layer_weights(d, self.shape.n_experts, self.km.K3MOE_HOST)
        self.km.k3moe_load_layer(self.h, i, w)
        del keep

    def close(self):
        if self.h:
            self.km.k3moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x_bits: np.ndarray, layer: int = 0, chain: int = 0):
        import torch
        T = x_bits.shape[0]
        x = torch.from_numpy(x_bits.view(np.int16).copy()).cuda()
        y = torch.empty_like(x)
        if chain:
            self.km.k3moe_forward_chain(self.h, layer, chain, x, y, T)
        else:
            self.km.k3moe_forward(self.h, layer, x, y, T)
        torch.cuda.synchronize()
        st = self.km.k3moe_sync_status(self.h)
        assert st == 0, self.km.strerror(st)
        return y.cpu().numpy().view(np.uint16)

    def forward_residual(self, h_f32: np.ndarray, layer: int = 0):
        """y (bf16 bits) of the layer on bf16(RMSNorm(h) * post-norm gain)."""
        import torch
        T = h_f32.shape[0]
        hd = torch.from_numpy(np.ascontiguousarray(h_f32, np.float32)).cuda()
        y = torch.empty((T, self.shape.hidden), dtype=torch.int16, device="cuda")
        self.km.k3moe_forward_residual(self.h, layer, hd, y, T)
        torch.cuda.synchronize()
        st = self.km.k3moe_sync_status(self.h)
        assert st == 0, self.km.strerror(st)
        return y.cpu().numpy().view(np.uint16)

    def layer_input(self, T):
        """bf16 bits [T, H] of the input the last residual forward made."""
        import torch
        buf = torch.empty((T, self.shape.hidden), dtype=torch.int16, device="cuda")
        self.km.k3moe_get_intermediate(self.h, self.km.K3MOE_T_X, buf, buf.numel() * 2)
        torch.cuda.synchronize()
        return buf.cpu().numpy().view(np.uint16)

    def routing(self, T):
        import torch
        s = self.shape
        ids = torch.empty((T, s.topk), dtype=torch.int32, device="cuda")
        w = torch.empty((T, s.topk), dtype=torch.float32, device="cuda")
        counts = torch.empty(s.n_experts, dtype=torch.int32, device="cuda")
        offsets = torch.empty(s.n_experts + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(T * s.topk, dtype=torch.int32, device="cuda")
        self.km.k3moe_get_routing(self.h, ids, w, counts, offsets, perm)
        torch.cuda.synchronize()
        return dict(ids=ids.cpu().numpy(), w=w.cpu().numpy(), counts=counts.cpu().numpy(),
                    offsets=offsets.cpu().numpy(), perm=perm.cpu().numpy())

    def intermediate(self, which, T, width):
        import torch
        buf = torch.empty((T, width), dtype=torch.float32, device="cuda")
        self.km.k3moe_get_intermediate(self.h, which, buf, buf.numel() * 4)
        torch.cuda.synchronize()
        return buf.cpu().numpy()


def bf16_to_f64(bits):
    return k3synth.bf16_bits_to_f32(bits).astype(np.float64)


def check_ids_and_weights(ids_gpu, w_gpu, oracle_ids, oracle_w, tol=1e-5):
    """Exact id sets per token; each picked expert's weight within tol."""
    assert ids_match(ids_gpu, oracle_ids), "expert id sets differ"
    for t in range(np.asarray(ids_gpu).shape[0]):
        og = dict(zip(np.asarray(oracle_ids)[t].tolist(), np.asarray(oracle_w)[t].tolist()))
        for e, wv in zip(np.asarray(ids_gpu)[t].tolist(), np.asarray(w_gpu)[t].tolist()):
            assert abs(wv - og[e]) < tol, (t, e, wv, og[e])


def check_routing(gpu: dict, shape, x_bits, oracle_ids, oracle_w):
    """Exact ids and permutation; weights to 1e-5."""
    T = x_bits.shape[0]
    assert ids_match(gpu["ids"], oracle_ids), "expert id sets differ"
    counts, offsets, perm = oracle.permutation(gpu["ids"], shape.n_experts)
    ref_c, ref_o, ref_p = oracle.permutation(oracle_ids, shape.n_experts)
    np.testing.assert_array_equal(gpu["counts"], ref_c)
    np.testing.assert_array_equal(gpu["offsets"], ref_o)
    # perm lists flat (t, j) pair indices; compare as (token, expert) pairs since
    # the slot j of an expert inside a token follows the per-token order
    # (only the first offsets[E] entries are pairs: a weight cut drops some)
    n = int(ref_o[-1])
    ids_g = gpu["ids"].ravel()
    pairs_g = np.stack([gpu["perm"][:n] // shape.topk, ids_g[gpu["perm"][:n]]], 1)
    ids_o = np.asarray(oracle_ids).ravel()
    pairs_o = np.stack([ref_p[:n] // shape.topk, ids_o[ref_p[:n]]], 1)
    np.testing.assert_array_equal(pairs_g, pairs_o)
    assert sorted(gpu["perm"][:n].tolist()) == np.flatnonzero(ids_g >= 0).tolist()
    # weights, matched by expert id
    for t in range(T):
        og = dict(zip(np.asarray(oracle_ids)[t].tolist(), np.asarray(oracle_w)[t].tolist()))
        for e, wv in zip(gpu["ids"][t].tolist(), gpu["w"][t].tolist()):
            assert abs(wv - og[e]) < 1e-5
