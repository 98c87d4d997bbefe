"""Seeded synthetic workloads of the five configurations (shapes, value distributions and tensor ids).

Only draws numbers (see ``synth.c``); the oracle and the CUDA path both take their inputs from here.

Value recipe (all seed 0 unless a test says otherwise):
  Q8_0 matrices  quants U[-127, 127]; block scales |N(0,1)| * 0.01 (router scales * 1e-3 in the spread-gate variant)
  activations    N(0,1); residual stream N(0,1); norm and QK-norm weights 1 + 0.1 * N(0,1)
  embedding      N(0,1) f32 [vocab, d];  KV cache N(0,1) f32, every position filled
"""
from __future__ import annotations

import numpy as np

from . import fill_f32_ptr, fill_i8_ptr, normal, q8_matrix

MAT = 0                 # Q8_0 matrix ids (streams 2t, 2t+1)
VEC = 1 << 44           # every other tensor


def layer_ids(l: int) -> dict:
    b = 1000 + 32 * l
    return dict(wq=b, wk=b + 1, wv=b + 2, wo=b + 3, router=b + 4, gate=b + 5, up=b + 6, down=b + 7,
                attn_norm=VEC + b + 8, ffn_norm=VEC + b + 9, q_norm=VEC + b + 10, k_norm=VEC + b + 11,
                k_cache=VEC + b + 12, v_cache=VEC + b + 13, shared_gate=b + 14, shared_up=b + 15,
                shared_down=b + 16, router_f32=VEC + b + 17)


EMBED = VEC + 1
FINAL_NORM = VEC + 2
LM_HEAD = 3

# config 4: 48 layers of d=2048, 32 query / 4 key-value heads of 128, 128 experts keep 8 of dff 768, vocab 151936,
# f32 cache of 4096 positions, RoPE theta 1e6, eps 1e-6
DECODE = dict(layers=48, d=2048, heads=32, kv_heads=4, hd=128, experts=128, k=8, dff=768, vocab=151936, ctx=4096,
              eps=1e-6, rope_theta=1e6)
MOE = dict(d=2048, experts=128, k=8, dff=768)


def moe_block(seed=0, d=2048, dff=768, experts=128, router_scale=0.01, l=0):
    """Host arrays of one mixture (config 2): router [E,d], gate/up [E*dff,d], down [E*d,dff]."""
    ids = layer_ids(l)
    return dict(
        router=q8_matrix(experts, d, seed, ids["router"], scale_mul=router_scale),
        gate=q8_matrix(experts * dff, d, seed, ids["gate"]),
        up=q8_matrix(experts * dff, d, seed, ids["up"]),
        down=q8_matrix(experts * d, dff, seed, ids["down"]),
    )


def _alloc_np(shape, dtype):
    return np.empty(shape, dtype)


def decode_model(cfg: dict, seed: int = 0, alloc=_alloc_np, ptr=lambda a: a.ctypes.data):
    """Every host array of a decode model.  ``alloc(shape, dtype)`` makes each array (numpy by default; pinned torch
    tensors for a fast upload) and ``ptr(a)`` gives its host address."""
    L, d, H, KV, hd = cfg["layers"], cfg["d"], cfg["heads"], cfg["kv_heads"], cfg["hd"]
    E, dff, V, ctx = cfg["experts"], cfg["dff"], cfg["vocab"], cfg["ctx"]

    def mat(n, k, t):
        q = alloc((n, k), np.int8)
        s = alloc((n, k // 32), np.float32)
        fill_i8_ptr(ptr(q), n * k, seed, 2 * t)
        fill_f32_ptr(ptr(s), n * (k // 32), seed, 2 * t + 1, mul=0.01, absval=True)
        return q, s

    def vec(shape, t, mul=1.0, add=0.0):
        a = alloc(shape, np.float32)
        fill_f32_ptr(ptr(a), int(np.prod(shape)), seed, t, mul=mul, add=add)
        return a

    out = dict(embed=vec((V, d), EMBED), final_norm=vec((d,), FINAL_NORM, 0.1, 1.0), lm_head=mat(V, d, LM_HEAD))
    for key in ("attn_norm", "ffn_norm", "q_norm", "k_norm", "wq", "wk", "wv", "wo", "router", "gate", "up", "down",
                "k_cache", "v_cache"):
        out[key] = []
    for l in range(L):
        ids = layer_ids(l)
        out["attn_norm"].append(vec((d,), ids["attn_norm"], 0.1, 1.0))
        out["ffn_norm"].append(vec((d,), ids["ffn_norm"], 0.1, 1.0))
        out["q_norm"].append(vec((hd,), ids["q_norm"], 0.1, 1.0))
        out["k_norm"].append(vec((hd,), ids["k_norm"], 0.1, 1.0))
        out["wq"].append(mat(H * hd, d, ids["wq"]))
        out["wk"].append(mat(KV * hd, d, ids["wk"]))
        out["wv"].append(mat(KV * hd, d, ids["wv"]))
        out["wo"].append(mat(d, H * hd, ids["wo"]))
        out["router"].append(mat(E, d, ids["router"]))
        out["gate"].append(mat(E * dff, d, ids["gate"]))
        out["up"].append(mat(E * dff, d, ids["up"]))
        out["down"].append(mat(E * d, dff, ids["down"]))
        out["k_cache"].append(vec((KV, ctx, hd), ids["k_cache"]))
        out["v_cache"].append(vec((KV, ctx, hd), ids["v_cache"]))
    return out


def mixture_variants(cfg: dict, seed: int = 0, shared_dff: int = 0, router_f32: bool = False, layers=None) -> dict:
    """The optional mixture variants of a model, per layer: a shared expert of width ``shared_dff`` (gate/up
    [shared_dff, d], down [d, shared_dff], Q8_0 as the experts) and routers of f32 values N(0,1) * 0.02 [E, d] (logits
    of about unit spread at d = 2048)."""
    L, d, E = cfg["layers"], cfg["d"], cfg["experts"]
    out = {}
    rng = range(L) if layers is None else layers
    if shared_dff:
        out["shared_gate"] = [q8_matrix(shared_dff, d, seed, layer_ids(l)["shared_gate"]) for l in rng]
        out["shared_up"] = [q8_matrix(shared_dff, d, seed, layer_ids(l)["shared_up"]) for l in rng]
        out["shared_down"] = [q8_matrix(d, shared_dff, seed, layer_ids(l)["shared_down"]) for l in rng]
    if router_f32:
        out["router_f32"] = [normal((E, d), seed, layer_ids(l)["router_f32"], mul=0.02) for l in rng]
    return out


def weight_bytes_per_token(cfg: dict) -> int:
    """Q8_0 bytes (quants + scales, 1.125 B per weight) one decode step reads: every dense projection, the router, the
    k kept experts' gate/up/down rows per layer, and the LM head."""
    L, d, H, KV, hd = cfg["layers"], cfg["d"], cfg["heads"], cfg["kv_heads"], cfg["hd"]
    per_layer = (H * hd * d + 2 * KV * hd * d + d * H * hd + cfg["experts"] * d + cfg["k"] * 3 * cfg["dff"] * d)
    return int((L * per_layer + cfg["vocab"] * d) * 9 // 8)


def kv_bytes_per_token(cfg: dict, pos: int) -> int:
    """f32 cache bytes the attention reads at position ``pos`` (rows 0..pos of every key/value head, keys and values)."""
    return int(cfg["layers"] * 2 * cfg["kv_heads"] * (pos + 1) * cfg["hd"] * 4)


def activations(rows, d, seed, tensor):
    return normal((rows, d), seed, VEC + tensor)
