"""CPU oracle (ctypes wrapper over ``liboracle.so``) — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import this package.  It shares no
code with the CUDA path and imports nothing from it.  Every function returns numpy arrays computed by the plain C
restatement in ``oracle.c`` (f64 unless the pages fix another precision).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

QBLOCK = 32


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler: IEEE arithmetic, no contraction, no fast-math; with OpenMP when the
    compiler has it (only for the optional all-cores mode), else single-threaded."""
    srcs = [os.path.join(_HERE, "oracle.c")]
    deps = srcs + [os.path.join(_HERE, "oracle.h")]
    if force or not os.path.exists(_LIB_PATH) or any(os.path.getmtime(_LIB_PATH) < os.path.getmtime(p) for p in deps):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-fPIC", "-shared", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", *srcs, "-o", tmp]
        if subprocess.run(base + ["-fopenmp", "-lm"], capture_output=True).returncode != 0:
            subprocess.check_call(base + ["-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Q8(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p)]


class Moe(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("dff", ctypes.c_int64), ("experts", ctypes.c_int64), ("k", ctypes.c_int),
                ("router", Q8), ("gate", Q8), ("up", Q8), ("down", Q8), ("router_f32", ctypes.c_void_p),
                ("sdff", ctypes.c_int64), ("sgate", Q8), ("sup", Q8), ("sdown", Q8)]


class Model(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int64), ("d", ctypes.c_int64), ("heads", ctypes.c_int64),
                ("kv_heads", ctypes.c_int64), ("hd", ctypes.c_int64), ("vocab", ctypes.c_int64),
                ("ctx", ctypes.c_int64), ("eps", ctypes.c_float), ("rope_theta", ctypes.c_double), ("moe", Moe),
                ("embed", ctypes.c_void_p), ("attn_norm", ctypes.c_void_p), ("ffn_norm", ctypes.c_void_p),
                ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("wq", ctypes.c_void_p), ("wk", ctypes.c_void_p), ("wv", ctypes.c_void_p), ("wo", ctypes.c_void_p),
                ("router", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("router_f32", ctypes.c_void_p), ("sgate", ctypes.c_void_p),
                ("sup", ctypes.c_void_p), ("sdown", ctypes.c_void_p), ("lm_head", Q8), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, f32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        sig = {
            "ora_set_threads": ([i32], i32),
            "ora_host_cores": ([], i32),
            "ora_q8_weight": ([vp, vp, i64, i64, i64], dbl),
            "ora_q8_dequant": ([vp, vp, i64, i64, vp], None),
            "ora_gemv_f32act": ([vp, vp, i64, i64, vp, vp], None),
            "ora_quantize": ([vp, i64, vp, vp], None),
            "ora_blockdots": ([vp, i64, i64, vp, vp], None),
            "ora_gemv_int8act": ([vp, vp, i64, i64, vp, vp, vp], None),
            "ora_gemv": ([i32, vp, vp, i64, i64, vp, vp], None),
            "ora_quantize2": ([vp, i64, vp, vp, vp], None),
            "ora_gemv_int8act2": ([vp, vp, i64, i64, vp, vp, vp, vp], None),
            "ora_add_rmsnorm": ([vp, vp, vp, i64, i64, f32, vp, vp], None),
            "ora_softmax": ([vp, i64, vp], None),
            "ora_topk": ([vp, i64, i32, vp], None),
            "ora_route": ([vp, i64, i32, vp, vp], None),
            "ora_silu": ([dbl], dbl),
            "ora_moe_row": ([i32, ctypes.POINTER(Moe), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp], None),
            "ora_gemv_f32w": ([vp, i64, i64, vp, vp], None),
            "ora_group": ([vp, i64, i32, i64, vp, vp, vp], None),
            "ora_rmsnorm_head": ([vp, vp, i64, f32, vp], None),
            "ora_rope": ([vp, i64, i64, dbl], None),
            "ora_attention": ([vp, vp, vp, i64, i64, vp], None),
            "ora_argmax": ([vp, i64], i64),
            "ora_decode_step": ([i32, ctypes.POINTER(Model), i64, i64, vp], i64),
            "ora_decode_layers": ([i32, ctypes.POINTER(Model), i64, i64, i64, vp], None),
            "ora_decode_layer": ([i32, ctypes.POINTER(Model), i64, i64, vp, vp], None),
            "ora_probe_arm": ([i32, vp, vp, vp, i32], None),
            "ora_decode_final": ([i32, ctypes.POINTER(Model), vp, vp], i64),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def set_threads(n: int) -> int:
    """Threads the oracle uses from now on (1 by default; the results do not depend on it); returns the count set."""
    return int(lib().ora_set_threads(int(n)))


def host_cores() -> int:
    return int(lib().ora_host_cores())


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---- Q8_0 projections ----------------------------------------------------------------------------------------------

def dequant(q, s):
    q, pq = _c(q, np.int8)
    s, ps = _c(s, np.float32)
    n, k = q.shape
    w = np.empty((n, k), np.float64)
    lib().ora_q8_dequant(pq, ps, n, k, w.ctypes.data)
    return w


def weight(q, s, o, t):
    q, pq = _c(q, np.int8)
    s, ps = _c(s, np.float32)
    return lib().ora_q8_weight(pq, ps, q.shape[1], o, t)


def quantize(x):
    """One int8 word per value plus an f32 scale per 32-value block (x's last axis a multiple of 32)."""
    x, px = _c(x, np.float32)
    xq = np.empty(x.shape, np.int8)
    xs = np.empty(x.shape[:-1] + (x.shape[-1] // QBLOCK,), np.float32)
    lib().ora_quantize(px, x.size, xq.ctypes.data, xs.ctypes.data)
    return xq, xs


def quantize2(x):
    """Two int8 words per value (high, low in 128ths of the scale) plus an f32 scale per 32-value block."""
    x, px = _c(x, np.float32)
    hi = np.empty(x.shape, np.int8)
    lo = np.empty(x.shape, np.int8)
    xs = np.empty(x.shape[:-1] + (x.shape[-1] // QBLOCK,), np.float32)
    lib().ora_quantize2(px, x.size, hi.ctypes.data, lo.ctypes.data, xs.ctypes.data)
    return hi, lo, xs


def gemv_int8act2(q, s, hi, lo, xs):
    q, pq = _c(q, np.int8)
    s, ps = _c(s, np.float32)
    hi, ph = _c(hi, np.int8)
    lo, pl = _c(lo, np.int8)
    xs, pxs = _c(xs, np.float32)
    n, k = q.shape
    y = np.empty(n, np.float64)
    lib().ora_gemv_int8act2(pq, ps, n, k, ph, pl, pxs, y.ctypes.data)
    return y


def blockdots(q, xq):
    q, pq = _c(q, np.int8)
    xq, px = _c(xq, np.int8)
    n, k = q.shape
    D = np.empty((n, k // QBLOCK), np.int32)
    lib().ora_blockdots(pq, n, k, px, D.ctypes.data)
    return D


def gemv_f32act(q, s, x):
    q, pq = _c(q, np.int8)
    s, ps = _c(s, np.float32)
    x, px = _c(x, np.float32)
    n, k = q.shape
    y = np.empty(n, np.float64)
    lib().ora_gemv_f32act(pq, ps, n, k, px, y.ctypes.data)
    return y


def gemv_int8act(q, s, xq, xs):
    q, pq = _c(q, np.int8)
    s, ps = _c(s, np.float32)
    xq, pxq = _c(xq, np.int8)
    xs, pxs = _c(xs, np.float32)
    n, k = q.shape
    y = np.empty(n, np.float64)
    lib().ora_gemv_int8act(pq, ps, n, k, pxq, pxs, y.ctypes.data)
    return y


def gemv(mode, q, s, x):
    """y = W x for one activation row (mode 0: f32 activations / f64 sums; mode 1: one-word int8 activations; mode 2:
    two-word int8 activations)."""
    q, pq = _c(q, np.int8)
    s, ps = _c(s, np.float32)
    x, px = _c(x, np.float32)
    n, k = q.shape
    y = np.empty(n, np.float64)
    lib().ora_gemv(int(mode), pq, ps, n, k, px, y.ctypes.data)
    return y


# ---- add + RMSNorm --------------------------------------------------------------------------------------------------

def add_rmsnorm(a, b, w, eps):
    """Returns (s f32 [rows, d], y f64 [rows, d]); b may be None (a plain RMSNorm of a)."""
    a, pa = _c(a, np.float32)
    if a.ndim == 1:
        a = a[None]
    rows, d = a.shape
    pb = None
    if b is not None:
        b, pb = _c(np.reshape(b, (rows, d)), np.float32)
    w, pw = _c(w, np.float32)
    s = np.empty((rows, d), np.float32)
    y = np.empty((rows, d), np.float64)
    lib().ora_add_rmsnorm(pa, pb, pw, rows, d, float(eps), s.ctypes.data, y.ctypes.data)
    return s, y


# ---- router and mixture ---------------------------------------------------------------------------------------------

def softmax(l):
    l, pl = _c(l, np.float64)
    p = np.empty_like(l)
    lib().ora_softmax(pl, l.size, p.ctypes.data)
    return p


def topk(p, k):
    p, pp = _c(p, np.float64)
    ids = np.empty(k, np.int32)
    lib().ora_topk(pp, p.size, k, ids.ctypes.data)
    return ids


def route(logits, k):
    logits, pl = _c(logits, np.float64)
    ids = np.empty(k, np.int32)
    g = np.empty(k, np.float64)
    lib().ora_route(pl, logits.size, k, ids.ctypes.data, g.ctypes.data)
    return ids, g


def silu(z):
    return lib().ora_silu(float(z))


class MoeWeights:
    """Host arrays of one mixture: router [E,d], stacked gate/up [E*dff,d], stacked down [E*d,dff] (Q8_0 each);
    optionally a router of f32 values [E,d] used in place of the Q8_0 router, and a shared expert (gate/up [sdff,d],
    down [d,sdff], Q8_0)."""

    def __init__(self, d, dff, experts, k, router, gate, up, down, router_f32=None, shared=None):
        self.d, self.dff, self.experts, self.k = d, dff, experts, k
        self.arrays = [np.ascontiguousarray(a[0], np.int8) for a in (router, gate, up, down)]
        self.scales = [np.ascontiguousarray(a[1], np.float32) for a in (router, gate, up, down)]
        self.router_f32 = None if router_f32 is None else np.ascontiguousarray(router_f32, np.float32)
        self.shared = None
        self.sdff = 0
        if shared is not None:
            self.shared = [(np.ascontiguousarray(q, np.int8), np.ascontiguousarray(s, np.float32))
                           for q, s in (shared["gate"], shared["up"], shared["down"])]
            self.sdff = self.shared[0][0].shape[0]

    def struct(self):
        q8 = [Q8(q.ctypes.data, s.ctypes.data) for q, s in zip(self.arrays, self.scales)]
        sh = [Q8(q.ctypes.data, s.ctypes.data) for q, s in self.shared] if self.shared else [Q8(), Q8(), Q8()]
        rf = None if self.router_f32 is None else self.router_f32.ctypes.data
        return Moe(self.d, self.dff, self.experts, self.k, *q8, rf, self.sdff, *sh)


PROBE_MOE_INPUT, PROBE_ATTN_OUT = 0, 1  # the probe's sites (oracle.h)


def _arm_probe(site, n, probe, flips):
    """Arms the rounding-boundary probe for the site's next activation row (see oracle.h, ora_probe_arm); returns the
    margins array it fills (0.5 wherever no one-word quantization of the row records one)."""
    margins = np.full(n, 0.5) if probe else None
    idx = np.array([int(i) for i, _ in flips] or [0], np.int64)
    dl = np.array([int(v) for _, v in flips] or [0], np.int32)
    lib().ora_probe_arm(int(site), None if margins is None else margins.ctypes.data, idx.ctypes.data, dl.ctypes.data,
                        len(flips))
    return margins


def moe_row_probed(mode, w: MoeWeights, x, flips=()):
    """One mixture row with the rounding-boundary probe (test support): returns (the row's outputs as moe_rows gives
    them for one row, the input's margins: per value the signed distance of x/d from the nearest rounding boundary
    in steps).  flips: (index, delta) pairs added to the input's one-word words before every product reads them."""
    x = np.ascontiguousarray(np.reshape(x, (1, w.d)), np.float32)
    margins = _arm_probe(PROBE_MOE_INPUT, w.d, True, flips)
    out = moe_rows(mode, w, x)
    return {k: v[0] for k, v in out.items()}, margins


def moe_rows(mode, w: MoeWeights, x, residual=None):
    """The mixture over each row of x [R, d]; returns dict of logits, ids, gates, hidden, expert_out, y."""
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    R = x.shape[0]
    st = w.struct()
    out = {
        "logits": np.empty((R, w.experts)), "ids": np.empty((R, w.k), np.int32), "gates": np.empty((R, w.k)),
        "hidden": np.empty((R, w.k, w.dff)), "expert_out": np.empty((R, w.k, w.d)), "y": np.empty((R, w.d)),
        "shared_hidden": np.empty((R, max(w.sdff, 1))), "shared_out": np.empty((R, w.d)),
    }
    res = None if residual is None else np.ascontiguousarray(np.reshape(residual, (R, w.d)), np.float32)
    for r in range(R):
        lib().ora_moe_row(int(mode), ctypes.byref(st), x[r].ctypes.data,
                          None if res is None else res[r].ctypes.data,
                          out["logits"][r].ctypes.data, out["ids"][r].ctypes.data, out["gates"][r].ctypes.data,
                          out["hidden"][r].ctypes.data, out["expert_out"][r].ctypes.data, out["y"][r].ctypes.data,
                          out["shared_hidden"][r].ctypes.data, out["shared_out"][r].ctypes.data)
    if not w.sdff:
        del out["shared_hidden"], out["shared_out"]
    return out


def gemv_f32w(w, x):
    """y = W x for a matrix of f32 values (an f32 router), f64 sums."""
    w, pw = _c(w, np.float32)
    x, px = _c(x, np.float32)
    n, k = w.shape
    y = np.empty(n, np.float64)
    lib().ora_gemv_f32w(pw, n, k, px, y.ctypes.data)
    return y


def group(ids, experts):
    ids, pi = _c(ids, np.int32)
    rows, k = ids.shape
    counts = np.empty(experts, np.int32)
    offsets = np.empty(experts + 1, np.int32)
    lists = np.empty(rows * k, np.int32)
    lib().ora_group(pi, rows, k, experts, counts.ctypes.data, offsets.ctypes.data, lists.ctypes.data)
    return counts, offsets, lists


# ---- decode-step pieces ---------------------------------------------------------------------------------------------

def rmsnorm_head(x, w, eps):
    x, px = _c(x, np.float64)
    w, pw = _c(w, np.float32)
    y = np.empty_like(x)
    lib().ora_rmsnorm_head(px, pw, x.size, float(eps), y.ctypes.data)
    return y


def rope(x, pos, theta):
    x = np.array(x, dtype=np.float64, copy=True)
    lib().ora_rope(x.ctypes.data, x.size, int(pos), float(theta))
    return x


def attention(q, kc, vc):
    q, pq = _c(q, np.float64)
    kc, pk = _c(kc, np.float32)
    vc, pv = _c(vc, np.float32)
    length, hd = kc.shape
    out = np.empty(hd, np.float64)
    lib().ora_attention(pq, pk, pv, length, hd, out.ctypes.data)
    return out


def argmax(x):
    x, px = _c(x, np.float64)
    return int(lib().ora_argmax(px, x.size))


class ModelArrays:
    """Host arrays of a whole model (per-layer lists); keeps every array alive while the C struct points at it."""

    def __init__(self, cfg, embed, attn_norm, ffn_norm, q_norm, k_norm, final_norm, wq, wk, wv, wo, router, gate, up,
                 down, lm_head, k_cache, v_cache, router_f32=None, shared_gate=None, shared_up=None,
                 shared_down=None):
        self.cfg = cfg
        keep = []

        def arr(a, dt):
            a = np.ascontiguousarray(a, dt)
            keep.append(a)
            return a

        def ptrs(lst, dt):
            arrs = [arr(a, dt) for a in lst]
            p = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
            keep.append(p)
            return ctypes.cast(p, ctypes.c_void_p).value, arrs

        def q8s(lst):
            items = []
            for q, s in lst:
                q = arr(q, np.int8)
                s = arr(s, np.float32)
                items.append(Q8(q.ctypes.data, s.ctypes.data))
            a = (Q8 * len(items))(*items)
            keep.append(a)
            return ctypes.cast(a, ctypes.c_void_p).value

        L = cfg["layers"]
        self.embed = arr(embed, np.float32)
        p_attn, _ = ptrs(attn_norm, np.float32)
        p_ffn, _ = ptrs(ffn_norm, np.float32)
        p_qn, _ = ptrs(q_norm, np.float32)
        p_kn, _ = ptrs(k_norm, np.float32)
        self.final_norm = arr(final_norm, np.float32)
        p_kc, self.k_cache = ptrs(k_cache, np.float32)
        p_vc, self.v_cache = ptrs(v_cache, np.float32)
        lq, ls = arr(lm_head[0], np.int8), arr(lm_head[1], np.float32)
        sdff = shared_gate[0][0].shape[0] if shared_gate is not None else 0
        moe = Moe(cfg["d"], cfg["dff"], cfg["experts"], cfg["k"], Q8(), Q8(), Q8(), Q8(), None, sdff, Q8(), Q8(),
                  Q8())
        p_rf = ptrs(router_f32, np.float32)[0] if router_f32 is not None else None
        self.struct = Model(L, cfg["d"], cfg["heads"], cfg["kv_heads"], cfg["hd"], cfg["vocab"], cfg["ctx"],
                            cfg["eps"], cfg["rope_theta"], moe, self.embed.ctypes.data, p_attn, p_ffn, p_qn, p_kn,
                            self.final_norm.ctypes.data, q8s(wq), q8s(wk), q8s(wv), q8s(wo), q8s(router), q8s(gate),
                            q8s(up), q8s(down), p_rf,
                            q8s(shared_gate) if sdff else None, q8s(shared_up) if sdff else None,
                            q8s(shared_down) if sdff else None,
                            Q8(lq.ctypes.data, ls.ctypes.data), p_kc, p_vc)
        self._keep = keep


def decode_step(mode, model: ModelArrays, tok, pos):
    """One token at ``pos``: updates the model's host caches in place; returns (next token, logits f64)."""
    logits = np.empty(model.cfg["vocab"], np.float64)
    nxt = lib().ora_decode_step(int(mode), ctypes.byref(model.struct), int(tok), int(pos), logits.ctypes.data)
    return int(nxt), logits


def decode_layers(mode, model: ModelArrays, tok, pos, layers):
    out = np.empty(model.cfg["d"], np.float64)
    lib().ora_decode_layers(int(mode), ctypes.byref(model.struct), int(tok), int(pos), int(layers), out.ctypes.data)
    return out


def decode_layer(mode, model: ModelArrays, l, pos, h, probe=False, flips=(), site=PROBE_MOE_INPUT):
    """Layer ``l`` alone from the residual stream ``h`` (f32 [d]) entering it; writes the layer's key/value rows at
    ``pos`` into the model's host caches.  Returns (the stream leaving the layer as f32, the router's logits f64), and
    with ``probe`` also the rounding margins (f64, see moe_row_probed) of the probe site's row: the mixture input
    (PROBE_MOE_INPUT, [d]) or the attention output the O projection reads (PROBE_ATTN_OUT, [heads * hd]); ``flips``
    adds (index, delta) pairs to that row's one-word words."""
    h = np.array(h, dtype=np.float32, copy=True)
    rl = np.empty(model.cfg["experts"], np.float64)
    n = model.cfg["d"] if site == PROBE_MOE_INPUT else model.cfg["heads"] * model.cfg["hd"]
    margins = _arm_probe(site, n, probe, flips) if (probe or flips) else None
    lib().ora_decode_layer(int(mode), ctypes.byref(model.struct), int(l), int(pos), h.ctypes.data, rl.ctypes.data)
    return (h, rl, margins) if probe else (h, rl)


def decode_final(mode, model: ModelArrays, h):
    """The final norm, LM head and greedy token from the residual stream ``h`` leaving the last layer."""
    h = np.ascontiguousarray(h, np.float32)
    logits = np.empty(model.cfg["vocab"], np.float64)
    nxt = lib().ora_decode_final(int(mode), ctypes.byref(model.struct), h.ctypes.data, logits.ctypes.data)
    return int(nxt), logits
