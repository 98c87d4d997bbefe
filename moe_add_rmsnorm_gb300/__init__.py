"""Python binding of the q8moe C ABI (include/q8moe.h): argument marshalling only.

Every computation runs in the CUDA library ``libq8moe.so`` built in-tree for sm_103a (``build.build()``).  There is no
fallback: importing this package without the built library raises ImportError.  Tensors are PyTorch tensors used only
as device memory; the current PyTorch stream is used unless a stream is passed.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq8moe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run moe_add_rmsnorm_gb300.build.build() (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)

F32ACT_F64SUM = 0
INT8ACT = 1
INT8ACT2 = 2  # the two-word activation (high words, low words in 128ths of the block scale)
QBLOCK = 32

STATUS = {0: "Q8_OK", -1: "Q8_EINVAL", -2: "Q8_EUNSUPPORTED", -3: "Q8_ECUDA", -4: "Q8_ETIMEOUT", -5: "Q8_ENOSPACE"}


class Q8Error(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class q8_mat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class q8_act(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("lo", ctypes.c_void_p)]


class q8_shared_expert(ctypes.Structure):
    _fields_ = [("gate", q8_mat), ("up", q8_mat), ("down", q8_mat)]


class q8_moe_plan(ctypes.Structure):
    _fields_ = [("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p), ("lists", ctypes.c_void_p),
                ("active", ctypes.c_void_p)]


class q8_model_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("layers", "d", "heads", "kv_heads", "head_dim", "experts", "k", "dff",
                                                "vocab", "ctx")] + [
        ("eps", ctypes.c_float), ("rope_theta", ctypes.c_double), ("mode", ctypes.c_int),
        ("embed", ctypes.c_void_p), ("attn_norm", ctypes.c_void_p), ("ffn_norm", ctypes.c_void_p),
        ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
        ("wq", ctypes.c_void_p), ("wk", ctypes.c_void_p), ("wv", ctypes.c_void_p), ("wo", ctypes.c_void_p),
        ("router", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
        ("lm_head", q8_mat), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("tok", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("logits", ctypes.c_void_p),
        ("router_f32", ctypes.c_void_p), ("shared_gate", ctypes.c_void_p), ("shared_up", ctypes.c_void_p),
        ("shared_down", ctypes.c_void_p), ("shared_dff", ctypes.c_int64), ("batch", ctypes.c_int64)]


_vp, _i64, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_P = ctypes.POINTER
_SIGS = {
    "q8_workspace_create": [_sz, _P(_vp)],
    "q8_workspace_destroy": [_vp],
    "q8_workspace_bytes": [_vp],
    "q8_quantize": [_vp, _i64, _i64, _P(q8_act), _vp],
    "add_rmsnorm_q8": [_vp, _vp, _vp, _i64, _i64, _f32, _vp, _vp, _P(q8_act), _vp],
    "q8_gemv": [_P(q8_mat), _i32, _vp, _P(q8_act), _i64, _vp, _vp, _vp],
    "q8_gemv_blockdots": [_P(q8_mat), _P(q8_act), _i64, _vp, _vp, _vp, _vp],
    "q8_gemv_noalloc": [_P(q8_mat), _i32, _vp, _P(q8_act), _i64, _vp, _vp],
    "q8_set_tensor_core_rows": [_i32],
    "q8_set_grouped_tensor_core_rows": [_i32],
    "q8_set_tensor_core_attention": [_i32],
    "q8_set_persistent_decode": [_i32],
    "q8_set_streamed_batch_attention": [_i32],
    "q8_model_persistent": [_vp],
    "moe_route_topk": [_P(q8_mat), _i32, _vp, _P(q8_act), _i64, _i32, _vp, _vp, _vp, _P(q8_moe_plan), _vp, _vp],
    "moe_route_topk_f32": [_vp, _i64, _i64, _vp, _i64, _i32, _vp, _vp, _vp, _P(q8_moe_plan), _vp, _vp],
    "moe_gate_up": [_P(q8_mat), _P(q8_mat), _i64, _i32, _vp, _P(q8_act), _i64, _i32, _vp, _P(q8_moe_plan), _vp,
                    _P(q8_act), _P(q8_shared_expert), _vp, _vp],
    "moe_down_combine": [_P(q8_mat), _i64, _i32, _vp, _P(q8_act), _i64, _i32, _vp, _vp, _P(q8_moe_plan), _vp, _vp,
                         _vp, _P(q8_shared_expert), _vp, _vp],
    "q8_model_create": [_P(q8_model_desc), _P(_vp)],
    "q8_model_destroy": [_vp],
    "decode_step": [_vp, _vp],
    "decode_step_launches": [_vp, _vp],
    "decode_step_trace": [_vp, _vp, _vp],
    "prefill_chunk": [_vp, _vp, _i64, _vp, _vp],
    "prefill_chunk_trace": [_vp, _vp, _i64, _vp, _vp, _vp],
    "q8_model_check": [_vp, _vp],
    "q8_model_wait_selftest": [_vp, ctypes.c_uint, _vp],
    "q8_model_launches_per_step": [_vp],
    "q8_last_error": [],
}
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
lib.q8_workspace_destroy.restype = None
lib.q8_model_destroy.restype = None
lib.q8_workspace_bytes.restype = ctypes.c_size_t
lib.q8_last_error.restype = ctypes.c_char_p
lib.q8_model_launches_per_step.restype = ctypes.c_int64

EXPORTS = tuple(_SIGS)


def last_error() -> str:
    return lib.q8_last_error().decode()


def _check(code):
    if code != 0:
        raise Q8Error(code, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def mat(q, s) -> q8_mat:
    """A q8_mat over device tensors q int8 [rows, cols] and s f32 [rows, cols/32]."""
    return q8_mat(q.data_ptr(), s.data_ptr(), q.shape[0], q.shape[1])


def act(q, s, lo=None) -> q8_act:
    return q8_act(q.data_ptr(), s.data_ptr(), lo.data_ptr() if lo is not None else None)


def _actref(q, s, lo=None):
    return ctypes.byref(act(q, s, lo)) if q is not None else None


class Workspace:
    def __init__(self, nbytes: int = 0):
        h = ctypes.c_void_p()
        _check(lib.q8_workspace_create(nbytes, ctypes.byref(h)))
        self.handle = h

    @property
    def nbytes(self):
        return lib.q8_workspace_bytes(self.handle)

    def close(self):
        if self.handle:
            lib.q8_workspace_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q8_quantize(x, q, s, stream=None, lo=None):
    """One word per value, or with `lo` the two-word form."""
    rows = x.shape[0] if x.dim() > 1 else 1
    _check(lib.q8_quantize(_ptr(x), rows, x.shape[-1], _actref(q, s, lo), _stream(stream)))


def add_rmsnorm_q8(a, b, w, eps, sum_out=None, y_out=None, yq=None, ys=None, stream=None, yl=None):
    rows = a.shape[0] if a.dim() > 1 else 1
    qa = _actref(yq, ys, yl)
    _check(lib.add_rmsnorm_q8(_ptr(a), _ptr(b), _ptr(w), rows, a.shape[-1], float(eps), _ptr(sum_out), _ptr(y_out),
                              qa, _stream(stream)))


def q8_gemv(q, s, mode, y, x=None, xq=None, xs=None, rows=1, ws=None, stream=None, xl=None):
    W = mat(q, s)
    qa = _actref(xq, xs, xl)
    _check(lib.q8_gemv(ctypes.byref(W), int(mode), _ptr(x), qa, rows, _ptr(y), ws.handle if ws else None,
                       _stream(stream)))


def q8_gemv_noalloc(q, s, mode, y, x=None, xq=None, xs=None, rows=1, stream=None, xl=None):
    """q8_gemv without a workspace: scratch comes from the library's fixed per-device array (see q8moe.h)."""
    W = mat(q, s)
    qa = _actref(xq, xs, xl)
    _check(lib.q8_gemv_noalloc(ctypes.byref(W), int(mode), _ptr(x), qa, rows, _ptr(y), _stream(stream)))


def q8_gemv_blockdots(q, s, xq, xs, dots, y, rows=1, ws=None, stream=None, xl=None):
    """With xl (two words) dots is [2, rows, n, nb]: the words' dots, then the low words'."""
    W = mat(q, s)
    qa = act(xq, xs, xl)
    _check(lib.q8_gemv_blockdots(ctypes.byref(W), ctypes.byref(qa), rows, _ptr(dots), _ptr(y),
                                 ws.handle if ws else None, _stream(stream)))


def set_tensor_core_rows(rows: int):
    """The fewest int8 activation rows (16..64) a dense projection takes to the tensor cores; 0: never; -1 (the
    default): one matrix of at least 2048 x 2048 from 32 rows on."""
    _check(lib.q8_set_tensor_core_rows(int(rows)))


def set_grouped_tensor_core_rows(rows: int):
    """The fewest rows (16..64) an int8 expert group of a chunk needs to take the tensor cores; 0: never (default 32)."""
    _check(lib.q8_set_grouped_tensor_core_rows(int(rows)))


def set_tensor_core_attention(on: bool):
    """Prefill chunks' causal attention on the tensor cores (default) or, with False, the CUDA cores."""
    _check(lib.q8_set_tensor_core_attention(1 if on else 0))


def set_persistent_decode(on: bool):
    """One-sequence int8 decode steps as one persistent launch, or (False, the default) six launches a layer."""
    _check(lib.q8_set_persistent_decode(1 if on else 0))


def set_streamed_batch_attention(min_batch: int):
    """Batch decode steps of at least min_batch sequences (default 8) attend in the streamed form; 0: never."""
    _check(lib.q8_set_streamed_batch_attention(int(min_batch)))


def plan_struct(counts, offsets, lists, active):
    return q8_moe_plan(counts.data_ptr(), offsets.data_ptr(), lists.data_ptr(), active.data_ptr())


def moe_route_topk(rq, rs, mode, k, ids, gates, x=None, xq=None, xs=None, rows=1, logits=None, plan=None, ws=None,
                   stream=None, xl=None):
    R = mat(rq, rs)
    qa = _actref(xq, xs, xl)
    pl = ctypes.byref(plan) if plan is not None else None
    _check(lib.moe_route_topk(ctypes.byref(R), int(mode), _ptr(x), qa, rows, int(k), _ptr(ids), _ptr(gates),
                              _ptr(logits), pl, ws.handle if ws else None, _stream(stream)))


def shared_expert(gate, up, down) -> q8_shared_expert:
    """A shared expert over (q, s) device tensor pairs: gate and up [sdff, d], down [d, sdff]."""
    return q8_shared_expert(mat(*gate), mat(*up), mat(*down))


def moe_route_topk_f32(router, k, ids, gates, x, rows=1, logits=None, plan=None, ws=None, stream=None):
    """The router of f32 values (device f32 [E, d]) over the f32 rows x, then top-k as moe_route_topk."""
    pl = ctypes.byref(plan) if plan is not None else None
    _check(lib.moe_route_topk_f32(_ptr(router), router.shape[0], router.shape[1], _ptr(x), rows, int(k), _ptr(ids),
                                  _ptr(gates), _ptr(logits), pl, ws.handle if ws else None, _stream(stream)))


def moe_gate_up(gq, gs, uq, us, dff, mode, k, ids, h, x=None, xq=None, xs=None, hq=None, hs=None, rows=1, plan=None,
                ws=None, stream=None, xl=None, hl=None, shared=None):
    G, U = mat(gq, gs), mat(uq, us)
    qa = _actref(xq, xs, xl)
    ha = _actref(hq, hs, hl)
    pl = ctypes.byref(plan) if plan is not None else None
    sh = ctypes.byref(shared) if shared is not None else None
    _check(lib.moe_gate_up(ctypes.byref(G), ctypes.byref(U), int(dff), int(mode), _ptr(x), qa, rows, int(k),
                           _ptr(ids), pl, _ptr(h), ha, sh, ws.handle if ws else None, _stream(stream)))


def moe_down_combine(dq, ds, d, mode, k, ids, gates, y, h=None, hq=None, hs=None, rows=1, plan=None, residual=None,
                     expert_out=None, ws=None, stream=None, hl=None, shared=None):
    Dm = mat(dq, ds)
    ha = _actref(hq, hs, hl)
    pl = ctypes.byref(plan) if plan is not None else None
    sh = ctypes.byref(shared) if shared is not None else None
    _check(lib.moe_down_combine(ctypes.byref(Dm), int(d), int(mode), _ptr(h), ha, rows, int(k), _ptr(ids),
                                _ptr(gates), pl, _ptr(residual), _ptr(y), _ptr(expert_out), sh,
                                ws.handle if ws else None, _stream(stream)))


class Model:
    """A decode model over caller-owned device tensors (see q8_model_desc in include/q8moe.h)."""

    def __init__(self, cfg: dict, t: dict, mode: int, tok, pos, logits=None):
        L = cfg["layers"]
        self._keep = []

        def ptr_array(tensors):
            arr = (ctypes.c_void_p * L)(*[x.data_ptr() for x in tensors])
            self._keep.append(arr)
            return ctypes.cast(arr, ctypes.c_void_p)

        def mat_array(pairs):
            arr = (q8_mat * L)(*[mat(q, s) for q, s in pairs])
            self._keep.append(arr)
            return ctypes.cast(arr, ctypes.c_void_p)

        d = q8_model_desc()
        for key in ("layers", "d", "heads", "kv_heads", "experts", "k", "dff", "vocab", "ctx"):
            setattr(d, key, int(cfg[key]))
        d.head_dim = int(cfg["hd"])
        d.batch = int(cfg.get("batch", 0))  # the batch form: tok, pos [batch], logits [batch, vocab], caches per layer
                                            # [batch, kv, ctx, hd]
        d.eps = float(cfg["eps"])
        d.rope_theta = float(cfg["rope_theta"])
        d.mode = int(mode)
        d.embed = t["embed"].data_ptr()
        d.attn_norm = ptr_array(t["attn_norm"])
        d.ffn_norm = ptr_array(t["ffn_norm"])
        d.q_norm = ptr_array(t["q_norm"])
        d.k_norm = ptr_array(t["k_norm"])
        d.final_norm = t["final_norm"].data_ptr()
        for key in ("wq", "wk", "wv", "wo", "router", "gate", "up", "down"):
            setattr(d, key, mat_array(t[key]))
        d.lm_head = mat(*t["lm_head"])
        d.k_cache = ptr_array(t["k_cache"])
        d.v_cache = ptr_array(t["v_cache"])
        d.tok = tok.data_ptr()
        d.pos = pos.data_ptr()
        d.logits = logits.data_ptr() if logits is not None else None
        if t.get("router_f32") is not None:  # optional: routers of f32 values
            d.router_f32 = ptr_array(t["router_f32"])
        if t.get("shared_gate") is not None:  # optional: a shared expert per layer
            for key in ("shared_gate", "shared_up", "shared_down"):
                setattr(d, key, mat_array(t[key]))
            d.shared_dff = int(t["shared_gate"][0][0].shape[0])
        h = ctypes.c_void_p()
        _check(lib.q8_model_create(ctypes.byref(d), ctypes.byref(h)))
        self.handle = h
        self.tensors = t

    def step(self, stream=None):
        _check(lib.decode_step(self.handle, _stream(stream)))

    def step_launches(self, stream=None):
        _check(lib.decode_step_launches(self.handle, _stream(stream)))

    def step_trace(self, hidden, stream=None):
        """Plain-launch step that also copies the residual stream entering layer 0 and leaving every layer into
        hidden (device f32 [layers + 1, d])."""
        _check(lib.decode_step_trace(self.handle, hidden.data_ptr(), _stream(stream)))

    def prefill(self, tokens, ws, stream=None):
        """tokens: device int32 [rows]; the chunk through every layer (plain launches), last row's token into tok."""
        _check(lib.prefill_chunk(self.handle, tokens.data_ptr(), tokens.numel(), ws.handle, _stream(stream)))

    def prefill_trace(self, tokens, ws, hidden, stream=None):
        """prefill() that also copies the residual rows entering every layer and the final ones into hidden (device
        f32 [layers + 1, rows, d])."""
        _check(lib.prefill_chunk_trace(self.handle, tokens.data_ptr(), tokens.numel(), ws.handle, hidden.data_ptr(),
                                       _stream(stream)))

    def check(self, stream=None):
        _check(lib.q8_model_check(self.handle, _stream(stream)))

    def wait_selftest(self, polls, stream=None):
        """A bounded wait on a barrier nothing arrives on; the next check() raises Q8_ETIMEOUT."""
        _check(lib.q8_model_wait_selftest(self.handle, int(polls), _stream(stream)))

    def launches_per_step(self):
        """Kernels one step launches (the captured graph's kernel nodes; 0 before the first step)."""
        return int(lib.q8_model_launches_per_step(self.handle))

    def persistent(self):
        """Whether the model's decode steps run their layers as one persistent launch."""
        return bool(lib.q8_model_persistent(self.handle))

    def close(self):
        if self.handle:
            lib.q8_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
