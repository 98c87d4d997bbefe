"""Seeded synthetic inputs, shared by the tests and the benchmark.

The draws are defined in ``synth.c`` (counter-based SplitMix64, Box-Muller normals).  Nothing here computes any part of
the method: the oracle and the CUDA path both receive the same arrays from these functions.

Tensor ids: a Q8_0 matrix with id ``t`` takes its int8 quants from stream ``2*t`` and its f32 block scales from stream
``2*t + 1``; every other tensor takes its own id directly.  Callers keep ids distinct per tensor and per layer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None

THREADS = max(1, min(32, os.cpu_count() or 1))


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` with the host C compiler (portable C, no architecture flags)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", src, "-o", tmp,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.synth_u64.argtypes = [u64, u64, u64]
        L.synth_u64.restype = u64
        L.synth_normal.argtypes = [u64, u64, u64]
        L.synth_normal.restype = dbl
        L.synth_fill_i8.argtypes = [u64, u64, u64, u64, vp, i32]
        L.synth_fill_i8.restype = None
        L.synth_fill_f32.argtypes = [u64, u64, u64, u64, dbl, dbl, i32, vp, i32]
        L.synth_fill_f32.restype = None
        _lib = L
    return _lib


def fill_i8_ptr(ptr: int, n: int, seed: int, tensor: int, offset: int = 0) -> None:
    """Write n int8 weights of stream ``tensor`` (starting at element ``offset``) to host address ``ptr``."""
    lib().synth_fill_i8(seed, tensor, offset, n, ptr, THREADS)


def fill_f32_ptr(ptr: int, n: int, seed: int, tensor: int, mul: float = 1.0, add: float = 0.0, absval: bool = False,
                 offset: int = 0) -> None:
    """Write n f32 values ``add + mul*z`` (``|z|`` when absval) of stream ``tensor`` to host address ``ptr``."""
    lib().synth_fill_f32(seed, tensor, offset, n, mul, add, int(absval), ptr, THREADS)


def int8(shape, seed: int, tensor: int, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.int8)
    if out.size:
        fill_i8_ptr(out.ctypes.data, out.size, seed, tensor, offset)
    return out


def normal(shape, seed: int, tensor: int, mul: float = 1.0, add: float = 0.0, absval: bool = False,
           offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    if out.size:
        fill_f32_ptr(out.ctypes.data, out.size, seed, tensor, mul, add, absval, offset)
    return out


def q8_matrix(n: int, k: int, seed: int, tensor: int, scale_mul: float = 0.01, row0: int = 0):
    """Rows ``row0 .. row0+n`` of a Q8_0 matrix with ``k`` columns: quants U[-127,127], scales |N(0,1)|*scale_mul."""
    assert k % 32 == 0
    q = int8((n, k), seed, 2 * tensor, offset=row0 * k)
    s = normal((n, k // 32), seed, 2 * tensor + 1, mul=scale_mul, absval=True, offset=row0 * (k // 32))
    return q, s


def u64(seed: int, tensor: int, i: int) -> int:
    return int(lib().synth_u64(seed, tensor, i))
