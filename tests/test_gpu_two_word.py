"""GPU parity of the two-word activation mode (Q8_INT8ACT2) against the oracle, through the C ABI.

The two-word form (lane/mod.rs module docs: "a two-word ~14-bit int8 activation (the default)"; lane/arena.rs,
array_bytes / quant_parts) is the one-word word plus a low word in 128ths of the block's one scale.  Both words of a
quantizer fed identical f32 input are bit-exact, and so are both words' block dots; floating outputs are within the
int8-activation tolerance 2e-3 of the oracle's same mode (and in practice far inside it: the quantization is shared).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from synth import recipes

pytestmark = pytest.mark.gpu

TOL = 2e-3


def rel_err(gpu, ora):
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    scale = np.max(np.abs(ora))
    return float(np.max(np.abs(gpu - ora)) / (scale if scale > 0 else 1.0))


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def empty(shape, dtype):
    import torch
    return torch.empty(shape, dtype=dtype, device="cuda")


@pytest.fixture(scope="module")
def ws(q8):
    w = q8.Workspace(256 << 20)
    yield w
    w.close()


def _quantize2_gpu(q8, x):
    import torch
    rows, cols = x.shape
    q = empty((rows, cols), torch.int8)
    lo = empty((rows, cols), torch.int8)
    s = empty((rows, cols // 32), torch.float32)
    q8.q8_quantize(dev(x), q, s, lo=lo)
    return host(q), host(lo), host(s)


def test_quantize2_golden_block_and_random(q8):
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))["quantize2_hand"]
    x = synth.normal((9, 2048), 0, recipes.VEC + 110, mul=3.0)
    x[0, :32] = np.array(g["x"], np.float32)
    x[1, :32] = 0.0
    hi, lo, s = _quantize2_gpu(q8, x)
    assert hi[0, :32].tolist() == g["hi"] and lo[0, :32].tolist() == g["lo"]
    ohi, olo, os_ = oracle.quantize2(x)
    np.testing.assert_array_equal(hi, ohi)
    np.testing.assert_array_equal(lo, olo)
    np.testing.assert_array_equal(s, os_)


def test_quantize2_near_half_steps_bitexact(q8):
    # values on, or one ulp either side of, the points where either word's rounding turns: (k + 1/2) d for the high
    # word and (k + j/128 + 1/256) d for the low word, over scales down to the subnormal range
    rng = np.random.default_rng(11)
    nblk = 4096
    amax = (10.0 ** rng.uniform(-40, 20, nblk)).astype(np.float32)
    d = (amax / np.float32(127)).astype(np.float32)
    k = rng.integers(-126, 126, (nblk, 31)).astype(np.float64)
    j = rng.integers(-64, 64, (nblk, 31)).astype(np.float64)
    frac = np.where(rng.random((nblk, 31)) < 0.5, 0.5, j / 128 + 1 / 256)
    base = ((k + frac) * d[:, None].astype(np.float64)).astype(np.float32)
    nudge = rng.integers(-1, 2, (nblk, 31))
    vals = np.where(nudge < 0, np.nextafter(base, np.float32(-np.inf)),
                    np.where(nudge > 0, np.nextafter(base, np.float32(np.inf)), base)).astype(np.float32)
    vals = np.clip(vals, -amax[:, None], amax[:, None])
    x = np.concatenate([amax[:, None] * np.where(rng.random((nblk, 1)) < 0.5, 1, -1).astype(np.float32), vals], 1)
    x = x.astype(np.float32).reshape(1, nblk * 32)
    hi, lo, s = _quantize2_gpu(q8, x)
    ohi, olo, os_ = oracle.quantize2(x)
    np.testing.assert_array_equal(s, os_)
    np.testing.assert_array_equal(hi, ohi)
    np.testing.assert_array_equal(lo, olo)


@pytest.mark.parametrize("rows,d", [(1, 2048), (3, 4096), (64, 2048), (5, 96)])
def test_add_rmsnorm_two_word_epilogue(q8, rows, d):
    # the epilogue's words are the quantizer's of the kernel's own f32 output, bit for bit
    import torch
    a = synth.normal((rows, d), 1, recipes.VEC + 111)
    b = synth.normal((rows, d), 1, recipes.VEC + 112)
    w = synth.normal(d, 1, recipes.VEC + 113, mul=0.1, add=1.0)
    y = empty((rows, d), torch.float32)
    yq = empty((rows, d), torch.int8)
    yl = empty((rows, d), torch.int8)
    ys = empty((rows, d // 32), torch.float32)
    q8.add_rmsnorm_q8(dev(a), dev(b), dev(w), 1e-6, y_out=y, yq=yq, ys=ys, yl=yl)
    gy = host(y)
    _, y_ora = oracle.add_rmsnorm(a, b, w, 1e-6)
    assert rel_err(gy, y_ora) < 1e-6
    ohi, olo, os_ = oracle.quantize2(gy)
    np.testing.assert_array_equal(host(yq), ohi)
    np.testing.assert_array_equal(host(yl), olo)
    np.testing.assert_array_equal(host(ys), os_)


GEMV_SHAPES = [(1024, 1024, 1), (4096, 2048, 1), (512, 2048, 1), (2048, 4096, 1), (128, 2048, 1), (1000, 96, 1),
               (33, 768, 1), (77, 32, 3), (4096, 2048, 2), (7, 8192, 1), (300, 2048, 5)]


@pytest.mark.parametrize("n,k,R", GEMV_SHAPES)
def test_q8_gemv_two_words(q8, ws, n, k, R):
    import torch
    q, s = synth.q8_matrix(n, k, 1, 140 + n % 7)
    x = synth.normal((R, k), 1, recipes.VEC + 141)
    hi, lo, xs = oracle.quantize2(x)
    ref = np.stack([oracle.gemv_int8act2(q, s, hi[r], lo[r], xs[r]) for r in range(R)])
    y = empty((R, n), torch.float32)
    q8.q8_gemv(dev(q), dev(s), 2, y, xq=dev(hi), xs=dev(xs), xl=dev(lo), rows=R, ws=ws)
    err = rel_err(host(y), ref)
    assert err < TOL, err
    assert err < 1e-5, err  # both sides read the same words: only the f32 summation differs
    # the call quantizing x itself gives the same words, hence the same result
    y2 = empty((R, n), torch.float32)
    q8.q8_gemv(dev(q), dev(s), 2, y2, x=dev(x), rows=R, ws=ws)
    np.testing.assert_array_equal(host(y2), host(y))
    # and the two-word product is nearer the f32-activation product than the one-word one
    y0 = np.stack([oracle.gemv_f32act(q, s, x[r]) for r in range(R)])
    y1 = np.stack([oracle.gemv(1, q, s, x[r]) for r in range(R)])
    assert rel_err(host(y), y0) < rel_err(y1, y0)


@pytest.mark.parametrize("n,k,R", [(1024, 1024, 1), (513, 2048, 2), (64, 768, 1), (5, 4096, 1)])
def test_blockdots_both_words_bitexact(q8, ws, n, k, R):
    import torch
    q, s = synth.q8_matrix(n, k, 2, 150)
    x = synth.normal((R, k), 2, recipes.VEC + 151)
    hi, lo, xs = oracle.quantize2(x)
    dots = empty((2, R, n, k // 32), torch.int32)
    y = empty((R, n), torch.float32)
    q8.q8_gemv_blockdots(dev(q), dev(s), dev(hi), dev(xs), dots, y, rows=R, ws=ws, xl=dev(lo))
    D = host(dots)
    for r in range(R):
        np.testing.assert_array_equal(D[0, r], oracle.blockdots(q, hi[r]))
        np.testing.assert_array_equal(D[1, r], oracle.blockdots(q, lo[r]))
    assert rel_err(host(y), np.stack([oracle.gemv_int8act2(q, s, hi[r], lo[r], xs[r]) for r in range(R)])) < 1e-5
