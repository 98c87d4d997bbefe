"""GPU parity of every kernel against the CPU oracle, through the C ABI.

Tolerances (from the spec contract): per-block int32 dots, int8 words of a quantizer fed identical f32 input,
expert ids and the chunk grouping are bit-exact; floating outputs are within max|gpu - oracle| / max|oracle| of 1e-4 in
the f32-activation / f64-sum mode and 2e-3 in the int8-activation mode (each compared with the oracle's same mode).
"""
import numpy as np
import pytest

import oracle
import synth
from synth import recipes

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 2e-3, 2: 2e-3}  # mode 2 (two words) is an int8-activation mode


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


# ---- quantizer and add + RMSNorm ------------------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 2048), (7, 96), (64, 768)])
def test_quantize_bitexact(q8, rows, cols):
    import torch
    x = synth.normal((rows, cols), 0, recipes.VEC + 10, mul=3.0)
    x[0, :32] = np.array(oracle_golden_ties(), np.float32)
    if rows > 1:
        x[1, :32] = 0.0
    q = empty((rows, cols), torch.int8)
    s = empty((rows, cols // 32), torch.float32)
    q8.q8_quantize(dev(x), q, s)
    oq, os_ = oracle.quantize(x)
    np.testing.assert_array_equal(host(q), oq)
    np.testing.assert_array_equal(host(s), os_)


def test_quantize_near_half_integers_bitexact(q8):
    # blocks whose values sit exactly on, or one ulp either side of, (k + 1/2) * d for the block's own d = amax / 127:
    # the quotients the round-half-away rule turns on
    import torch
    rng = np.random.default_rng(7)
    nblk = 4096
    amax = (10.0 ** rng.uniform(-44, 20, nblk)).astype(np.float32)  # down to subnormal scales
    d = (amax / np.float32(127)).astype(np.float32)
    k = rng.integers(-127, 127, (nblk, 31)).astype(np.float32)
    base = ((k + np.float32(0.5)) * d[:, None]).astype(np.float32)
    nudge = rng.integers(-1, 2, (nblk, 31))
    vals = np.where(nudge < 0, np.nextafter(base, np.float32(-np.inf)),
                    np.where(nudge > 0, np.nextafter(base, np.float32(np.inf)), base)).astype(np.float32)
    vals = np.clip(vals, -amax[:, None], amax[:, None])
    x = np.concatenate([amax[:, None] * np.where(rng.random((nblk, 1)) < 0.5, 1, -1).astype(np.float32), vals], 1)
    x = x.astype(np.float32).reshape(1, nblk * 32)
    q = empty((1, nblk * 32), torch.int8)
    sc = empty((1, nblk), torch.float32)
    q8.q8_quantize(dev(x), q, sc)
    oq, os_ = oracle.quantize(x)
    np.testing.assert_array_equal(host(sc), os_)
    np.testing.assert_array_equal(host(q), oq)


def oracle_golden_ties():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))
    return g["quantize_ties"]["x"]


@pytest.mark.parametrize("rows,d,with_b", [(1, 2048, True), (1, 2048, False), (3, 4096, True), (64, 2048, True),
                                           (5, 96, True), (2, 8192, True), (1, 4000, False)])
def test_add_rmsnorm_q8(q8, rows, d, with_b):
    import torch
    a = synth.normal((rows, d), 0, recipes.VEC + 20)
    b = synth.normal((rows, d), 0, recipes.VEC + 21) if with_b else None
    w = synth.normal(d, 0, recipes.VEC + 22, mul=0.1, add=1.0)
    eps = 1e-6
    s_ora, y_ora = oracle.add_rmsnorm(a, b, w, eps)
    y32_ora = y_ora.astype(np.float32)
    s_out = empty((rows, d), torch.float32)
    y_out = empty((rows, d), torch.float32)
    quant = d % 32 == 0
    yq = empty((rows, d), torch.int8) if quant else None
    ys = empty((rows, d // 32), torch.float32) if quant else None
    q8.add_rmsnorm_q8(dev(a), dev(b) if b is not None else None, dev(w), eps, sum_out=s_out, y_out=y_out, yq=yq, ys=ys)
    np.testing.assert_array_equal(host(s_out), s_ora)          # one f32 add, bit-exact
    y = host(y_out)
    assert rel_err(y, y_ora) < 1e-6
    # the norm runs in f64 and rounds once: the f32 results equal the oracle's rounded f64 value but for values
    # within an f64 rounding of an f32 midpoint (at most one ulp, and rare)
    ulp = np.abs(y.view(np.int32).astype(np.int64) - y32_ora.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1 and (ulp > 0).mean() < 1e-4
    if quant:
        oq, os_ = oracle.quantize(y32_ora)
        gq, gs = host(yq), host(ys)
        same_block = (ulp.reshape(rows, d // 32, 32).max(-1) == 0)
        np.testing.assert_array_equal(gs[same_block], os_[same_block])
        np.testing.assert_array_equal(gq.reshape(rows, d // 32, 32)[same_block],
                                      oq.reshape(rows, d // 32, 32)[same_block])


def test_add_rmsnorm_in_place_residual(q8):
    a = synth.normal((2, 2048), 1, recipes.VEC + 23)
    b = synth.normal((2, 2048), 1, recipes.VEC + 24)
    w = synth.normal(2048, 1, recipes.VEC + 25, mul=0.1, add=1.0)
    s_ora, y_ora = oracle.add_rmsnorm(a, b, w, 1e-6)
    ta = dev(a)
    y = empty((2, 2048), __import__("torch").float32)
    q8.add_rmsnorm_q8(ta, dev(b), dev(w), 1e-6, sum_out=ta, y_out=y)
    np.testing.assert_array_equal(host(ta), s_ora)
    assert rel_err(host(y), y_ora) < 1e-6


# ---- the Q8_0 projection -------------------------------------------------------------------------------------------

GEMV_SHAPES = [(1024, 1024, 1), (4096, 2048, 1), (512, 2048, 1), (2048, 4096, 1), (128, 2048, 1), (1000, 96, 1),
               (33, 768, 1), (2048, 768, 1), (77, 32, 3), (4096, 2048, 2), (7, 8192, 1), (300, 2048, 5)]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("n,k,R", GEMV_SHAPES)
def test_q8_gemv(q8, ws, mode, n, k, R):
    import torch
    q, s = synth.q8_matrix(n, k, 0, 40 + n % 7)
    x = synth.normal((R, k), 0, recipes.VEC + 41)
    y = empty((R, n), torch.float32)
    if mode == 0:
        ref = np.stack([oracle.gemv_f32act(q, s, x[r]) for r in range(R)])
        q8.q8_gemv(dev(q), dev(s), 0, y, x=dev(x), rows=R, ws=ws)
    else:
        xq, xs = oracle.quantize(x)
        ref = np.stack([oracle.gemv_int8act(q, s, xq[r], xs[r]) for r in range(R)])
        q8.q8_gemv(dev(q), dev(s), 1, y, xq=dev(xq), xs=dev(xs), rows=R, ws=ws)
    err = rel_err(host(y), ref)
    assert err < TOL[mode], err
    if mode == 1:
        # the kernel's own quantisation of x (xq omitted) gives the same words, hence the same result
        y2 = empty((R, n), torch.float32)
        q8.q8_gemv(dev(q), dev(s), 1, y2, x=dev(x), rows=R, ws=ws)
        np.testing.assert_array_equal(host(y2), host(y))


@pytest.mark.parametrize("n,k,R", [(1024, 1024, 1), (513, 2048, 2), (64, 768, 1), (5, 4096, 1)])
def test_blockdots_bitexact(q8, ws, n, k, R):
    import torch
    q, s = synth.q8_matrix(n, k, 2, 50)
    x = synth.normal((R, k), 2, recipes.VEC + 51)
    xq, xs = oracle.quantize(x)
    dots = empty((R, n, k // 32), torch.int32)
    y = empty((R, n), torch.float32)
    q8.q8_gemv_blockdots(dev(q), dev(s), dev(xq), dev(xs), dots, y, rows=R, ws=ws)
    D = host(dots)
    for r in range(R):
        np.testing.assert_array_equal(D[r], oracle.blockdots(q, xq[r]))


def test_gemv_repeatable_and_counters_reset(q8, ws):
    import torch
    q, s = synth.q8_matrix(512, 4096, 3, 52)
    x = dev(synth.normal((1, 4096), 3, recipes.VEC + 53))
    outs = []
    for _ in range(3):
        y = empty((1, 512), torch.float32)
        q8.q8_gemv(dev(q), dev(s), 0, y, x=x, ws=ws)
        outs.append(host(y))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_refusals(q8, ws):
    import torch
    q = empty((4, 40), torch.int8)
    s = empty((4, 1), torch.float32)
    y = empty((1, 4), torch.float32)
    x = empty((1, 40), torch.float32)
    with pytest.raises(q8.Q8Error, match="EUNSUPPORTED.*32-value"):
        q8.q8_gemv(q, s, 0, y, x=x, ws=ws)
    with pytest.raises(q8.Q8Error, match="EINVAL.*mode"):
        q8.q8_gemv(empty((4, 32), torch.int8), s, 5, y, x=x, ws=ws)


# ---- the mixture -----------------------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def moe_host():
    return recipes.moe_block(seed=0)


@pytest.fixture(scope="module")
def moe_dev(moe_host):
    return {k: (dev(v[0]), dev(v[1])) for k, v in moe_host.items()}


def _near_tie(logits, k):
    """True when the k-th and (k+1)-th logits are too close for f32 and f64 sums to agree on the choice."""
    if k >= len(logits):
        return False
    srt = np.sort(logits)[::-1]
    return (srt[k - 1] - srt[k]) < 1e-5 * np.max(np.abs(logits))


def _plan_tensors(E, choices):
    import torch
    return (empty((E,), torch.int32), empty((E + 1,), torch.int32), empty((choices,), torch.int32),
            empty((E + 1,), torch.int32))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("R", [1, 2, 16, 64])
@pytest.mark.parametrize("router_scale", [0.01, 1e-5])
def test_route_topk(q8, ws, mode, R, router_scale):
    import torch
    E, K, d = 128, 8, 2048
    rq, rs = synth.q8_matrix(E, d, 0, recipes.layer_ids(0)["router"], scale_mul=router_scale)
    x = synth.normal((R, d), 0, recipes.VEC + 60)
    ids = empty((R, K), torch.int32)
    gates = empty((R, K), torch.float32)
    logits = empty((R, E), torch.float32)
    pt = _plan_tensors(E, R * K)
    plan = q8.plan_struct(*pt)
    if mode == 0:
        q8.moe_route_topk(dev(rq), dev(rs), 0, K, ids, gates, x=dev(x), rows=R, logits=logits, plan=plan, ws=ws)
    else:
        xq, xs = oracle.quantize(x)
        q8.moe_route_topk(dev(rq), dev(rs), 1, K, ids, gates, xq=dev(xq), xs=dev(xs), rows=R, logits=logits, plan=plan,
                          ws=ws)
    gi, gg, gl = host(ids), host(gates), host(logits)
    for r in range(R):
        l = oracle.gemv(mode, rq, rs, x[r])
        oi, og = oracle.route(l, K)
        assert rel_err(gl[r], l) < TOL[mode]
        if not _near_tie(l, K):
            np.testing.assert_array_equal(gi[r], oi)
            assert rel_err(gg[r], og) < TOL[mode]
        assert abs(gg[r].sum() - 1.0) < 1e-5
    counts, offsets, lists = oracle.group(gi, E)
    np.testing.assert_array_equal(host(pt[0]), counts)
    np.testing.assert_array_equal(host(pt[1]), offsets)
    np.testing.assert_array_equal(host(pt[2]), lists)
    act = host(pt[3])
    active = np.nonzero(counts)[0]
    assert act[0] == len(active)
    np.testing.assert_array_equal(act[1:1 + len(active)], active)


def test_route_topk_grouping_many_rows(q8, ws):
    """2100 rows x 8 choices: more choices than the grouping stages in shared memory (it reads them from L2), and
    the rows spread over many CTAs whose last arrival groups them; the grouping is checked exactly."""
    import torch
    E, K, d, R = 128, 8, 2048, 2100
    rq, rs = synth.q8_matrix(E, d, 0, recipes.layer_ids(0)["router"])
    x = synth.normal((R, d), 0, recipes.VEC + 61)
    xq, xs = oracle.quantize(x)
    ids = empty((R, K), torch.int32)
    gates = empty((R, K), torch.float32)
    logits = empty((R, E), torch.float32)
    pt = _plan_tensors(E, R * K)
    q8.moe_route_topk(dev(rq), dev(rs), 1, K, ids, gates, xq=dev(xq), xs=dev(xs), rows=R, logits=logits,
                      plan=q8.plan_struct(*pt), ws=ws)
    gi = host(ids)
    for r in range(0, R, 97):  # sampled rows against the oracle
        l = oracle.gemv(1, rq, rs, x[r])
        if not _near_tie(l, K):
            np.testing.assert_array_equal(gi[r], oracle.route(l, K)[0])
    counts, offsets, lists = oracle.group(gi, E)
    np.testing.assert_array_equal(host(pt[0]), counts)
    np.testing.assert_array_equal(host(pt[1]), offsets)
    np.testing.assert_array_equal(host(pt[2]), lists)


def _run_moe_gpu(q8, ws, md, mode, x, K, residual=None, expert_out=True, route_plan=True, down_reads_h=True):
    import torch
    R, d = x.shape
    dff = md["gate"][0].shape[0] // md["router"][0].shape[0]
    E = md["router"][0].shape[0]
    ids = empty((R, K), torch.int32)
    gates = empty((R, K), torch.float32)
    logits = empty((R, E), torch.float32)
    pt = _plan_tensors(E, R * K)
    plan = q8.plan_struct(*pt) if R > 1 else None
    h = empty((R * K, dff), torch.float32)
    hq = empty((R * K, dff), torch.int8) if mode >= 1 else None
    hl = empty((R * K, dff), torch.int8) if mode == 2 else None
    hs = empty((R * K, dff // 32), torch.float32) if mode >= 1 else None
    y = empty((R, d), torch.float32)
    eo = empty((R, K, d), torch.float32) if expert_out else None
    tx = dev(x)
    xq = xs = xl = None
    if mode == 1:
        oq, os_ = oracle.quantize(x)
        xq, xs = dev(oq), dev(os_)
    elif mode == 2:
        oq, ol, os_ = oracle.quantize2(x)
        xq, xl, xs = dev(oq), dev(ol), dev(os_)
    q8.moe_route_topk(*md["router"], mode, K, ids, gates, x=tx, xq=xq, xs=xs, xl=xl, rows=R, logits=logits,
                      plan=q8.plan_struct(*pt) if route_plan else None, ws=ws)
    q8.moe_gate_up(*md["gate"], *md["up"], dff, mode, K, ids, h, x=tx, xq=xq, xs=xs, xl=xl, hq=hq, hs=hs, hl=hl,
                   rows=R, plan=plan, ws=ws)
    q8.moe_down_combine(*md["down"], d, mode, K, ids, gates, y, h=h if (down_reads_h or mode == 0) else None,
                        hq=hq, hs=hs, hl=hl, rows=R, plan=plan,
                        residual=dev(residual) if residual is not None else None, expert_out=eo, ws=ws)
    return dict(ids=host(ids), gates=host(gates), logits=host(logits), h=host(h).reshape(R, K, dff),
                y=host(y), expert_out=host(eo) if expert_out else None, hq=host(hq) if hq is not None else None,
                hs=host(hs) if hs is not None else None, hl=host(hl) if hl is not None else None)


def _compare_moe(out, ref, mode, K):
    """Row by row against the oracle.  A row whose oracle router logits hold a near tie at the K-th choice (within
    1e-5 of the largest magnitude) may choose either expert: it is counted, its outputs are still compared when the
    GPU chose the oracle's experts, and such rows must stay rare."""
    R = out["y"].shape[0]
    ties = 0
    for r in range(R):
        if _near_tie(ref["logits"][r], K):
            ties += 1
            if not np.array_equal(out["ids"][r], ref["ids"][r]):
                continue
        np.testing.assert_array_equal(out["ids"][r], ref["ids"][r])
        assert rel_err(out["gates"][r], ref["gates"][r]) < TOL[mode]
        for j in range(K):  # each expert separately: the gates are nearly one-hot at these router scales
            assert rel_err(out["h"][r, j], ref["hidden"][r, j]) < TOL[mode]
            if out["expert_out"] is not None:
                assert rel_err(out["expert_out"][r, j], ref["expert_out"][r, j]) < TOL[mode]
        assert rel_err(out["y"][r], ref["y"][r]) < TOL[mode]
    assert ties <= max(1, R // 16), f"{ties} of {R} rows hold a near tie"
    if out["hq"] is not None:  # gate-up's int8 epilogue = the quantizer applied to its own f32 rows, bit for bit
        h = out["h"].reshape(-1, out["h"].shape[-1])
        if mode == 2:
            oq, ol, os_ = oracle.quantize2(h)
            np.testing.assert_array_equal(out["hl"], ol)
        else:
            oq, os_ = oracle.quantize(h)
        np.testing.assert_array_equal(out["hq"], oq)
        np.testing.assert_array_equal(out["hs"].reshape(os_.shape), os_)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_moe_block_batch1(q8, ws, moe_host, moe_dev, mode):
    x = synth.normal((1, 2048), 0, recipes.VEC + 70)
    res = synth.normal((1, 2048), 0, recipes.VEC + 71)
    w = oracle.MoeWeights(2048, 768, 128, 8, **moe_host)
    ref = oracle.moe_rows(mode, w, x, residual=res)
    out = _run_moe_gpu(q8, ws, moe_dev, mode, x, 8, residual=res)
    _compare_moe(out, ref, mode, 8)


@pytest.mark.parametrize("mode,down_reads_h", [(0, True), (1, True), (1, False), (2, True), (2, False)])
@pytest.mark.parametrize("spread", [False, True])
def test_moe_one_row_fused_path(q8, ws, moe_host, moe_dev, mode, down_reads_h, spread):
    # one row, no plan, no per-expert outputs: the router and its top-k in one cluster launch, gate-up quantizing its
    # own rows, and the down-and-combine that loads its weights before waiting
    mh, md = moe_host, moe_dev
    if spread:
        mh = dict(moe_host)
        mh["router"] = synth.q8_matrix(128, 2048, 0, recipes.layer_ids(0)["router"], scale_mul=1e-5)
        md = dict(moe_dev)
        md["router"] = (dev(mh["router"][0]), dev(mh["router"][1]))
    for seed in range(3):
        x = synth.normal((1, 2048), seed, recipes.VEC + 74)
        res = synth.normal((1, 2048), seed, recipes.VEC + 75)
        ref = oracle.moe_rows(mode, oracle.MoeWeights(2048, 768, 128, 8, **mh), x, residual=res)
        # down_reads_h: f32 hidden rows staged in shared memory with the weights; else the int8 rows read directly
        out = _run_moe_gpu(q8, ws, md, mode, x, 8, residual=res, expert_out=False, route_plan=False,
                           down_reads_h=down_reads_h)
        assert rel_err(out["logits"][0], ref["logits"][0]) < TOL[mode]
        _compare_moe(out, ref, mode, 8)
        assert abs(out["gates"][0].sum() - 1.0) < 1e-5


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("E,K,d", [(4, 4, 64), (16, 3, 1024), (64, 32, 2048), (1000, 8, 4096), (1024, 1, 32)])
def test_route_one_row_shapes(q8, ws, mode, E, K, d):
    # the one-cluster router: experts not a multiple of the cluster, K = E, K = 32, the widest rows, one block (the f32
    # one-row router holds at most 2048 values a row: wider f32 rows take the projection + top-k launches)
    import torch
    rq, rs = synth.q8_matrix(E, d, 5, 95)
    x = synth.normal((1, d), 5, recipes.VEC + 96)
    ids = empty((1, K), torch.int32)
    gates = empty((1, K), torch.float32)
    logits = empty((1, E), torch.float32)
    if mode == 0:
        q8.moe_route_topk(dev(rq), dev(rs), 0, K, ids, gates, x=dev(x), rows=1, logits=logits, ws=ws)
    elif mode == 1:
        xq, xs = oracle.quantize(x)
        q8.moe_route_topk(dev(rq), dev(rs), 1, K, ids, gates, xq=dev(xq), xs=dev(xs), rows=1, logits=logits, ws=ws)
    else:
        xq, xl, xs = oracle.quantize2(x)
        q8.moe_route_topk(dev(rq), dev(rs), 2, K, ids, gates, xq=dev(xq), xs=dev(xs), xl=dev(xl), rows=1,
                          logits=logits, ws=ws)
    l = oracle.gemv(mode, rq, rs, x[0])
    gl = host(logits)[0]
    assert rel_err(gl, l) < TOL[mode]
    # ids and gates: the oracle's routing of the oracle's logits (descending, ties to the lower index)
    ora_ids, ora_g = oracle.route(l, K)
    if _near_tie(l, K):
        pytest.skip("the oracle's logits hold a near tie at the K-th choice (flagged)")
    np.testing.assert_array_equal(host(ids)[0], ora_ids)
    assert rel_err(host(gates)[0], ora_g) < TOL[mode]


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_moe_block_spread_gates(q8, ws, moe_host, mode):
    # router scales x1e-3: logits of std ~0.03, so all eight gates carry weight in the combine
    mh = dict(moe_host)
    mh["router"] = synth.q8_matrix(128, 2048, 0, recipes.layer_ids(0)["router"], scale_mul=1e-5)
    md = {k: (dev(v[0]), dev(v[1])) for k, v in mh.items()}
    x = synth.normal((1, 2048), 0, recipes.VEC + 72)
    w = oracle.MoeWeights(2048, 768, 128, 8, **mh)
    ref = oracle.moe_rows(mode, w, x)
    assert ref["gates"][0].min() > 0.05
    out = _run_moe_gpu(q8, ws, md, mode, x, 8)
    _compare_moe(out, ref, mode, 8)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("R", [2, 4, 8, 16, 32, 64])
def test_moe_chunk(q8, ws, moe_host, moe_dev, mode, R):
    x = synth.normal((R, 2048), 1, recipes.VEC + 80)
    w = oracle.MoeWeights(2048, 768, 128, 8, **moe_host)
    ref = oracle.moe_rows(mode, w, x)
    out = _run_moe_gpu(q8, ws, moe_dev, mode, x, 8)
    _compare_moe(out, ref, mode, 8)


@pytest.mark.parametrize("mode,R,grouped", [(0, 32, None), (1, 16, 16), (1, 16, 0), (1, 32, 16), (1, 32, None),
                                            (1, 64, None), (1, 64, 0), (2, 64, None)])
def test_moe_chunk_correlated_rows(q8, ws, moe_host, moe_dev, mode, R, grouped):
    # every row near one x0: the rows share their experts, so each expert's group holds all R rows.  Int8 mode: groups
    # of `grouped`..64 rows take the tensor-core products (None: the library's default of 32; 0: the CUDA cores only)
    x0 = synth.normal((1, 2048), 2, recipes.VEC + 81)
    x = (x0 + 0.01 * synth.normal((R, 2048), 2, recipes.VEC + 82)).astype(np.float32)
    w = oracle.MoeWeights(2048, 768, 128, 8, **moe_host)
    ref = oracle.moe_rows(mode, w, x)
    if grouped is not None:
        q8.set_grouped_tensor_core_rows(grouped)
    try:
        out = _run_moe_gpu(q8, ws, moe_dev, mode, x, 8)
    finally:
        q8.set_grouped_tensor_core_rows(32)
    _compare_moe(out, ref, mode, 8)


def test_moe_chunk_two_clusters_mixed_groups(q8, ws, moe_host, moe_dev):
    # 40 rows near x0 and 8 near x1: x0's experts get groups of 40 (tensor cores), x1's groups of 8 (CUDA cores),
    # experts both clusters choose get 48
    x0 = synth.normal((1, 2048), 5, recipes.VEC + 84)
    x1 = synth.normal((1, 2048), 5, recipes.VEC + 85)
    x = np.concatenate([x0 + 0.01 * synth.normal((40, 2048), 5, recipes.VEC + 86),
                        x1 + 0.01 * synth.normal((8, 2048), 5, recipes.VEC + 87)]).astype(np.float32)
    w = oracle.MoeWeights(2048, 768, 128, 8, **moe_host)
    ref = oracle.moe_rows(1, w, x)
    out = _run_moe_gpu(q8, ws, moe_dev, 1, x, 8)
    _compare_moe(out, ref, 1, 8)


def test_moe_chunk_equals_rows_one_by_one(q8, ws, moe_dev):
    # the chunk form computes each row exactly as the batch-1 form does (same ids; values within f32 rounding)
    x = synth.normal((8, 2048), 3, recipes.VEC + 83)
    chunk = _run_moe_gpu(q8, ws, moe_dev, 1, x, 8)
    for r in range(8):
        one = _run_moe_gpu(q8, ws, moe_dev, 1, x[r:r + 1], 8)
        np.testing.assert_array_equal(chunk["ids"][r], one["ids"][0])
        assert rel_err(chunk["y"][r], one["y"][0]) < 1e-6


def test_moe_small_shapes_and_k_equals_e(q8, ws):
    # E = K = 4 with zero router: equal gates, every expert kept, y = mean of the expert outputs (oracle pinned)
    import torch
    d, dff, E = 64, 32, 4
    mh = dict(router=(np.zeros((E, d), np.int8), np.zeros((E, 2), np.float32)),
              gate=synth.q8_matrix(E * dff, d, 4, 90), up=synth.q8_matrix(E * dff, d, 4, 91),
              down=synth.q8_matrix(E * d, dff, 4, 92))
    md = {k: (dev(v[0]), dev(v[1])) for k, v in mh.items()}
    for mode in (0, 1, 2):
        x = synth.normal((3, d), 4, recipes.VEC + 93)
        ref = oracle.moe_rows(mode, oracle.MoeWeights(d, dff, E, E, **mh), x)
        out = _run_moe_gpu(q8, ws, md, mode, x, E)
        np.testing.assert_array_equal(out["ids"], np.tile(np.arange(E), (3, 1)))
        np.testing.assert_allclose(out["gates"], 0.25, rtol=1e-6)
        assert rel_err(out["y"], ref["y"]) < TOL[mode]
        assert rel_err(out["y"], out["expert_out"].mean(1)) < 1e-5
    del torch


@pytest.mark.parametrize("n,k,R", [(4096, 2048, 16), (512, 2048, 32), (2048, 4096, 64), (128, 2048, 48),
                                   (640, 768, 17)])
def test_q8_gemv_rows_on_tensor_cores(q8, n, k, R):
    """16..64 int8 activation rows: the weight tiles go through the tensor-core kernel once for all rows (a workspace
    with room for it); the result equals the oracle, and the CUDA-core form (a workspace too small for the tensor
    path's lists) to f32 summation order."""
    import torch
    q, s = synth.q8_matrix(n, k, 6, 160 + n % 7)
    x = synth.normal((R, k), 6, recipes.VEC + 161)
    xq, xs = oracle.quantize(x)
    ref = np.stack([oracle.gemv_int8act(q, s, xq[r], xs[r]) for r in range(R)])
    big = q8.Workspace(64 << 20)
    y = empty((R, n), torch.float32)
    q8.set_tensor_core_rows(16)
    try:
        q8.q8_gemv(dev(q), dev(s), 1, y, xq=dev(xq), xs=dev(xs), rows=R, ws=big)
        gy = host(y)
    finally:
        q8.set_tensor_core_rows(-1)
    assert rel_err(gy, ref) < TOL[1], rel_err(gy, ref)
    small = q8.Workspace(1024)
    y2 = empty((R, n), torch.float32)
    try:
        q8.q8_gemv(dev(q), dev(s), 1, y2, xq=dev(xq), xs=dev(xs), rows=R, ws=small)
        assert rel_err(gy, host(y2)) < 1e-5
    except q8.Q8Error as e:  # the CUDA-core form cut along k needs more than the small workspace: skip the cross-check
        assert "ENOSPACE" in str(e)
    big.close()
    small.close()
