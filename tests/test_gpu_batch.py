"""The batch form (lane/mod.rs: Form / FormKind::Batch, batch_io): B sequences step together, every weight read once
for all of them, each sequence attending its own cache at its own position.  Each sequence's logits, token, position
and new cache rows equal the oracle's decode step of that sequence alone (same weights, its own caches)."""
import numpy as np
import pytest

import oracle
import synth
from layer_parity import check_token, layer_vs_oracle
from synth import recipes

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 2e-3, 2: 2e-3}


def rel_err(gpu, ora):
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    return float(np.max(np.abs(gpu - ora)) / max(np.max(np.abs(ora)), 1e-300))


SMALL = dict(layers=2, d=256, heads=8, kv_heads=2, hd=128, experts=16, k=4, dff=64, vocab=1000, ctx=96, eps=1e-6,
             rope_theta=1e6)


def _near_tie(logits, k):
    srt = np.sort(np.asarray(logits, np.float64))[::-1]
    return srt[k - 1] - srt[k] < 1e-5 * np.max(np.abs(srt))


def _batch_model(q8, cfg, B, seed, mode, variants=None):
    import torch
    arr = recipes.decode_model(cfg, seed)
    if variants:
        arr.update(recipes.mixture_variants(cfg, seed, **variants))
    L, KV, ctx, hd = cfg["layers"], cfg["kv_heads"], cfg["ctx"], cfg["hd"]
    # sequence b's caches: its own seeded values (sequence 0 keeps the model's)
    kc = [[arr["k_cache"][l]] + [synth.normal((KV, ctx, hd), seed + b, 9000 + l) for b in range(1, B)] for l in range(L)]
    vc = [[arr["v_cache"][l]] + [synth.normal((KV, ctx, hd), seed + b, 9100 + l) for b in range(1, B)] for l in range(L)]

    def dv(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    t = {}
    for key, v in arr.items():
        if key in ("k_cache", "v_cache"):
            continue
        if isinstance(v, list):
            t[key] = [tuple(dv(x) for x in e) if isinstance(e, tuple) else dv(e) for e in v]
        elif isinstance(v, tuple):
            t[key] = tuple(dv(x) for x in v)
        else:
            t[key] = dv(v)
    t["k_cache"] = [dv(np.stack(kc[l])) for l in range(L)]
    t["v_cache"] = [dv(np.stack(vc[l])) for l in range(L)]
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, cfg["vocab"], dtype=torch.float32, device="cuda")
    m = q8.Model(dict(cfg, batch=B), t, mode, tok, pos, logits)
    oms = []
    for b in range(B):
        ab = dict(arr)
        ab["k_cache"] = [kc[l][b].copy() for l in range(L)]
        ab["v_cache"] = [vc[l][b].copy() for l in range(L)]
        oms.append(oracle.ModelArrays(cfg, **ab))
    return m, oms, t, tok, pos, logits


def _oracle_step(mode, om, cfg, tok, pos):
    """The oracle's decode step layer by layer, with whether any layer's router held a near tie on the way (the
    K-th and (K+1)-th logits within 1e-5 of the largest: a choice last-bit differences may flip)."""
    h = om.embed[tok]
    tie = False
    for l in range(cfg["layers"]):
        h, rl = oracle.decode_layer(mode, om, l, pos, h)
        tie = tie or _near_tie(rl, cfg["k"])
    nxt, logits = oracle.decode_final(mode, om, h)
    return nxt, logits, tie


def _steps_vs_oracle(q8, cfg, B, mode, toks, poss, steps, seed, variants=None):
    """B sequences stepped together, each against its own oracle decode steps.  A sequence whose oracle path met a
    router near tie is flagged and left out from then on (its path may fork from the GPU's there); such forks must
    stay rare."""
    import torch
    m, oms, t, tok, pos, logits = _batch_model(q8, cfg, B, seed, mode, variants)
    tok.copy_(torch.tensor(toks, dtype=torch.int32))
    pos.copy_(torch.tensor(poss, dtype=torch.int32))
    cur_t, cur_p = list(toks), list(poss)
    forked = set()
    for step in range(steps):
        (m.step if step % 2 == 0 else m.step_launches)()
        torch.cuda.synchronize()
        gl = logits.cpu().numpy()
        gt, gp = tok.cpu().numpy(), pos.cpu().numpy()
        for b in range(B):
            assert gp[b] == cur_p[b] + 1
            if b not in forked:
                nxt, ora, tie = _oracle_step(mode, oms[b], cfg, cur_t[b], cur_p[b])
                if tie:
                    forked.add(b)
                else:
                    assert rel_err(gl[b], ora) < TOL[mode], (step, b, rel_err(gl[b], ora))
                    check_token(gt[b], ora, TOL[mode])
                    for l in range(cfg["layers"]):
                        kcb = t["k_cache"][l][b].cpu().numpy()
                        vcb = t["v_cache"][l][b].cpu().numpy()
                        assert rel_err(kcb[:, cur_p[b]], oms[b].k_cache[l][:, cur_p[b]]) < TOL[mode]
                        assert rel_err(vcb[:, cur_p[b]], oms[b].v_cache[l][:, cur_p[b]]) < TOL[mode]
            cur_t[b], cur_p[b] = int(gt[b]), cur_p[b] + 1
    assert len(forked) <= max(1, B // 4), forked
    m.check()
    return m


@pytest.fixture(params=["chunked", "streamed"])
def attn_form(q8, request):
    """The batch attention's two forms: chunks folded in clusters, or splits streamed through a copy ring (forced for
    every batch size here)."""
    q8.set_streamed_batch_attention(0 if request.param == "chunked" else 2)
    yield request.param
    q8.set_streamed_batch_attention(8)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("B", [2, 5])
def test_batch_step_equals_independent_steps(q8, mode, B, attn_form):
    toks = [3, 500, 77, 999, 12][:B]
    poss = [10, 63, 0, 94, 40][:B]  # different lengths, from one row to the cache's end
    m = _steps_vs_oracle(q8, SMALL, B, mode, toks, poss, 2 if max(poss) >= 94 else 3, 41)
    m.close()


@pytest.mark.parametrize("mode", [1, 0])
def test_batch_long_caches_split_over_positions(q8, mode, attn_form):
    """Caches of 1536 rows: the streamed form cuts each (sequence, head) into three splits of eight 64-position stages,
    so one row, a stage exactly, a stage boundary, several splits (some empty at short lengths) and the cache's
    last rows all occur; the chunked form folds up to three clusters."""
    cfg = dict(SMALL, ctx=1536)
    m = _steps_vs_oracle(q8, cfg, 5, mode, [3, 500, 77, 999, 12], [0, 63, 64, 700, 1534], 2, 48)
    m.close()


def test_batch_step_with_mixture_variants(q8):
    m = _steps_vs_oracle(q8, SMALL, 3, 1, [1, 2, 3], [20, 30, 40], 2, 42,
                         variants=dict(shared_dff=64, router_f32=True))
    m.close()


@pytest.mark.parametrize("mode", [1, 0, 2])
def test_batch_full_width_layer_by_layer(q8, mode):
    """Teacher-forced over two steps, as the single-sequence full-configuration test: each batch step exports every
    sequence's residual stream entering each layer; the oracle runs each layer of each sequence from that same input
    (its own cache, which it appends to as the GPU does), and each layer's output and increment, its new key and value
    rows, and the final norm / LM head from the last stream are within the mode's tolerance.  The second step reads the
    cache rows the first wrote.  (End to end, untethered, two correctly rounding implementations drift apart through
    the layers at a rate set by the random weights' conditioning; the per-layer comparison is the one a kernel fault
    cannot hide from.)"""
    import torch
    cfg = dict(recipes.DECODE, layers=4, vocab=1000)
    L, K, d = cfg["layers"], cfg["k"], cfg["d"]
    toks, poss = [5, 6, 7, 8], [4000, 4050, 3000, 4093]
    B = len(toks)
    m, oms, t, tok, pos, logits = _batch_model(q8, cfg, B, 46, mode)
    tok.copy_(torch.tensor(toks, dtype=torch.int32))
    pos.copy_(torch.tensor(poss, dtype=torch.int32))
    arr_embed = recipes.decode_model(dict(cfg, layers=1), 46)["embed"]
    flagged, worst = [], {}
    cur_t, cur_p = list(toks), list(poss)
    hidden = torch.empty(L + 1, B, d, device="cuda")
    for step in range(2):
        m.step_trace(hidden)
        torch.cuda.synchronize()
        hid = hidden.cpu().numpy()
        gl = logits.cpu().numpy()
        for b in range(B):
            np.testing.assert_array_equal(hid[0, b], arr_embed[cur_t[b]])
            for l in range(L):
                h_ora, rl = oracle.decode_layer(mode, oms[b], l, cur_p[b], hid[l, b])
                if _near_tie(rl, K):
                    flagged.append((step, b, l))
                    continue
                err_out = rel_err(hid[l + 1, b], h_ora)
                err_inc = rel_err(hid[l + 1, b].astype(np.float64) - hid[l, b],
                                  h_ora.astype(np.float64) - hid[l, b])
                kcb = t["k_cache"][l][b].cpu().numpy()[:, cur_p[b]]
                vcb = t["v_cache"][l][b].cpu().numpy()[:, cur_p[b]]
                err_k = rel_err(kcb, oms[b].k_cache[l][:, cur_p[b]])
                err_v = rel_err(vcb, oms[b].v_cache[l][:, cur_p[b]])
                for name, e in (("out", err_out), ("inc", err_inc), ("k", err_k), ("v", err_v)):
                    worst[name] = max(worst.get(name, 0.0), e)
                assert max(err_out, err_inc, err_k, err_v) < TOL[mode], (step, b, l, err_out, err_inc, err_k, err_v)
            _, ora_logits = oracle.decode_final(mode, oms[b], hid[L, b])
            worst["logits"] = max(worst.get("logits", 0.0), rel_err(gl[b], ora_logits))
            assert rel_err(gl[b], ora_logits) < TOL[mode], (step, b, rel_err(gl[b], ora_logits))
        nt, np_ = tok.cpu().tolist(), pos.cpu().tolist()
        assert np_ == [p + 1 for p in cur_p]
        cur_t, cur_p = nt, np_
    print(f"batch mode {mode}: worst per-layer relative errors {worst}; near-tie layers {flagged}")
    assert len(flagged) <= 2, flagged
    m.close()


def test_batch_32_sequences_layer_by_layer(q8):
    """32 sequences at full width (two layers, one graph step, int8 mode): the step's projections and mixture have 32
    rows, so the O projection and the expert groups that 16 or more sequences share reach the tensor cores inside the
    captured graph.  Teacher forced: every sequence's layers against the oracle from the GPU's own inputs, a word on a
    rounding boundary rounded either way (layer_vs_oracle); its key and value rows and logits within the tolerance."""
    import torch
    cfg = dict(recipes.DECODE, layers=2, vocab=1000)
    L, K, d, B = cfg["layers"], cfg["k"], cfg["d"], 32
    rng = np.random.default_rng(32)
    toks = [int(v) for v in rng.integers(0, cfg["vocab"], B)]
    poss = [int(v) for v in rng.integers(3500, 4095, B)]
    q8.set_grouped_tensor_core_rows(16)
    try:
        m, oms, t, tok, pos, logits = _batch_model(q8, cfg, B, 47, 1)
        tok.copy_(torch.tensor(toks, dtype=torch.int32))
        pos.copy_(torch.tensor(poss, dtype=torch.int32))
        hidden = torch.empty(L + 1, B, d, device="cuda")
        m.step_trace(hidden)
        torch.cuda.synchronize()
        m.check()
    finally:
        q8.set_grouped_tensor_core_rows(32)
    hid = hidden.cpu().numpy()
    gl = logits.cpu().numpy()
    flagged, rounded, worst = [], [], 0.0
    for b in range(B):
        for l in range(L):
            rl, err, word = layer_vs_oracle(1, oms[b], l, poss[b], hid[l, b], hid[l + 1, b], TOL[1])
            kcb = t["k_cache"][l][b].cpu().numpy()[:, poss[b]]
            vcb = t["v_cache"][l][b].cpu().numpy()[:, poss[b]]
            err_kv = max(rel_err(kcb, oms[b].k_cache[l][:, poss[b]]), rel_err(vcb, oms[b].v_cache[l][:, poss[b]]))
            assert err_kv < TOL[1], (b, l, err_kv)
            if _near_tie(rl, K):
                flagged.append((b, l))
                continue
            if word is not None:
                rounded.append((b, l, word))
            worst = max(worst, err, err_kv)
            assert err < TOL[1], (b, l, err)
        _, ora_logits = oracle.decode_final(1, oms[b], hid[L, b])
        assert rel_err(gl[b], ora_logits) < TOL[1], (b, rel_err(gl[b], ora_logits))
    assert len(flagged) <= 3, flagged
    assert len(rounded) <= 6, rounded
    print(f"32 sequences: worst per-layer relative error {worst:.3e}; near ties {flagged}; rounded {rounded}")
    m.close()


def test_batch_graph_equals_launches_bitwise(q8, attn_form):
    import torch
    outs = []
    for use_graph in (True, False):
        m, oms, t, tok, pos, logits = _batch_model(q8, SMALL, 3, 44, 2)
        tok.copy_(torch.tensor([4, 5, 6], dtype=torch.int32))
        pos.copy_(torch.tensor([7, 8, 9], dtype=torch.int32))
        for _ in range(3):
            (m.step if use_graph else m.step_launches)()
        torch.cuda.synchronize()
        outs.append((logits.cpu().numpy().copy(), tok.cpu().numpy().copy(), t["k_cache"][1].cpu().numpy().copy()))
        m.close()
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)


def test_batch_bad_position_is_flagged_and_nothing_advances(q8, attn_form):
    import torch
    m, oms, t, tok, pos, logits = _batch_model(q8, SMALL, 3, 45, 0)
    tok.copy_(torch.tensor([1, 2, 3], dtype=torch.int32))
    pos.copy_(torch.tensor([5, SMALL["ctx"], 7], dtype=torch.int32))  # sequence 1 is past its cache
    m.step()
    torch.cuda.synchronize()
    assert pos.cpu().tolist() == [5, SMALL["ctx"], 7] and tok.cpu().tolist() == [1, 2, 3]
    with pytest.raises(q8.Q8Error, match="position"):
        m.check()
    m.close()
