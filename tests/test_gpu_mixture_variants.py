"""GPU parity of the mixture's variants against the oracle, through the C ABI: a router of f32 values
(lane_link.rs, Link::prim Router::F32) and a shared expert fused with the mixture (Link::class_launch
SharedExpertFusion), alone and together, for one token row (the fused one-row kernels), for chunks of rows and
through the decode step and prefill, in every numerics mode.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import recipes

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 2e-3, 2: 2e-3}


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


def near_tie(logits, k):
    if k >= len(logits):
        return False
    srt = np.sort(logits)[::-1]
    return (srt[k - 1] - srt[k]) < 1e-5 * np.max(np.abs(logits))


@pytest.fixture(scope="module")
def ws(q8):
    w = q8.Workspace(256 << 20)
    yield w
    w.close()


D, DFF, E, K = 2048, 768, 128, 8


@pytest.fixture(scope="module")
def mix_host():
    m = recipes.moe_block(seed=0)
    cfg = dict(layers=1, d=D, experts=E)
    v = recipes.mixture_variants(cfg, seed=0, shared_dff=1536, router_f32=True)
    m["shared"] = dict(gate=v["shared_gate"][0], up=v["shared_up"][0], down=v["shared_down"][0])
    m["router_f32"] = v["router_f32"][0]
    return m


@pytest.fixture(scope="module")
def mix_dev(mix_host):
    out = {k: (dev(v[0]), dev(v[1])) for k, v in mix_host.items() if k in ("router", "gate", "up", "down")}
    out["shared"] = {k: (dev(v[0]), dev(v[1])) for k, v in mix_host["shared"].items()}
    out["router_f32"] = dev(mix_host["router_f32"])
    return out


def _run(q8, ws, md, mode, x, residual, use_rf, use_shared, sdff):
    import torch
    R = x.shape[0]
    ids = empty((R, K), torch.int32)
    gates = empty((R, K), torch.float32)
    logits = empty((R, E), torch.float32)
    pt = [empty((E,), torch.int32), empty((E + 1,), torch.int32), empty((R * K,), torch.int32),
          empty((E + 1,), torch.int32)]
    plan = q8.plan_struct(*pt) if R > 1 else None
    nh = R * K * DFF + (R * sdff if use_shared else 0)
    h = empty((nh,), torch.float32)
    hq = empty((nh,), torch.int8) if mode >= 1 else None
    hl = empty((nh,), torch.int8) if mode == 2 else None
    hs = empty((nh // 32,), torch.float32) if mode >= 1 else None
    y = empty((R, D), torch.float32)
    tx = dev(x)
    xq = xs = xl = None
    if mode == 1:
        a, b = oracle.quantize(x)
        xq, xs = dev(a), dev(b)
    elif mode == 2:
        a, c, b = oracle.quantize2(x)
        xq, xl, xs = dev(a), dev(c), dev(b)
    sh = q8.shared_expert(md["shared"]["gate"], md["shared"]["up"], md["shared"]["down"]) if use_shared else None
    if use_rf:
        q8.moe_route_topk_f32(md["router_f32"], K, ids, gates, tx, rows=R, logits=logits, plan=plan, ws=ws)
    else:
        q8.moe_route_topk(*md["router"], mode, K, ids, gates, x=tx, xq=xq, xs=xs, xl=xl, rows=R, logits=logits,
                          plan=plan, ws=ws)
    q8.moe_gate_up(*md["gate"], *md["up"], DFF, mode, K, ids, h, x=tx, xq=xq, xs=xs, xl=xl, hq=hq, hs=hs, hl=hl,
                   rows=R, plan=plan, ws=ws, shared=sh)
    q8.moe_down_combine(*md["down"], D, mode, K, ids, gates, y, h=h, hq=hq, hs=hs, hl=hl, rows=R, plan=plan,
                        residual=dev(residual), ws=ws, shared=sh)
    return dict(ids=host(ids), gates=host(gates), logits=host(logits), h=host(h), y=host(y))


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("R", [1, 5, 16])
@pytest.mark.parametrize("use_rf,use_shared", [(True, False), (False, True), (True, True)],
                         ids=["f32router", "shared", "both"])
def test_mixture_variants_match_oracle(q8, ws, mix_host, mix_dev, mode, R, use_rf, use_shared):
    sdff = 1536
    x = synth.normal((R, D), 3, recipes.VEC + 120)
    res = synth.normal((R, D), 3, recipes.VEC + 121)
    w = oracle.MoeWeights(D, DFF, E, K, mix_host["router"], mix_host["gate"], mix_host["up"], mix_host["down"],
                          router_f32=mix_host["router_f32"] if use_rf else None,
                          shared=mix_host["shared"] if use_shared else None)
    ref = oracle.moe_rows(mode, w, x, residual=res)
    out = _run(q8, ws, mix_dev, mode, x, res, use_rf, use_shared, sdff)
    # the f32 router's logits are an f32-activation product: the f32 tolerance in every mode
    assert rel_err(out["logits"], ref["logits"]) < (TOL[0] if use_rf else TOL[mode])
    ties = 0
    for r in range(R):
        if near_tie(ref["logits"][r], K):
            ties += 1
            if not np.array_equal(out["ids"][r], ref["ids"][r]):
                continue
        np.testing.assert_array_equal(out["ids"][r], ref["ids"][r])
        assert rel_err(out["gates"][r], ref["gates"][r]) < TOL[mode]
        assert rel_err(out["y"][r], ref["y"][r]) < TOL[mode], (r, rel_err(out["y"][r], ref["y"][r]))
    assert ties <= max(1, R // 8)
    if use_shared:  # the shared expert's hidden rows follow the routed ones
        hsh = out["h"][R * K * DFF:].reshape(R, sdff)
        assert rel_err(hsh, ref["shared_hidden"]) < TOL[mode]


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_shared_expert_of_the_experts_width_one_row(q8, ws, mix_host, mode):
    # sdff = dff: the shared expert as a ninth row set of the fused one-row kernels
    import torch
    v = recipes.mixture_variants(dict(layers=1, d=D, experts=E), seed=1, shared_dff=DFF)
    shared = dict(gate=v["shared_gate"][0], up=v["shared_up"][0], down=v["shared_down"][0])
    md = {k: (dev(mix_host[k][0]), dev(mix_host[k][1])) for k in ("router", "gate", "up", "down")}
    md["shared"] = {k: (dev(a), dev(b)) for k, (a, b) in shared.items()}
    x = synth.normal((1, D), 4, recipes.VEC + 122)
    res = synth.normal((1, D), 4, recipes.VEC + 123)
    ref = oracle.moe_rows(mode, oracle.MoeWeights(D, DFF, E, K, mix_host["router"], mix_host["gate"], mix_host["up"],
                                                  mix_host["down"], shared=shared), x, residual=res)
    out = _run(q8, ws, md, mode, x, res, False, True, DFF)
    if not near_tie(ref["logits"][0], K):
        np.testing.assert_array_equal(out["ids"][0], ref["ids"][0])
        assert rel_err(out["y"][0], ref["y"][0]) < TOL[mode]
    del torch


# ---- through the decode step and prefill -----------------------------------------------------------------------

SMALL = dict(layers=2, d=256, heads=8, kv_heads=2, hd=128, experts=16, k=4, dff=64, vocab=1000, ctx=96, eps=1e-6,
             rope_theta=1e6)


def _model(q8, cfg, seed, mode, sdff, rf):
    import torch
    arr = recipes.decode_model(cfg, seed)
    arr.update(recipes.mixture_variants(cfg, seed, shared_dff=sdff, router_f32=rf))

    def up(v):
        if isinstance(v, list):
            return [up(e) for e in v]
        if isinstance(v, tuple):
            return tuple(up(e) for e in v)
        return dev(v)

    t = {k: up(v) for k, v in arr.items()}
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    m = q8.Model(cfg, t, mode, tok, pos, logits)
    om = oracle.ModelArrays(cfg, **arr)
    return m, om, t, tok, pos, logits


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("sdff,rf", [(64, False), (0, True), (128, True)], ids=["shared", "f32router", "both"])
def test_decode_with_variants_matches_oracle(q8, mode, sdff, rf):
    import torch
    m, om, t, tok, pos, logits = _model(q8, SMALL, 31, mode, sdff, rf)
    cur_tok, cur_pos = 11, 50
    tok.fill_(cur_tok)
    pos.fill_(cur_pos)
    for step in range(3):
        nxt, ora = oracle.decode_step(mode, om, cur_tok, cur_pos)
        (m.step if step % 2 == 0 else m.step_launches)()
        torch.cuda.synchronize()
        assert rel_err(logits.cpu().numpy(), ora) < TOL[mode], (step, rel_err(logits.cpu().numpy(), ora))
        for l in range(SMALL["layers"]):
            kc, vc = t["k_cache"][l].cpu().numpy(), t["v_cache"][l].cpu().numpy()
            assert rel_err(kc[:, cur_pos], om.k_cache[l][:, cur_pos]) < TOL[mode]
            assert rel_err(vc[:, cur_pos], om.v_cache[l][:, cur_pos]) < TOL[mode]
        cur_tok, cur_pos = int(tok.item()), cur_pos + 1
    m.check()
    m.close()


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_prefill_with_variants_matches_oracle(q8, mode):
    import torch
    m, om, t, tok, pos, logits = _model(q8, SMALL, 32, mode, 96, True)
    ws = q8.Workspace(64 << 20)
    tokens = [7, 300, 21, 999, 5, 64, 128]
    pos.fill_(40)
    m.prefill(torch.tensor(tokens, dtype=torch.int32, device="cuda"), ws)
    torch.cuda.synchronize()
    for r, tk in enumerate(tokens):
        nxt, ora = oracle.decode_step(mode, om, tk, 40 + r)
    assert rel_err(logits.cpu().numpy(), ora) < TOL[mode]
    assert int(pos.item()) == 40 + len(tokens)
    for l in range(SMALL["layers"]):
        kc = t["k_cache"][l].cpu().numpy()
        assert rel_err(kc[:, 40:40 + len(tokens)], om.k_cache[l][:, 40:40 + len(tokens)]) < TOL[mode]
    m.check()
    ws.close()
    m.close()
