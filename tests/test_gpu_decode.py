"""The decode step (embedding, 48-layer shape, LM head, greedy token) against the oracle, and graph replay."""
import numpy as np
import pytest

import oracle
from layer_parity import check_token, layer_vs_oracle
from synth import recipes

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 2e-3, 2: 2e-3}  # mode 2: the two-word activation, an int8-activation mode


def rel_err(gpu, ora):
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    return float(np.max(np.abs(gpu - ora)) / max(np.max(np.abs(ora)), 1e-300))


def build(q8, cfg, seed, mode):
    import torch
    arr = recipes.decode_model(cfg, seed)

    def dv(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    t = {}
    for key, v in arr.items():
        if isinstance(v, list):
            t[key] = [tuple(dv(x) for x in e) if isinstance(e, tuple) else dv(e) for e in v]
        elif isinstance(v, tuple):
            t[key] = tuple(dv(x) for x in v)
        else:
            t[key] = dv(v)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(cfg["vocab"], dtype=torch.float32, device="cuda")
    m = q8.Model(cfg, t, mode, tok, pos, logits)
    return m, arr, t, tok, pos, logits


SMALL = dict(layers=2, d=256, heads=8, kv_heads=2, hd=128, experts=16, k=4, dff=64, vocab=1000, ctx=96, eps=1e-6,
             rope_theta=1e6)


# d = 160: no projection takes the TMA path or a norm prologue, so every norm is a launch of its own
UNFUSED = dict(layers=2, d=160, heads=4, kv_heads=2, hd=128, experts=8, k=2, dff=32, vocab=300, ctx=70, eps=1e-6,
               rope_theta=1e6)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("cfg,launches", [(SMALL, lambda L: 6 * L + 2), (UNFUSED, lambda L: 8 * L + 3)],
                         ids=["fused", "unfused"])
def test_decode_small_matches_oracle_over_steps(q8, mode, cfg, launches):
    import torch
    m, arr, t, tok, pos, logits = build(q8, cfg, 5, mode)
    om = oracle.ModelArrays(cfg, **arr)
    cur_tok, cur_pos = 7, min(60, cfg["ctx"] - 5)
    tok.fill_(cur_tok)
    pos.fill_(cur_pos)
    for step in range(4):
        nxt, ora_logits = oracle.decode_step(mode, om, cur_tok, cur_pos)
        if step % 2 == 0:
            m.step()            # graph replay (captured on the first call)
        else:
            m.step_launches()   # plain launches
        torch.cuda.synchronize()
        gl = logits.cpu().numpy()
        assert rel_err(gl, ora_logits) < TOL[mode], (step, rel_err(gl, ora_logits))
        check_token(int(tok.item()), ora_logits, TOL[mode])
        assert int(pos.item()) == cur_pos + 1
        # the step wrote its key/value rows at cur_pos
        for l in range(cfg["layers"]):
            kc, vc = t["k_cache"][l].cpu().numpy(), t["v_cache"][l].cpu().numpy()
            assert rel_err(kc[:, cur_pos], om.k_cache[l][:, cur_pos]) < TOL[mode]
            assert rel_err(vc[:, cur_pos], om.v_cache[l][:, cur_pos]) < TOL[mode]
        cur_tok, cur_pos = int(tok.item()), cur_pos + 1
    # fused: per layer q/k/v (+norm), attention (+QK-norm, RoPE, append), O, router (+norm, top-k), gate-up, down;
    # then LM head (+final norm) and arg-max.  Unfused adds the two norms per layer and the final norm.
    assert m.launches_per_step() == launches(cfg["layers"])
    m.check()
    m.close()


# dff a multiple of 128 and 4 key/value heads (38 attention CTAs a head on 152 SMs, as in the full configuration): the
# int8 modes can run the layers as one persistent launch (q8_set_persistent_decode)
PERSIST = dict(SMALL, dff=128, heads=16, kv_heads=4)


@pytest.fixture
def persistent(q8):
    """The persistent step switched on for one test (the library's default is six launches a layer)."""
    q8.set_persistent_decode(True)
    yield
    q8.set_persistent_decode(False)


@pytest.mark.parametrize("mode", [1, 2])
def test_decode_persistent_matches_oracle_over_steps(q8, persistent, mode):
    """The persistent step (one launch for all layers, then LM head and arg-max) over four steps, teacher forced: each
    step exports the residual stream entering every layer, every layer's output (and its increment) is within the
    mode's tolerance of the oracle's layer run from the GPU's own input (a word on a rounding boundary may be rounded
    the other way, _layer_vs_oracle), the oracle's cache rows at the step's position come from those same inputs, and
    the logits and token follow from the GPU's final residual row.  (End to end, an activation word or a router choice
    decided by the last bits of an input can send the GPU and the oracle down two equally valid paths.)"""
    import torch
    m, arr, t, tok, pos, logits = build(q8, PERSIST, 5, mode)
    assert m.persistent()
    om = oracle.ModelArrays(PERSIST, **arr)
    L = PERSIST["layers"]
    cur_tok, cur_pos = 7, 60
    tok.fill_(cur_tok)
    pos.fill_(cur_pos)
    for step in range(4):
        hidden = torch.empty(L + 1, PERSIST["d"], device="cuda")
        m.step_trace(hidden)
        torch.cuda.synchronize()
        hid = hidden.cpu().numpy()
        np.testing.assert_array_equal(hid[0], arr["embed"][cur_tok])
        for l in range(L):
            _, e, _ = _layer_vs_oracle(mode, om, l, cur_pos, hid[l], hid[l + 1])
            assert e < TOL[mode], (step, l, e)
            kc, vc = t["k_cache"][l][:, cur_pos].cpu().numpy(), t["v_cache"][l][:, cur_pos].cpu().numpy()
            assert rel_err(kc, om.k_cache[l][:, cur_pos]) < TOL[mode]
            assert rel_err(vc, om.v_cache[l][:, cur_pos]) < TOL[mode]
        nxt, ora_logits = oracle.decode_final(mode, om, hid[L])
        gl = logits.cpu().numpy()
        assert rel_err(gl, ora_logits) < TOL[mode], (step, rel_err(gl, ora_logits))
        check_token(int(tok.item()), ora_logits, TOL[mode])
        assert int(pos.item()) == cur_pos + 1
        cur_tok, cur_pos = int(tok.item()), cur_pos + 1
    m.step()  # the captured graph: the layers, the LM head (+final norm), the arg-max
    torch.cuda.synchronize()
    assert m.launches_per_step() == 3
    m.check()
    m.close()


@pytest.mark.parametrize("pos0", [0, 1, 75, 95], ids=["first", "second", "mid", "last"])
def test_decode_persistent_equals_launch_per_stage(q8, pos0):
    """The persistent step and the six-launches-a-layer step on the same model and cache: every layer's residual
    stream and the logits agree to the attention's summation order (the other stages' arithmetic is the same), and both
    write the same new key and value rows; at every cache length, the shortest ones included (most attention CTAs then
    hold no position)."""
    import torch
    outs = []
    for on in (True, False):
        q8.set_persistent_decode(on)
        try:
            m, arr, t, tok, pos, logits = build(q8, PERSIST, 9, 1)
            assert m.persistent() == on
            tok.fill_(11)
            pos.fill_(pos0)
            hidden = torch.empty(PERSIST["layers"] + 1, PERSIST["d"], device="cuda")
            m.step_trace(hidden)
            torch.cuda.synchronize()
            outs.append((hidden.cpu().numpy(), logits.cpu().numpy().copy(),
                         [c[:, pos0].cpu().numpy() for c in t["k_cache"]],
                         [c[:, pos0].cpu().numpy() for c in t["v_cache"]]))
            m.check()
            m.close()
        finally:
            q8.set_persistent_decode(False)
    (h1, l1, k1, v1), (h0, l0, k0, v0) = outs
    np.testing.assert_array_equal(h1[0], h0[0])
    for l in range(1, PERSIST["layers"] + 1):
        assert rel_err(h1[l], h0[l]) < 1e-4, (l, rel_err(h1[l], h0[l]))
    assert rel_err(l1, l0) < 1e-4
    for a, b in zip(k1 + v1, k0 + v0):
        assert rel_err(a, b) < 1e-5


@pytest.mark.parametrize("mode", [1, 2])
def test_decode_persistent_full_dims_layer_by_layer(q8, persistent, mode):
    """Every dimension of the full configuration with 8 layers, at the last cache position, through the persistent step
    (152 CTAs: 34 q/k/v rows, 38 attention CTAs a key/value head of 108 positions each, 14 O and down rows, 41 gate-up
    row pairs a CTA), teacher forced layer by layer as in the 48-layer test, then the final norm, LM head and token."""
    import torch
    cfg = dict(recipes.DECODE, layers=8)
    L = cfg["layers"]
    m, arr, t, tok, pos, logits = build(q8, cfg, 0, mode)
    if not m.persistent():
        pytest.skip("the persistent step does not fit this device")
    om = oracle.ModelArrays(cfg, **arr)
    P = cfg["ctx"] - 1
    tok.fill_(0)
    pos.fill_(P)
    hidden = torch.empty(L + 1, cfg["d"], device="cuda")
    m.step_trace(hidden)
    torch.cuda.synchronize()
    hid = hidden.cpu().numpy()
    np.testing.assert_array_equal(hid[0], arr["embed"][0])
    flagged = []
    for l in range(L):
        rl, e, _ = _layer_vs_oracle(mode, om, l, P, hid[l], hid[l + 1])
        if _near_tie(rl, cfg["k"]):
            flagged.append(l)
            continue
        assert e < TOL[mode], (l, e)
        kc, vc = t["k_cache"][l][:, P].cpu().numpy(), t["v_cache"][l][:, P].cpu().numpy()
        assert rel_err(kc, om.k_cache[l][:, P]) < TOL[mode]
        assert rel_err(vc, om.v_cache[l][:, P]) < TOL[mode]
    assert len(flagged) <= 1, flagged
    nxt, ora_logits = oracle.decode_final(mode, om, hid[L])
    assert rel_err(logits.cpu().numpy(), ora_logits) < TOL[mode]
    m.check()
    m.close()


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("cfg", [dict(PERSIST, d=1024), dict(PERSIST, d=4096, heads=8)], ids=["d1024", "d4096"])
def test_decode_persistent_other_widths_layer_by_layer(q8, persistent, mode, cfg):
    """The persistent step's other row widths (the kernel's instances for d up to 1024 and up to 4096), teacher forced
    layer by layer against the oracle, then the final norm and LM head."""
    import torch
    m, arr, t, tok, pos, logits = build(q8, cfg, 21, mode)
    assert m.persistent()
    om = oracle.ModelArrays(cfg, **arr)
    L, P = cfg["layers"], 50
    tok.fill_(9)
    pos.fill_(P)
    hidden = torch.empty(L + 1, cfg["d"], device="cuda")
    m.step_trace(hidden)
    torch.cuda.synchronize()
    hid = hidden.cpu().numpy()
    for l in range(L):
        _, e, _ = _layer_vs_oracle(mode, om, l, P, hid[l], hid[l + 1])
        assert e < TOL[mode], (l, e)
        assert rel_err(t["k_cache"][l][:, P].cpu().numpy(), om.k_cache[l][:, P]) < TOL[mode]
    nxt, ora_logits = oracle.decode_final(mode, om, hid[L])
    assert rel_err(logits.cpu().numpy(), ora_logits) < TOL[mode]
    m.check()
    m.close()


def test_decode_persistent_graph_equals_launches_bitwise(q8, persistent):
    import torch
    outs = []
    for use_graph in (True, False):
        m, arr, t, tok, pos, logits = build(q8, PERSIST, 6, 1)
        assert m.persistent()
        tok.fill_(3)
        pos.fill_(10)
        for _ in range(3):
            (m.step if use_graph else m.step_launches)()
        torch.cuda.synchronize()
        outs.append((logits.cpu().numpy().copy(), int(tok.item()), int(pos.item()),
                     t["k_cache"][1].cpu().numpy().copy()))
        m.close()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    assert outs[0][1:3] == outs[1][1:3]
    np.testing.assert_array_equal(outs[0][3], outs[1][3])


def test_decode_persistent_bad_position_is_refused_on_device(q8, persistent):
    import torch
    m, arr, t, tok, pos, logits = build(q8, PERSIST, 7, 1)
    assert m.persistent()
    tok.fill_(1)
    pos.fill_(PERSIST["ctx"])  # one past the cache
    before = [c.clone() for c in t["k_cache"] + t["v_cache"]]
    m.step()
    torch.cuda.synchronize()
    assert int(pos.item()) == PERSIST["ctx"] and int(tok.item()) == 1
    for a, b in zip(before, t["k_cache"] + t["v_cache"]):
        assert torch.equal(a, b)
    with pytest.raises(q8.Q8Error, match="position"):
        m.check()
    m.close()


def test_decode_persistent_step_after_a_timeout_waits_for_nothing(q8, persistent):
    """With a timeout on record (the bounded-wait self-test leaves one), a persistent step skips every wait, grid and
    copy alike, and runs to its end instead of waiting on CTAs that may have given up; q8_model_check reports the
    timeout and resets the grid-barrier counters, and the next step is valid again."""
    import torch
    m, arr, t, tok, pos, logits = build(q8, PERSIST, 8, 1)
    assert m.persistent()
    om = oracle.ModelArrays(PERSIST, **arr)
    m.wait_selftest(64)
    tok.fill_(2)
    pos.fill_(30)
    m.step()
    torch.cuda.synchronize()
    with pytest.raises(q8.Q8Error, match="Q8_ETIMEOUT"):
        m.check()
    m.check()  # cleared
    # the cache row at 30 may hold anything now: rerun from the oracle's row 30 onwards on a clean cache copy
    for l in range(PERSIST["layers"]):
        t["k_cache"][l].copy_(torch.from_numpy(arr["k_cache"][l]))
        t["v_cache"][l].copy_(torch.from_numpy(arr["v_cache"][l]))
    tok.fill_(2)
    pos.fill_(30)
    m.step()
    torch.cuda.synchronize()
    nxt, ora_logits = oracle.decode_step(1, om, 2, 30)
    assert rel_err(logits.cpu().numpy(), ora_logits) < TOL[1]
    assert int(pos.item()) == 31
    m.check()
    m.close()


def test_decode_graph_equals_launches_bitwise(q8):
    import torch
    cfg = SMALL
    outs = []
    for use_graph in (True, False):
        m, arr, t, tok, pos, logits = build(q8, cfg, 6, 1)
        tok.fill_(3)
        pos.fill_(10)
        for _ in range(3):
            (m.step if use_graph else m.step_launches)()
        torch.cuda.synchronize()
        outs.append((logits.cpu().numpy().copy(), int(tok.item()), int(pos.item()),
                     t["k_cache"][1].cpu().numpy().copy()))
        m.close()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    assert outs[0][1:3] == outs[1][1:3]
    np.testing.assert_array_equal(outs[0][3], outs[1][3])


def test_decode_bad_position_is_refused_on_device(q8):
    import torch
    m, arr, t, tok, pos, logits = build(q8, SMALL, 7, 0)
    tok.fill_(1)
    pos.fill_(SMALL["ctx"])  # one past the cache
    before = [c.clone() for c in t["k_cache"]]
    m.step()
    torch.cuda.synchronize()
    assert int(pos.item()) == SMALL["ctx"] and int(tok.item()) == 1
    for a, b in zip(before, t["k_cache"]):
        assert torch.equal(a, b)
    with pytest.raises(q8.Q8Error, match="position"):
        m.check()
    m.close()


def test_bounded_wait_gives_up_and_is_reported(q8):
    """A pipeline wait on a barrier that nothing arrives on gives up after its poll limit instead of hanging, records
    the timeout in the model's error word, and q8_model_check reports it once (then the word is clear); the model's
    next step is unaffected."""
    import torch
    m, arr, t, tok, pos, logits = build(q8, SMALL, 8, 1)
    m.wait_selftest(64)
    torch.cuda.synchronize()
    with pytest.raises(q8.Q8Error, match="Q8_ETIMEOUT"):
        m.check()
    m.check()  # cleared
    tok.fill_(2)
    pos.fill_(30)
    m.step()
    torch.cuda.synchronize()
    assert int(pos.item()) == 31
    m.check()
    m.close()


@pytest.mark.parametrize("mode", [1, 0, 2])
def test_decode_full_dims_eight_layers(q8, mode):
    """Every dimension of the full configuration (d 2048, 32/4 heads, 128 experts keep 8, vocab 151936, cache 4096)
    with 8 layers, at the last cache position (every cached row attended): logits within tolerance, same token."""
    import torch
    cfg = dict(recipes.DECODE, layers=8)
    m, arr, t, tok, pos, logits = build(q8, cfg, 0, mode)
    om = oracle.ModelArrays(cfg, **arr)
    tok.fill_(0)
    pos.fill_(cfg["ctx"] - 1)
    m.step()
    torch.cuda.synchronize()
    nxt, ora_logits = oracle.decode_step(mode, om, 0, cfg["ctx"] - 1)
    gl = logits.cpu().numpy()
    err = rel_err(gl, ora_logits)
    assert err < TOL[mode], err
    check_token(int(tok.item()), ora_logits, TOL[mode])
    for l in range(cfg["layers"]):
        assert rel_err(t["k_cache"][l].cpu().numpy()[:, -1], om.k_cache[l][:, -1]) < TOL[mode]
    m.close()


def _near_tie(logits, k):
    """The oracle's K-th and (K+1)-th router logits within 1e-5 of the largest magnitude: an expert choice there may
    fall either way (flagged, not compared)."""
    srt = np.sort(np.asarray(logits, np.float64))[::-1]
    return srt[k - 1] - srt[k] < 1e-5 * np.max(np.abs(srt))


@pytest.mark.slow
@pytest.mark.parametrize("mode,form", [(1, "launches"), (0, "launches"), (2, "launches"), (1, "persistent"),
                                       (2, "persistent")])
def test_decode_full_config_layer_by_layer(q8, mode, form):
    """The full 48-layer configuration at the last cache position (every cached row attended), teacher-forced: the
    GPU step exports the residual stream entering every layer, the oracle runs each layer from that same input, and
    each layer's output (and its increment, the attention and mixture sums), its new key and value rows, then the
    final norm, LM head and token from the GPU's last stream, are each within the stated tolerance.  The graph replay
    the benchmark times gives the same logits bit for bit as the traced plain launches.  Both forms of the step: six
    launches a layer and (the int8 modes) all layers as one persistent launch."""
    q8.set_persistent_decode(form == "persistent")
    try:
        _full_config_layer_by_layer(q8, mode, form)
    finally:
        q8.set_persistent_decode(False)


def _full_config_layer_by_layer(q8, mode, form):
    import torch
    cfg = recipes.DECODE
    L, K = cfg["layers"], cfg["k"]
    m, arr, t, tok, pos, logits = build(q8, cfg, 0, mode)
    if form == "persistent" and not m.persistent():
        pytest.skip("the persistent step does not fit this device")
    om = oracle.ModelArrays(cfg, **arr)
    P = cfg["ctx"] - 1
    tok.fill_(0)
    pos.fill_(P)
    hidden = torch.empty(L + 1, cfg["d"], device="cuda")
    m.step_trace(hidden)
    torch.cuda.synchronize()
    hid = hidden.cpu().numpy()
    gl = logits.cpu().numpy().copy()
    gtok = int(tok.item())
    assert int(pos.item()) == cfg["ctx"]
    np.testing.assert_array_equal(hid[0], arr["embed"][0])
    flagged, worst = [], 0.0
    for l in range(L):
        h_ora, rl = oracle.decode_layer(mode, om, l, P, hid[l])
        if _near_tie(rl, K):
            flagged.append(l)
            continue
        err_out = rel_err(hid[l + 1], h_ora)
        err_inc = rel_err(hid[l + 1].astype(np.float64) - hid[l], h_ora.astype(np.float64) - hid[l])
        kc, vc = t["k_cache"][l][:, P].cpu().numpy(), t["v_cache"][l][:, P].cpu().numpy()
        err_k, err_v = rel_err(kc, om.k_cache[l][:, P]), rel_err(vc, om.v_cache[l][:, P])
        worst = max(worst, err_out, err_inc, err_k, err_v)
        assert max(err_out, err_inc, err_k, err_v) < TOL[mode], (l, err_out, err_inc, err_k, err_v)
    assert len(flagged) <= 2, flagged
    nxt, ora_logits = oracle.decode_final(mode, om, hid[L])
    assert rel_err(gl, ora_logits) < TOL[mode], rel_err(gl, ora_logits)
    check_token(gtok, ora_logits, TOL[mode])
    # the captured graph (what the benchmark replays) computes the same step bit for bit
    tok.fill_(0)
    pos.fill_(P)
    m.step()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(logits.cpu().numpy(), gl)
    assert int(tok.item()) == gtok
    print(f"mode {mode} ({form}): worst per-layer relative error {worst:.3e}; near-tie layers {flagged}")
    m.close()


# ---- prefill chunks: R token rows through every layer ---------------------------------------------------------------

def _layer_vs_oracle(mode, om, l, pos, h_in, h_out):
    return layer_vs_oracle(mode, om, l, pos, h_in, h_out, TOL[mode])


def _prefill_vs_oracle(q8, cfg, mode, R, pos0, tokens, seed, cache_layers=None):
    import torch
    m, arr, t, tok, pos, logits = build(q8, cfg, seed, mode)
    om = oracle.ModelArrays(cfg, **arr)
    ws = q8.Workspace(128 << 20)
    pos.fill_(pos0)
    tok.fill_(0)
    toks = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    m.prefill(toks, ws)
    torch.cuda.synchronize()
    for r, tk in enumerate(tokens):  # the oracle: R decode steps fed the same tokens
        nxt, ora_logits = oracle.decode_step(mode, om, tk, pos0 + r)
    gl = logits.cpu().numpy()
    assert rel_err(gl, ora_logits) < TOL[mode], rel_err(gl, ora_logits)
    check_token(int(tok.item()), ora_logits, TOL[mode])
    assert int(pos.item()) == pos0 + R
    for l in (range(cfg["layers"]) if cache_layers is None else cache_layers):  # every row's key and value
        kc, vc = t["k_cache"][l].cpu().numpy(), t["v_cache"][l].cpu().numpy()
        rows = slice(pos0, pos0 + R)
        assert rel_err(kc[:, rows], om.k_cache[l][:, rows]) < TOL[mode]
        assert rel_err(vc[:, rows], om.v_cache[l][:, rows]) < TOL[mode]
    m.check()
    ws.close()
    return m, tok, pos, logits


@pytest.mark.parametrize("attention", ["tensor", "cuda"])
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("cfg,R", [(SMALL, 1), (SMALL, 5), (SMALL, 17), (UNFUSED, 6)], ids=["s1", "s5", "s17", "u6"])
def test_prefill_chunk_matches_oracle(q8, mode, cfg, R, attention):
    """Both forms of the chunk attention (tensor cores with split f16 operands; CUDA cores in f32)."""
    rng = np.random.default_rng(R)
    tokens = [int(v) for v in rng.integers(0, cfg["vocab"], R)]
    q8.set_tensor_core_attention(attention == "tensor")
    try:
        m, tok, pos, logits = _prefill_vs_oracle(q8, cfg, mode, R, 40 if cfg is SMALL else 30, tokens, 11)
    finally:
        q8.set_tensor_core_attention(True)
    m.close()


def test_prefill_chunk_tensor_core_projections_small(q8):
    """The 17-row chunk of the small model with its dense int8 projections (q/k/v and O with its residual) on the
    tensor cores: every layer's cache rows and the logits against the oracle."""
    rng = np.random.default_rng(17)
    tokens = [int(v) for v in rng.integers(0, SMALL["vocab"], 17)]
    q8.set_tensor_core_rows(16)
    try:
        m, tok, pos, logits = _prefill_vs_oracle(q8, SMALL, 1, 17, 40, tokens, 11)
    finally:
        q8.set_tensor_core_rows(-1)
    m.close()


def test_prefill_chunk_same_token_rows_group_experts(q8):
    """Eight copies of one token: every row routes alike at the first layer, so the chunk's expert groups hold all
    rows (the grouped products with their largest groups)."""
    m, tok, pos, logits = _prefill_vs_oracle(q8, SMALL, 1, 8, 20, [5] * 8, 12)
    m.close()


def test_prefill_then_decode_continues(q8):
    """A prefill leaves token and position where the next decode step starts: prefill(tokens[:-1]) then one decode
    step of tokens[-1] gives the oracle's logits after all of them."""
    import torch
    cfg, mode = SMALL, 1
    tokens = [3, 141, 59, 26, 535, 897]
    m, arr, t, tok, pos, logits = build(q8, cfg, 13, mode)
    om = oracle.ModelArrays(cfg, **arr)
    ws = q8.Workspace(64 << 20)
    pos.fill_(50)
    m.prefill(torch.tensor(tokens[:-1], dtype=torch.int32, device="cuda"), ws)
    torch.cuda.synchronize()
    assert int(pos.item()) == 50 + len(tokens) - 1
    tok.fill_(tokens[-1])
    m.step()
    torch.cuda.synchronize()
    for r, tk in enumerate(tokens):
        _, ora_logits = oracle.decode_step(mode, om, tk, 50 + r)
    assert rel_err(logits.cpu().numpy(), ora_logits) < TOL[mode]
    m.check()
    ws.close()
    m.close()


def test_prefill_past_the_cache_is_flagged(q8):
    import torch
    m, arr, t, tok, pos, logits = build(q8, SMALL, 14, 0)
    ws = q8.Workspace(64 << 20)
    pos.fill_(SMALL["ctx"] - 2)  # rows 2 and 3 of 4 fall past the cache
    m.prefill(torch.tensor([1, 2, 3, 4], dtype=torch.int32, device="cuda"), ws)
    torch.cuda.synchronize()
    assert int(pos.item()) == SMALL["ctx"] - 2  # an error leaves the position where it was
    with pytest.raises(q8.Q8Error, match="position"):
        m.check()
    ws.close()
    m.close()


@pytest.mark.parametrize("mode", [1, 2])
def test_prefill_full_width_tensor_core_rows(q8, mode):
    """A 32-row chunk at full layer width with its dense int8 projections (q/k/v and O with its residual) on the
    tensor cores, layer by layer against the oracle (_prefill_per_layer; the int8 modes' words decided by last bits
    make an end-to-end comparison fork)."""
    q8.set_tensor_core_rows(16)
    try:
        worst, flagged, rounded = _prefill_per_layer(q8, mode, 32, 4000, 16, 32)
    finally:
        q8.set_tensor_core_rows(-1)
    print(f"mode {mode}: worst per-layer relative error {worst:.3e}; near-tie rows {flagged}; rounded {rounded}")


def test_prefill_full_width_tensor_core_rows_f32_mode_end_to_end(q8):
    """The same 32-row chunk in the f32 mode (whose projections stay on the CUDA cores), end to end."""
    cfg = dict(recipes.DECODE, layers=2, vocab=1000)
    rng = np.random.default_rng(32)
    tokens = [int(v) for v in rng.integers(0, cfg["vocab"], 32)]
    q8.set_tensor_core_rows(16)
    try:
        m, tok, pos, logits = _prefill_vs_oracle(q8, cfg, 0, 32, 4000, tokens, 16)
    finally:
        q8.set_tensor_core_rows(-1)
    m.close()


@pytest.mark.parametrize("attention", ["tensor", "cuda"])
def test_prefill_full_width_two_layers(q8, attention):
    """The full layer width (d 2048, 32 q / 4 kv heads, 128 experts, top-8, dff 768) on two layers, a chunk of 8 rows
    near the end of a 4096-row cache, against the oracle end to end in the f32 mode, with either form of the chunk
    attention (the int8 modes at this width are checked layer by layer below: an activation word decided by the last
    bits of an input can differ from the oracle's, and downstream layers then follow another, equally valid path)."""
    cfg = dict(recipes.DECODE, layers=2, vocab=1000)
    rng = np.random.default_rng(3)
    tokens = [int(v) for v in rng.integers(0, cfg["vocab"], 8)]
    q8.set_tensor_core_attention(attention == "tensor")
    try:
        m, tok, pos, logits = _prefill_vs_oracle(q8, cfg, 0, 8, 4000, tokens, 15)
    finally:
        q8.set_tensor_core_attention(True)
    m.close()


def _prefill_per_layer(q8, mode, R, P, seed, token_seed):
    """A chunk of R rows at full width on two layers (positions P.., a 4096-row cache), teacher forced: the chunk
    exports the residual rows entering every layer, and the oracle runs each layer for the chunk's rows in order from
    the GPU's own inputs (its cache rows for the chunk come from those inputs too).  Every layer's output rows, their
    increments and the key/value rows it wrote are within the mode's tolerance, against the oracle's result or, in the
    one-word mode, the result with a word on a rounding boundary rounded the other way (_layer_vs_oracle); a row whose
    oracle router held a near tie (the K-th and (K+1)-th logits within 1e-5 of the largest) is left out.  The last
    row's logits follow from the GPU's final residual row.  Returns (worst error, near-tie rows, rounded words)."""
    import torch
    cfg = dict(recipes.DECODE, layers=2, vocab=1000)
    L, D, K = cfg["layers"], cfg["d"], cfg["k"]
    rng = np.random.default_rng(token_seed)
    tokens = [int(v) for v in rng.integers(0, cfg["vocab"], R)]
    m, arr, t, tok, pos, logits = build(q8, cfg, seed, mode)
    ws = q8.Workspace(256 << 20)
    hidden = torch.empty((L + 1, R, D), dtype=torch.float32, device="cuda")
    pos.fill_(P)
    m.prefill_trace(torch.tensor(tokens, dtype=torch.int32, device="cuda"), ws, hidden)
    torch.cuda.synchronize()
    m.check()
    hid = hidden.cpu().numpy()
    gl = logits.cpu().numpy()
    om = oracle.ModelArrays(cfg, **arr)
    for r in range(R):
        np.testing.assert_array_equal(hid[0][r], arr["embed"][tokens[r]])
    flagged, rounded, worst = [], [], 0.0
    for l in range(L):
        kc, vc = t["k_cache"][l].cpu().numpy(), t["v_cache"][l].cpu().numpy()
        for r in range(R):
            rl, err, word = _layer_vs_oracle(mode, om, l, P + r, hid[l][r], hid[l + 1][r])
            err_k = rel_err(kc[:, P + r], om.k_cache[l][:, P + r])
            err_v = rel_err(vc[:, P + r], om.v_cache[l][:, P + r])
            assert max(err_k, err_v) < TOL[mode], (l, r, err_k, err_v)
            if _near_tie(rl, K):
                flagged.append((l, r))
                continue
            if word is not None:
                rounded.append((l, r, word))
            worst = max(worst, err, err_k, err_v)
            assert err < TOL[mode], (l, r, err)
    assert len(flagged) <= 2, flagged
    assert len(rounded) <= max(4, R // 8), rounded
    nxt, ora_logits = oracle.decode_final(mode, om, hid[L][R - 1])
    assert rel_err(gl, ora_logits) < TOL[mode], rel_err(gl, ora_logits)
    ws.close()
    m.close()
    return worst, flagged, rounded


@pytest.mark.parametrize("attention", ["tensor", "cuda"])
@pytest.mark.parametrize("mode", [1, 0, 2])
def test_prefill_per_layer_teacher_forced(q8, mode, attention):
    """20 rows (a full and a partial block of 16 rows) at positions 4000..4019, layer by layer (_prefill_per_layer),
    with either form of the chunk attention."""
    q8.set_tensor_core_attention(attention == "tensor")
    try:
        worst, flagged, rounded = _prefill_per_layer(q8, mode, 20, 4000, 18, 20)
    finally:
        q8.set_tensor_core_attention(True)
    print(f"mode {mode}, {attention} attention: worst per-layer relative error {worst:.3e}; near-tie rows {flagged}; "
          f"words rounded the other way {rounded}")


def test_prefill_attention_forms_agree_full_width(q8):
    """One 64-row chunk at full width (every row block of 16 and every position group of the 4096-row cache in use),
    f32 mode, run with the tensor-core attention and with the CUDA-core attention from the same state: the logits and
    the second layer's cache rows (which depend on the first layer's attention) agree to 1e-5, and the tensor-core
    form's result matches the oracle's decode steps."""
    import torch
    cfg = dict(recipes.DECODE, layers=2, vocab=1000)
    rng = np.random.default_rng(64)
    tokens = [int(v) for v in rng.integers(0, cfg["vocab"], 64)]
    out = {}
    for form in ("tensor", "cuda"):
        q8.set_tensor_core_attention(form == "tensor")
        try:
            m, arr, t, tok, pos, logits = build(q8, cfg, 17, 0)
            ws = q8.Workspace(256 << 20)
            pos.fill_(3000)
            m.prefill(torch.tensor(tokens, dtype=torch.int32, device="cuda"), ws)
            torch.cuda.synchronize()
            m.check()
            out[form] = (logits.cpu().numpy(), t["k_cache"][1][:, 3000:3064].cpu().numpy(),
                         t["v_cache"][1][:, 3000:3064].cpu().numpy())
            ws.close()
            m.close()
        finally:
            q8.set_tensor_core_attention(True)
    for a, b in zip(out["tensor"], out["cuda"]):
        assert rel_err(a, b) < 1e-5, rel_err(a, b)
    om = oracle.ModelArrays(cfg, **arr)
    for r, tk in enumerate(tokens):
        _, ora_logits = oracle.decode_step(0, om, tk, 3000 + r)
    assert rel_err(out["tensor"][0], ora_logits) < TOL[0]

