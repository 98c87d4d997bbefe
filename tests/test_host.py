"""Host-side checks that need no GPU: the C-ABI library loads, exports every declared entry point, and refuses bad
arguments by name before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q8():
    import __graft_entry__
    __graft_entry__.build()
    import moe_add_rmsnorm_gb300 as m
    return m


def declared():
    text = open(os.path.join(ROOT, "include", "q8moe.h")).read()
    return re.findall(r"^Q8_API\s+[\w\s\*]*?\b(\w+)\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared())
    for n in ("q8_gemv", "add_rmsnorm_q8", "moe_route_topk", "moe_gate_up", "moe_down_combine", "decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol(q8):
    lib = ctypes.CDLL(q8.LIB_PATH)
    for name in declared():
        assert hasattr(lib, name), name
    assert set(declared()) == set(q8.EXPORTS)


def test_refusals_before_any_launch(q8):
    lib = q8.lib
    W = q8.q8_mat(None, None, 4, 64)
    assert lib.q8_gemv(ctypes.byref(W), 0, None, None, 1, None, None, None) == -1
    assert "y: null" in q8.last_error()
    assert lib.q8_gemv(ctypes.byref(W), 0, None, None, 1, ctypes.c_void_p(256), None, None) == -1
    assert "W" in q8.last_error()
    W = q8.q8_mat(64, 64, 4, 40)  # fake aligned addresses: refused on shape before any use
    y = ctypes.c_void_p(256)
    assert lib.q8_gemv(ctypes.byref(W), 0, ctypes.c_void_p(512), None, 1, y, None, None) == -2
    assert "32-value" in q8.last_error()
    R = q8.q8_mat(64, 64, 128, 2048)
    ids = ctypes.c_void_p(1024)
    assert lib.moe_route_topk(ctypes.byref(R), 0, ctypes.c_void_p(512), None, 1, 33, ids, ids, None, None,
                              ctypes.c_void_p(8), None) == -2
    assert "k 33" in q8.last_error()
    assert lib.moe_route_topk(ctypes.byref(R), 0, ctypes.c_void_p(512), None, 1, 0, ids, ids, None, None,
                              ctypes.c_void_p(8), None) == -2
    Rbig = q8.q8_mat(64, 64, 8193, 2048)
    assert lib.moe_route_topk(ctypes.byref(Rbig), 0, ctypes.c_void_p(512), None, 1, 8, ids, ids, None, None,
                              ctypes.c_void_p(8), None) == -2
    assert "8192" in q8.last_error()
    assert lib.add_rmsnorm_q8(ctypes.c_void_p(512), None, ctypes.c_void_p(512), 1, 2048, ctypes.c_float(-1.0), None,
                              ctypes.c_void_p(512), None, None) == -1
    assert "eps" in q8.last_error()
    d = q8.q8_model_desc()
    d.layers, d.d, d.heads, d.kv_heads, d.head_dim = 1, 2048, 32, 4, 64
    d.experts, d.k, d.dff, d.vocab, d.ctx = 128, 8, 768, 100, 16
    h = ctypes.c_void_p()
    assert lib.q8_model_create(ctypes.byref(d), ctypes.byref(h)) == -2
    assert "head_dim" in q8.last_error()
    assert lib.prefill_chunk(None, ctypes.c_void_p(256), 4, ctypes.c_void_p(8), None) == -1
    assert "model" in q8.last_error()
    assert lib.decode_step(None, None) == -1


def test_tensor_core_thresholds_refuse_bad_row_counts(q8):
    lib = q8.lib
    for setter in (lib.q8_set_tensor_core_rows, lib.q8_set_grouped_tensor_core_rows):
        for bad in (1, 15, 65, -16):
            assert setter(bad) == -1
            assert "0 (off) or 16 to 64" in q8.last_error()
    assert lib.q8_set_grouped_tensor_core_rows(16) == 0
    assert lib.q8_set_grouped_tensor_core_rows(32) == 0  # the default again
    assert lib.q8_set_tensor_core_rows(0) == 0
    assert lib.q8_set_tensor_core_rows(-1) == 0  # the default again


def test_on_off_switches_refuse_other_values(q8):
    lib = q8.lib
    for setter in (lib.q8_set_persistent_decode, lib.q8_set_tensor_core_attention):
        for bad in (-1, 2, 7):
            assert setter(bad) == -1
            assert "0 or 1" in q8.last_error()
    assert lib.q8_set_persistent_decode(0) == 0  # the default again
    assert lib.q8_set_tensor_core_attention(1) == 0  # the default again
    assert lib.q8_model_persistent(None) == 0
    for bad in (-1, 1):
        assert lib.q8_set_streamed_batch_attention(bad) == -1
        assert "0 or at least 2" in q8.last_error()
    assert lib.q8_set_streamed_batch_attention(8) == 0  # the default again


_RANK = r"""
import json, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank={rank}, world_size=2)
import bench
s = bench.slowest({sec}, 2, "cpu")
print(json.dumps({{"rank": {rank}, "sec": s, "rate": bench.job_rate(10, 2, s)}}))
dist.destroy_process_group()
"""


def test_replicas_report_the_slowest_rank():
    """Two gloo ranks on the host: the job's time is the slower rank's on both, and the rate counts both ranks' units
    (the aggregation bench.py applies to its replicas)."""
    import json
    import socket
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    procs = [subprocess.Popen([sys.executable, "-c", _RANK.format(root=root, port=port, rank=r, sec=sec)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r, sec in ((0, 0.5), (1, 0.8))]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    for r in res:
        assert r["sec"] == 0.8
        assert abs(r["rate"] - 2 * 10 / 0.8) < 1e-12


def test_token_check_follows_the_tolerance():
    """The GPU tests' greedy-token check: outside the tolerance band the token must be the oracle's arg-max; inside it
    (the top two closer than the logits' error bound allows to separate) either close candidate passes, and nothing
    else does."""
    from layer_parity import check_token
    lg = np.array([10.0, 9.99, 0.0, -3.0])  # top two 0.01 apart; the band at 2e-3 is 2 * 2e-3 * 10 = 0.04
    check_token(0, lg, 2e-3)
    check_token(1, lg, 2e-3)
    with pytest.raises(AssertionError):
        check_token(2, lg, 2e-3)
    with pytest.raises(AssertionError):
        check_token(1, lg, 1e-4)  # band 2e-3 < 0.01: the gap decides
    check_token(0, lg, 1e-4)

