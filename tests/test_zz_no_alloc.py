"""q8_gemv_noalloc — the projection for callers that cannot allocate device memory when they call it.

Such callers (code inside an allocator's callbacks, loops that forbid allocation after start-up, hosts whose device
memory another runtime has already handed out) cannot create a workspace.  This entry point takes its scratch from an
array the library holds on the device, so the test checks it against q8_gemv (which uses a workspace) on shapes that
do need scratch: a matrix cut along k, and an int8-mode call that quantizes its activation into scratch.  Two calls in
a row each, so the second call starts from whatever the first left in the shared array.  The file is named to run
last, so a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from synth import recipes

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 2e-3}


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("mode,n,k,R,give_xq", [(0, 512, 2048, 1, False), (0, 128, 4096, 3, False),
                                               (1, 128, 4096, 1, False), (1, 1000, 96, 2, True)])
def test_noalloc_matches_workspace_projection(q8, mode, n, k, R, give_xq):
    import torch
    q, s = synth.q8_matrix(n, k, 7, 300 + n % 5)
    x = synth.normal((R, k), 7, recipes.VEC + 301)
    tq, ts = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    tx = torch.from_numpy(x).cuda()
    xq = xs = None
    if give_xq:
        oq, os_ = oracle.quantize(x)
        xq, xs = torch.from_numpy(oq).cuda(), torch.from_numpy(os_).cuda()
    ws = q8.Workspace(64 << 20)
    ref = torch.empty(R, n, device="cuda")
    q8.q8_gemv(tq, ts, mode, ref, x=tx, xq=xq, xs=xs, rows=R, ws=ws)
    torch.cuda.synchronize()
    ref_h = ref.cpu().numpy()
    # the workspace call itself against the oracle, so both sides of the comparison are known good
    if mode == 0:
        ora = np.stack([oracle.gemv_f32act(q, s, x[r]) for r in range(R)])
    else:
        ora = np.stack([oracle.gemv(1, q, s, x[r]) for r in range(R)])
    assert rel_err(ref_h, ora) < TOL[mode]
    W = q8.mat(tq, ts)
    qa = ctypes.byref(q8.q8_act(xq.data_ptr(), xs.data_ptr())) if give_xq else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full((R, n), float("nan"), device="cuda")
        code = q8.lib.q8_gemv_noalloc(ctypes.byref(W), mode, ctypes.c_void_p(tx.data_ptr()), qa, R,
                                      ctypes.c_void_p(y.data_ptr()), stream)
        assert code == 0, q8.last_error()
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.isfinite(got).all()
        assert rel_err(got, ref_h) < TOL[mode], (call, rel_err(got, ref_h))
    ws.close()


def test_noalloc_refuses_calls_past_its_fixed_scratch(q8):
    import torch
    # 64 rows of an 8192 x 4096 matrix in the f32 mode: the partial sums alone are over the fixed size
    n, k, R = 8192, 4096, 64
    tq = torch.zeros(n, k, dtype=torch.int8, device="cuda")
    ts = torch.zeros(n, k // 32, dtype=torch.float32, device="cuda")
    tx = torch.zeros(R, k, device="cuda")
    y = torch.zeros(R, n, device="cuda")
    W = q8.mat(tq, ts)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = q8.lib.q8_gemv_noalloc(ctypes.byref(W), 0, ctypes.c_void_p(tx.data_ptr()), None, R,
                                  ctypes.c_void_p(y.data_ptr()), stream)
    assert code == -5 and "scratch" in q8.last_error()
    torch.cuda.synchronize()
    assert not y.any()  # nothing was launched
