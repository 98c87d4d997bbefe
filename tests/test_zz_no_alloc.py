"""q8_gemv_noalloc — the projection for callers that cannot allocate device memory when they call it.

Such callers (code inside an allocator's callbacks, loops that forbid allocation after start-up, hosts whose device
memory another runtime has already handed out) cannot create a workspace.  This entry point takes its scratch from an
array the library holds on the device, so the test checks it against q8_gemv (which uses a workspace) on shapes that
need scratch: matrices cut along k (one of them because its scales are 4-byte but not 16-byte aligned, which keeps it
off the bulk-copy path), and int8-mode calls that quantize their activation into scratch.  Two calls in a row each,
so the second call starts from whatever the first left in the shared array; neither may allocate device memory.  The
file is named to run last, so a run that stops at the first failure has already run every other test.
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


@pytest.mark.parametrize("mode,n,k,R,give_xq,scale_offset", [(0, 512, 2048, 1, False, 1), (0, 128, 4096, 3, False, 0),
                                                            (1, 128, 4096, 1, False, 0), (1, 1000, 96, 2, True, 0),
                                                            (1, 512, 2048, 1, False, 1)])
def test_noalloc_matches_workspace_projection(q8, mode, n, k, R, give_xq, scale_offset):
    import torch
    q, s = synth.q8_matrix(n, k, 7, 300 + n % 5)
    x = synth.normal((R, k), 7, recipes.VEC + 301)
    tq = torch.from_numpy(q).cuda()
    # scales placed `scale_offset` floats into their buffer: 4-byte aligned, and with an offset of 1 not 16-byte
    # aligned, which sends a one-row call to the projection cut along k (arrival counters in the scratch)
    sbuf = torch.zeros(s.size + 4, dtype=torch.float32, device="cuda")
    ts = sbuf[scale_offset:scale_offset + s.size].view(n, k // 32)
    ts.copy_(torch.from_numpy(s))
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
    ys = [torch.full((R, n), float("nan"), device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    held = torch.cuda.memory_allocated()
    for call in range(2):
        free_before = torch.cuda.mem_get_info()[0]
        code = q8.lib.q8_gemv_noalloc(ctypes.byref(W), mode, ctypes.c_void_p(tx.data_ptr()), qa, R,
                                      ctypes.c_void_p(ys[call].data_ptr()), stream)
        assert code == 0, q8.last_error()
        torch.cuda.synchronize()
        if call == 1:  # the first call may load the kernels' code; the second allocates nothing at all
            assert torch.cuda.mem_get_info()[0] == free_before
        got = ys[call].cpu().numpy()
        assert np.isfinite(got).all()
        assert rel_err(got, ref_h) < TOL[mode], (call, rel_err(got, ref_h))
    assert torch.cuda.memory_allocated() == held
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
