"""Decode-step throughput of the Q8_0 mixture-of-experts model on GB300.

Workload: the full decode step of 48 layers (d=2048, 32 query / 4 key-value heads of 128, RoPE theta 1e6, f32 KV cache
of 4096 positions, 128 experts keep 8 of dff 768, vocab 151936 Q8_0 LM head, greedy arg-max), random-init Q8_0 weights
from the seeded generator.  One step = one token = one replay of the captured CUDA graph; the position advances each
step (a growing cache, tg-style) and ends at the last cache position.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="int8", choices=["int8", "f32", "int8x2"])
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--roofline-only", action="store_true",
                    help="only the dominant kernel's timing loop (for a profiler capture of that kernel)")
    ap.add_argument("--decode-only", action="store_true",
                    help="only the warm-up and timed decode steps (for profiler launch lists); prints tokens/s")
    ap.add_argument("--chunk-only", type=int, default=0, metavar="R",
                    help="only the R-row chunk timing through the mixture block (for a profiler capture of its kernels)")
    ap.add_argument("--correlated", action="store_true", help="with --chunk-only: rows that share their experts")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="R",
                    help="only the R-row prefill timing through the model (for a profiler capture of its kernels)")
    ap.add_argument("--batch-only", type=int, default=0, metavar="B",
                    help="only the batch form's timing with B sequences (for a profiler capture of its kernels)")
    ap.add_argument("--tensor-core-rows", type=int, default=None, metavar="N",
                    help="dense int8 projections of N..64 rows on the tensor cores (-1: automatic, the library default; 0: off)")
    ap.add_argument("--grouped-tensor-core-rows", type=int, default=None, metavar="N",
                    help="int8 expert groups of N..64 rows on the tensor cores (0: off; the library's default is 32)")
    ap.add_argument("--persistent", type=int, default=None, choices=[0, 1],
                    help="one-sequence int8 decode steps as one persistent launch for all layers (1) or six launches "
                         "a layer (0, the library's default)")
    ap.add_argument("--tensor-core-attention", type=int, default=None, choices=[0, 1],
                    help="prefill chunks' attention on the tensor cores (1, the library's default) or CUDA cores (0)")
    ap.add_argument("--streamed-batch-attention", type=int, default=None, metavar="B",
                    help="batch steps of B or more sequences attend in the streamed form (0: never; the library's "
                         "default is 8)")
    ap.add_argument("--configs-only", action="store_true",
                    help="only the single-operation configurations (projection, attention-side projections, mixture)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


METRIC = "decode tokens/s and Q8_0 weight-stream GB/s (% of GB300 HBM peak), 1 GPU"


MODE_NAMES = {0: "f32-activation/f64-sum", 1: "int8-activation", 2: "two-word int8-activation"}


def workload_config(cfg, mode, world):
    """The `config` object of both arms' lines (the same workload, whichever implementation runs it)."""
    return {"workload": f"decode step, {cfg['layers']} layers d=2048 32q/4kv hd128 E=128 K=8 dff=768 vocab=151936 "
                        "ctx=4096 (full decode configuration), tg-style growing cache",
            "mode": MODE_NAMES[int(mode)],
            "l2": "inputs larger than L2: every step streams 3.42 GB of weights and ~0.8 GB of cache",
            "parallelism": "replicas" if world > 1 else "1 GPU"}


def slowest(sec, world, device):
    """The whole job's time for `world` replicas: the slowest rank's (max over ranks; one rank: its own)."""
    if world <= 1:
        return sec
    import torch
    import torch.distributed as dist
    t = torch.tensor([sec], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, sec):
    """Units all ranks processed per second of the job's time."""
    return world * units_per_rank / sec


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """nvidia-smi samples of one GPU during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_model_tensors(cfg, seed=0):
    """Host arrays in pinned memory (from the seeded generator) and their device copies."""
    import numpy as np
    import torch
    from synth import recipes

    dtypes = {np.dtype(np.int8): torch.int8, np.dtype(np.float32): torch.float32}
    host = recipes.decode_model(cfg, seed, alloc=lambda shape, dt: torch.empty(shape, dtype=dtypes[np.dtype(dt)],
                                                                               pin_memory=True),
                                ptr=lambda t: t.data_ptr())

    def up(v):
        if isinstance(v, list):
            return [up(e) for e in v]
        if isinstance(v, tuple):
            return tuple(up(e) for e in v)
        return v.cuda(non_blocking=True)

    dev = {k: up(v) for k, v in host.items()}
    torch.cuda.synchronize()
    return host, dev


# DRAM traffic per launch of the roofline kernel (gate_row_kernel through moe_gate_up, int8 mode), from the ncu capture
# summarised in profiles/moe_gate_up_roofline_kernel_int8.md; valid only while the kernel's sources are the captured ones.
ROOFLINE_TRAFFIC = {"bytes": 28344491, "sources": ["moe_add_rmsnorm_gb300/csrc/moe_row.cu",
                                                   "moe_add_rmsnorm_gb300/csrc/common.cuh"],
                    "sha256_16": "565a6e58b25e8cbb", "profile": "profiles/moe_gate_up_roofline_kernel_int8.md"}


def roofline_traffic(mode_int8):
    """The captured traffic per launch, or None when the kernel changed since the capture (or in the f32 mode)."""
    import hashlib
    if not mode_int8:
        return None
    h = hashlib.sha256()
    for f in ROOFLINE_TRAFFIC["sources"]:
        h.update(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), f), "rb").read())
    return ROOFLINE_TRAFFIC["bytes"] if h.hexdigest()[:16] == ROOFLINE_TRAFFIC["sha256_16"] else None


def time_dominant_kernel(q8, cfg, dev, mode, reps, stream):
    """The mixture's gate-up kernel at the decode shape (8 experts x 768 gate and 768 up rows of 2048), launched over
    the layers' own stacked matrices in turn (each launch reads weights no earlier launch brought into L2), the L
    launches captured in one CUDA graph, timed with CUDA events on its stream.  Returns (average seconds per launch, algorithmic bytes per launch)."""
    import torch
    L, d, dff, K, E = cfg["layers"], cfg["d"], cfg["dff"], cfg["k"], cfg["experts"]
    ws = q8.Workspace(64 << 20)
    s = torch.cuda.ExternalStream(stream)
    with torch.cuda.stream(s):
        gen = torch.Generator(device="cuda")
        gen.manual_seed(0)
        x = torch.randn(1, d, device="cuda", generator=gen)
        xq = torch.empty(1, d, dtype=torch.int8, device="cuda")
        xs = torch.empty(1, d // 32, dtype=torch.float32, device="cuda")
        q8.q8_quantize(x, xq, xs, stream=stream)
        ids = torch.stack([torch.randperm(E, device="cuda", generator=gen)[:K] for _ in range(L)]).to(torch.int32)
        h = torch.empty(K, dff, device="cuda")

        def one(l):
            g, u = dev["gate"][l], dev["up"][l]
            if mode == 1:
                q8.moe_gate_up(*g, *u, dff, 1, K, ids[l], h, xq=xq, xs=xs, ws=ws, stream=stream)
            else:
                q8.moe_gate_up(*g, *u, dff, 0, K, ids[l], h, x=x, ws=ws, stream=stream)

        for l in range(min(L, 4)):
            one(l)
        # the L launches captured in one graph, so that host calls put no gaps between them
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for l in range(L):
                one(l)
        g.replay()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.synchronize()
        start.record(s)
        for _ in range(reps):
            g.replay()
        end.record(s)
        end.synchronize()
        n = reps * L
        del g
    ws.close()
    sec = start.elapsed_time(end) / 1e3 / n
    return sec, K * 2 * dff * d * 9 // 8


def oracle_model(cfg, host):
    """The oracle's view of the benchmark's host arrays (its own copies of the caches, which a step writes)."""
    import oracle

    def np_(v):
        if isinstance(v, list):
            return [np_(e) for e in v]
        if isinstance(v, tuple):
            return tuple(np_(e) for e in v)
        return v.numpy() if hasattr(v, "numpy") else v

    arr = {k: np_(v) for k, v in host.items()}
    arr["k_cache"] = [c.copy() for c in arr["k_cache"]]
    arr["v_cache"] = [c.copy() for c in arr["v_cache"]]
    return oracle.ModelArrays(cfg, **arr)


def cpu_baseline_oracle(cfg, host, mode, tok, pos, runs=3):
    """The oracle's whole decode step for one token on this host: single-threaded, and on every host core (threads
    over independent rows and heads; the same results).  Median of `runs` steps each; weights generated beforehand."""
    import oracle
    om = oracle_model(cfg, host)
    cores = oracle.host_cores()
    out = {}
    for name, threads in (("single_thread", 1), ("all_cores", cores)):
        used = oracle.set_threads(threads)
        times = []
        for _ in range(runs):
            t0 = time.perf_counter()
            oracle.decode_step(mode, om, tok, pos)
            times.append(time.perf_counter() - t0)
        out[name] = {"tokens_per_s": 1.0 / statistics.median(times), "threads": used,
                     "median_s": statistics.median(times), "runs": runs}
    oracle.set_threads(1)
    return out, cores


def run_reference(args):
    """The reference arm: the CPU oracle (the only other implementation of what the pages define) on every host core,
    one whole decode step (48 layers, LM head, greedy token) per step, at the same growing positions as the GPU arm,
    from the same seeded weights (generated before the timing)."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from synth import recipes
    cfg = dict(recipes.DECODE, layers=args.layers)
    mode = {"int8": 1, "f32": 0, "int8x2": 2}[args.mode]
    host = recipes.decode_model(cfg, seed=0)
    om = oracle_model(cfg, host)
    threads = oracle.set_threads(oracle.host_cores())
    total = args.warmup + args.steps
    start_pos = cfg["ctx"] - total
    times = []
    tok = 0
    for step in range(total):
        t0 = time.perf_counter()
        tok, _ = oracle.decode_step(mode, om, tok, start_pos + step)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    sec = float(np.sum(times))
    value = args.steps / sec
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8" if mode else "f32", "data": "synthetic",
        "config": workload_config(cfg, mode, 1),
        "positions": [start_pos + args.warmup, cfg["ctx"] - 1],
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "host_cores": oracle.host_cores(),
                         "kind": "oracle",
                         "sample": f"{args.steps} whole decode steps ({cfg['layers']} layers, LM head, greedy token) at "
                                   f"positions {start_pos + args.warmup}..{cfg['ctx'] - 1}, f64 C oracle on {threads} "
                                   "threads, each step timed whole"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    oracle.set_threads(1)
    print(json.dumps(line), flush=True)


def _graph_time(stream, body, n, reps):
    """`body(i)` for i < n captured in one CUDA graph, replayed once to warm up and then `reps` times between CUDA events
    on `stream`; returns seconds per body call."""
    import torch
    s = torch.cuda.ExternalStream(stream)
    with torch.cuda.stream(s):
        for i in range(min(n, 2)):
            body(i)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                body(i)
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.synchronize()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
        e1.synchronize()
        del g
    return e0.elapsed_time(e1) / 1e3 / (reps * n)


def time_configs(q8, cfg, dev, stream, peak, reps=4):
    """The single-operation configurations, each as a user calls it through the C ABI, captured in CUDA graphs and
    timed with CUDA events; `cold` walks over copies or layers whose weights together exceed L2 several times (each
    call reads weights no recent call touched), `hot` repeats one call whose weights stay in L2.
      config 0: one Q8_0 projection 1024 x 1024, batch 1, both numerics (int8 mode: the activation quantized once
                beforehand, as a producer's epilogue leaves it)
      config 1: add_rmsnorm_q8 feeding the q, k and v projections (2048 -> 4096, 512, 512), and the o projection
                (4096 -> 2048) of a fresh activation: the dense attention-side projections of one layer
      config 2: the mixture block for one token row: moe_route_topk, moe_gate_up, moe_down_combine (router and 8 of 128
                experts)"""
    import torch
    import synth
    from synth import recipes
    L, d = cfg["layers"], cfg["d"]
    s = torch.cuda.ExternalStream(stream)
    ws = q8.Workspace(64 << 20)
    out = {}

    def entry(sec, nbytes, **kw):
        gbs = nbytes / sec / 1e9
        return dict(us=sec * 1e6, weight_gbs=gbs, frac_of_peak=gbs / peak, **kw)

    with torch.cuda.stream(s):
        # ---- config 0 ----
        n = k = 1024
        q0, s0 = synth.q8_matrix(n, k, 0, recipes.MAT)
        x0 = torch.from_numpy(recipes.activations(1, k, 0, 0)).cuda()
        nrep = 448  # 448 x 1.18 MB = 528 MB of copies, over four times the L2
        qrep = torch.from_numpy(q0).cuda().unsqueeze(0).repeat(nrep, 1, 1)
        srep = torch.from_numpy(s0).cuda().unsqueeze(0).repeat(nrep, 1, 1)
        xq0 = torch.empty(1, k, dtype=torch.int8, device="cuda")
        xs0 = torch.empty(1, k // 32, dtype=torch.float32, device="cuda")
        q8.q8_quantize(x0, xq0, xs0, stream=stream)
        y0 = torch.empty(1, n, device="cuda")
        nbytes0 = n * k * 9 // 8
        c0 = {}
        for mode, name in ((q8.F32ACT_F64SUM, "f32-activation/f64-sum"), (q8.INT8ACT, "int8-activation")):
            def gemv(i, mode=mode):
                if mode == q8.INT8ACT:
                    q8.q8_gemv(qrep[i], srep[i], mode, y0, xq=xq0, xs=xs0, ws=ws, stream=stream)
                else:
                    q8.q8_gemv(qrep[i], srep[i], mode, y0, x=x0, ws=ws, stream=stream)
            c0[name] = {"cold": entry(_graph_time(stream, gemv, nrep, reps), nbytes0),
                        "hot": entry(_graph_time(stream, lambda i: gemv(0), nrep, reps), nbytes0)}
        out["config0"] = {"what": "Q8_0 projection 1024 x 1024, batch 1 (weights 1,179,648 B)", **c0}
        del qrep, srep
        # ---- config 1 ----
        H, KV, HD = cfg["heads"], cfg["kv_heads"], cfg["hd"]
        a1 = torch.from_numpy(recipes.activations(1, d, 0, 10)).cuda()
        b1 = torch.from_numpy(recipes.activations(1, d, 0, 11)).cuda()
        xo = torch.from_numpy(recipes.activations(1, H * HD, 0, 12)).cuda()
        sum1 = torch.empty(1, d, device="cuda")
        x1 = torch.empty(1, d, device="cuda")
        xq1 = torch.empty(1, d, dtype=torch.int8, device="cuda")
        xs1 = torch.empty(1, d // 32, dtype=torch.float32, device="cuda")
        xqo = torch.empty(1, H * HD, dtype=torch.int8, device="cuda")
        xso = torch.empty(1, H * HD // 32, dtype=torch.float32, device="cuda")
        q8.q8_quantize(xo, xqo, xso, stream=stream)
        yq, yk, yv = (torch.empty(1, m, device="cuda") for m in (H * HD, KV * HD, KV * HD))
        yo = torch.empty(1, d, device="cuda")
        nbytes1 = ((H * HD + 2 * KV * HD) * d + d * H * HD) * 9 // 8
        c1 = {}
        for mode, name in ((q8.INT8ACT, "int8-activation"), (q8.F32ACT_F64SUM, "f32-activation/f64-sum")):
            def attn_side(l, mode=mode):
                if mode == q8.INT8ACT:
                    q8.add_rmsnorm_q8(a1, b1, dev["attn_norm"][l], cfg["eps"], sum_out=sum1, yq=xq1, ys=xs1,
                                      stream=stream)
                    for w, y in (("wq", yq), ("wk", yk), ("wv", yv)):
                        q8.q8_gemv(*dev[w][l], mode, y, xq=xq1, xs=xs1, ws=ws, stream=stream)
                    q8.q8_gemv(*dev["wo"][l], mode, yo, xq=xqo, xs=xso, ws=ws, stream=stream)
                else:
                    q8.add_rmsnorm_q8(a1, b1, dev["attn_norm"][l], cfg["eps"], sum_out=sum1, y_out=x1, stream=stream)
                    for w, y in (("wq", yq), ("wk", yk), ("wv", yv)):
                        q8.q8_gemv(*dev[w][l], mode, y, x=x1, ws=ws, stream=stream)
                    q8.q8_gemv(*dev["wo"][l], mode, yo, x=xo, ws=ws, stream=stream)
            c1[name] = {"cold": entry(_graph_time(stream, attn_side, L, reps), nbytes1, launches=5),
                        "hot": entry(_graph_time(stream, lambda i: attn_side(0), L, reps), nbytes1, launches=5)}
        out["config1"] = {"what": "add_rmsnorm_q8 -> q/k/v projections, o projection at d = 2048 (weights "
                                  f"{nbytes1:,} B); cold = the 48 layers' matrices in turn", **c1}
        # ---- config 2 ----
        E, K, dff = cfg["experts"], cfg["k"], cfg["dff"]
        x2 = torch.from_numpy(recipes.activations(1, d, 0, 20)).cuda()
        r2 = torch.from_numpy(recipes.activations(1, d, 0, 21)).cuda()
        xq2 = torch.empty(1, d, dtype=torch.int8, device="cuda")
        xs2 = torch.empty(1, d // 32, dtype=torch.float32, device="cuda")
        q8.q8_quantize(x2, xq2, xs2, stream=stream)
        ids = torch.empty(1, K, dtype=torch.int32, device="cuda")
        gates = torch.empty(1, K, device="cuda")
        h = torch.empty(K, dff, device="cuda")
        hq = torch.empty(K, dff, dtype=torch.int8, device="cuda")
        hs = torch.empty(K, dff // 32, device="cuda")
        y2 = torch.empty(1, d, device="cuda")
        nbytes2 = (E * d + K * 3 * dff * d) * 9 // 8
        c2 = {}
        for mode, name in ((q8.INT8ACT, "int8-activation"), (q8.F32ACT_F64SUM, "f32-activation/f64-sum")):
            def block(l, mode=mode):
                if mode == q8.INT8ACT:
                    q8.moe_route_topk(*dev["router"][l], mode, K, ids, gates, xq=xq2, xs=xs2, ws=ws, stream=stream)
                    q8.moe_gate_up(*dev["gate"][l], *dev["up"][l], dff, mode, K, ids, h, xq=xq2, xs=xs2, hq=hq, hs=hs,
                                   ws=ws, stream=stream)
                    q8.moe_down_combine(*dev["down"][l], d, mode, K, ids, gates, y2, h=h, hq=hq, hs=hs, residual=r2,
                                        ws=ws, stream=stream)
                else:
                    q8.moe_route_topk(*dev["router"][l], mode, K, ids, gates, x=x2, ws=ws, stream=stream)
                    q8.moe_gate_up(*dev["gate"][l], *dev["up"][l], dff, mode, K, ids, h, x=x2, ws=ws, stream=stream)
                    q8.moe_down_combine(*dev["down"][l], d, mode, K, ids, gates, y2, h=h, residual=r2, ws=ws,
                                        stream=stream)
            c2[name] = {"cold": entry(_graph_time(stream, block, L, reps), nbytes2, launches=3),
                        "hot": entry(_graph_time(stream, lambda i: block(0), L, reps), nbytes2, launches=3)}
        out["config2"] = {"what": "mixture block, one token row: route + top-8 of 128, gate-up SwiGLU, down-and-combine "
                                  f"(weights touched {nbytes2:,} B); cold = the 48 layers' experts in turn", **c2}
    ws.close()
    return out


def time_chunks(q8, cfg, dev, stream, reps=4, correlated=False, rows=(2, 4, 8, 16, 32, 64)):
    """Chunks of R token rows through the mixture block in the int8 mode: quantize the rows, route them with the
    expert grouping, gate-up, down-and-combine onto a residual; each chunk uses another layer's router and experts (8
    layers in turn, so the experts come from HBM), one CUDA graph of 8 chunks per R, replayed `reps` times and timed
    with CUDA events.  tokens/s = R / time per chunk; the Q8_0 bytes counted per chunk are the router's plus those of
    the experts the routing touched (unique experts read from the grouping).  `correlated`: rows x0 + 0.01 N(0,1),
    so all rows share their experts (the groups the tensor-core products take)."""
    import torch
    L, d, dff, K, E = cfg["layers"], cfg["d"], cfg["dff"], cfg["k"], cfg["experts"]
    G = min(L, 8)
    ws = q8.Workspace(256 << 20)
    s = torch.cuda.ExternalStream(stream)
    expert_bytes = 3 * dff * d * 9 // 8
    router_bytes = E * d * 9 // 8
    out = []
    for R in rows:
        with torch.cuda.stream(s):
            gen = torch.Generator(device="cuda")
            gen.manual_seed(1000 + R)
            if correlated:
                x = torch.randn(1, d, device="cuda", generator=gen) + 0.01 * torch.randn(R, d, device="cuda",
                                                                                        generator=gen)
            else:
                x = torch.randn(R, d, device="cuda", generator=gen)
            res = torch.randn(R, d, device="cuda", generator=gen)
            xq = torch.empty(R, d, dtype=torch.int8, device="cuda")
            xs = torch.empty(R, d // 32, dtype=torch.float32, device="cuda")
            ids = torch.empty(R, K, dtype=torch.int32, device="cuda")
            gates = torch.empty(R, K, dtype=torch.float32, device="cuda")
            logits = torch.empty(R, E, dtype=torch.float32, device="cuda")
            pt = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                  torch.empty(R * K, dtype=torch.int32, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda")]
            plan = q8.plan_struct(*pt) if R > 1 else None
            h = torch.empty(R * K, dff, device="cuda")
            hq = torch.empty(R * K, dff, dtype=torch.int8, device="cuda")
            hs = torch.empty(R * K, dff // 32, dtype=torch.float32, device="cuda")
            y = torch.empty(R, d, device="cuda")

            def step(l):
                q8.q8_quantize(x, xq, xs, stream=stream)
                q8.moe_route_topk(*dev["router"][l], 1, K, ids, gates, xq=xq, xs=xs, rows=R, logits=logits, plan=plan,
                                  ws=ws, stream=stream)
                q8.moe_gate_up(*dev["gate"][l], *dev["up"][l], dff, 1, K, ids, h, xq=xq, xs=xs, hq=hq, hs=hs, rows=R,
                               plan=plan, ws=ws, stream=stream)
                q8.moe_down_combine(*dev["down"][l], d, 1, K, ids, gates, y, h=h, hq=hq, hs=hs, rows=R, plan=plan,
                                    residual=res, ws=ws, stream=stream)

            uniq = []
            for l in range(G):
                step(l)
                s.synchronize()
                uniq.append(len(set(ids.cpu().flatten().tolist())))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for l in range(G):
                    step(l)
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.synchronize()
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
            e1.synchronize()
            t = e0.elapsed_time(e1) / 1e3 / (reps * G)
            u = sum(uniq) / len(uniq)
            out.append({"rows": R, "tokens_per_s": R / t, "us_per_chunk": t * 1e6, "unique_experts": u,
                        "weight_gbs": (router_bytes + u * expert_bytes) / t / 1e9})
            del g
    ws.close()
    return out


def time_prefill(q8, model, cfg, tok, pos, stream, rows=(16, 64), reps=3):
    """Prefill chunks of R token rows through the whole model (every layer, the last row's LM head and token),
    starting at position ctx - 128 - R, timed with CUDA events around `reps` calls (plain launches, no graph); the
    caches' rows are rewritten each call.  tokens/s = R / time per chunk; weight bytes per chunk count every dense
    matrix once, the router, and the experts the chunk's routing touched at every layer (estimated from uniform routing
    as E * (1 - (1 - K/E)^R))."""
    import torch
    L, d, E, K, dff = cfg["layers"], cfg["d"], cfg["experts"], cfg["k"], cfg["dff"]
    H, KV, HD = cfg["heads"], cfg["kv_heads"], cfg["hd"]
    dense = (H * HD + 2 * KV * HD) * d + d * H * HD + E * d
    expert = 3 * dff * d
    ws = q8.Workspace(512 << 20)
    s = torch.cuda.ExternalStream(stream)
    out = []
    with torch.cuda.stream(s):
        gen = torch.Generator(device="cuda")
        gen.manual_seed(7)
        for R in rows:
            toks = torch.randint(0, cfg["vocab"], (R,), dtype=torch.int32, device="cuda", generator=gen)
            p0 = cfg["ctx"] - 128 - R
            pos.fill_(p0)
            model.prefill(toks, ws, stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.synchronize()
            e0.record(s)
            for _ in range(reps):
                pos.fill_(p0)
                model.prefill(toks, ws, stream)
            e1.record(s)
            e1.synchronize()
            t = e0.elapsed_time(e1) / 1e3 / reps
            u = E * (1.0 - (1.0 - K / E) ** R)
            wbytes = L * (dense + u * expert) * 9 // 8 + cfg["vocab"] * d * 9 // 8
            out.append({"rows": R, "tokens_per_s": R / t, "ms_per_chunk": t * 1e3, "weight_gbs": wbytes / t / 1e9,
                        "unique_experts_per_layer_est": u})
    ws.close()
    return out


def time_batch(q8, cfg, dev, stream, mode, batches=(2, 4, 8, 16, 32, 64), steps=8, warmup=3):
    """The batch form: B sequences per step through the whole model (one captured graph), each with its own f32 cache
    of the full length (seeded N(0,1), generated on the device) at positions ctx - steps - warmup .. ctx - 1.
    tokens/s = B / time per step; weight bytes per step count every dense matrix and the LM head once and the experts
    the sequences' routing touched at every layer (estimated from uniform routing as E (1 - (1 - K/E)^B))."""
    import torch
    L, d, E, K, dff = cfg["layers"], cfg["d"], cfg["experts"], cfg["k"], cfg["dff"]
    H, KV, HD, ctx = cfg["heads"], cfg["kv_heads"], cfg["hd"], cfg["ctx"]
    dense = (H * HD + 2 * KV * HD) * d + d * H * HD + E * d
    expert = 3 * dff * d
    s = torch.cuda.ExternalStream(stream)
    out = []
    for B in batches:
        with torch.cuda.stream(s):
            gen = torch.Generator(device="cuda")
            gen.manual_seed(100 + B)
            t = dict(dev)
            t["k_cache"] = [torch.randn(B, KV, ctx, HD, device="cuda", generator=gen) for _ in range(L)]
            t["v_cache"] = [torch.randn(B, KV, ctx, HD, device="cuda", generator=gen) for _ in range(L)]
            tok = torch.randint(0, cfg["vocab"], (B,), dtype=torch.int32, device="cuda", generator=gen)
            pos = torch.full((B,), ctx - steps - warmup, dtype=torch.int32, device="cuda")
            logits = torch.empty(B, cfg["vocab"], device="cuda")
            m = q8.Model(dict(cfg, batch=B), t, mode, tok, pos, logits)
            for _ in range(warmup):
                m.step(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.synchronize()
            e0.record(s)
            for _ in range(steps):
                m.step(stream)
            e1.record(s)
            e1.synchronize()
            m.check(stream)
            sec = e0.elapsed_time(e1) / 1e3 / steps
            u = E * (1.0 - (1.0 - K / E) ** B)
            wbytes = (L * (dense + u * expert) + cfg["vocab"] * d) * 9 // 8
            # every sequence reads its key and value rows 0..pos at every layer (f32), the timed steps' mean length
            cbytes = B * L * KV * 2 * HD * 4 * (ctx - (steps - 1) / 2)
            out.append({"batch": B, "tokens_per_s": B / sec, "ms_per_step": sec * 1e3, "weight_gbs": wbytes / sec / 1e9,
                        "cache_gbs": cbytes / sec / 1e9, "hbm_gbs": (wbytes + cbytes) / sec / 1e9,
                        "unique_experts_per_layer_est": u, "launches_per_step": m.launches_per_step()})
            m.close()
            del t, m
            torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import numpy as np
    import torch
    import moe_add_rmsnorm_gb300 as q8
    from synth import recipes

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    cfg = dict(recipes.DECODE, layers=args.layers)
    mode = {"int8": q8.INT8ACT, "f32": q8.F32ACT_F64SUM, "int8x2": q8.INT8ACT2}[args.mode]
    host, dev = make_model_tensors(cfg, seed=0)
    total = args.warmup + args.steps
    start_pos = cfg["ctx"] - total
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.full((1,), start_pos, dtype=torch.int32, device="cuda")
    logits = torch.empty(cfg["vocab"], device="cuda")
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    if args.tensor_core_rows is not None:
        q8.set_tensor_core_rows(args.tensor_core_rows)
    if args.grouped_tensor_core_rows is not None:
        q8.set_grouped_tensor_core_rows(args.grouped_tensor_core_rows)
    if args.tensor_core_attention is not None:
        q8.set_tensor_core_attention(bool(args.tensor_core_attention))
    if args.persistent is not None:
        q8.set_persistent_decode(bool(args.persistent))
    if args.streamed_batch_attention is not None:
        q8.set_streamed_batch_attention(args.streamed_batch_attention)
    if args.chunk_only:
        res = time_chunks(q8, cfg, dev, sh, reps=max(1, args.steps), correlated=args.correlated,
                          rows=(args.chunk_only,))
        print(json.dumps({"chunk_only": True, "correlated": args.correlated, **res[0]}), flush=True)
        return
    if args.roofline_only:
        dom_sec, dom_bytes = time_dominant_kernel(q8, cfg, dev, mode, reps=args.steps, stream=sh)
        print(json.dumps({"roofline_only": True, "us_per_launch": dom_sec * 1e6, "algorithmic_bytes": dom_bytes,
                          "gbs": dom_bytes / dom_sec / 1e9}), flush=True)
        return
    if args.batch_only:
        res = time_batch(q8, cfg, dev, sh, mode, batches=(args.batch_only,), steps=max(1, args.steps),
                         warmup=max(1, args.warmup))
        print(json.dumps({"batch_only": True, **res[0]}), flush=True)
        return
    if args.configs_only:
        print(json.dumps({"configs_only": True, **time_configs(q8, cfg, dev, sh, peaks()[0],
                                                                reps=max(1, args.steps))}), flush=True)
        return
    model = q8.Model(cfg, dev, mode, tok, pos, logits)
    if args.prefill_only:
        res = time_prefill(q8, model, cfg, tok, pos, sh, rows=(args.prefill_only,), reps=max(1, args.steps))
        print(json.dumps({"prefill_only": True, **res[0]}), flush=True)
        model.close()
        return

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # device-timed region: inputs resident in HBM, one graph replay per token
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            model.step(sh)
        stream.synchronize()
        barrier()
        clocks = Clocks(local)
        clocks.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            model.step(sh)
        e1.record(stream)
        e1.synchronize()
        clk = clocks.stop()
        torch.cuda.synchronize()
        barrier()
    sec = slowest(e0.elapsed_time(e1) / 1e3, world, "cuda")
    model.check(sh)
    value = job_rate(args.steps, world, sec)
    ms_per_step = sec / args.steps * 1e3
    if args.decode_only:
        if rank == 0:
            print(json.dumps({"decode_only": True, "tokens_per_s": value, "ms_per_step": ms_per_step,
                              "launches_per_step": model.launches_per_step(), "layers": cfg["layers"]}), flush=True)
        model.close()
        return

    # end to end: each token's inputs (token, position) copied from pinned host memory, the next token read back
    pin_in = torch.zeros(2, dtype=torch.int32).pin_memory()
    pin_out = torch.zeros(1, dtype=torch.int32).pin_memory()
    e2e_steps = min(args.steps, 64)
    with torch.cuda.stream(stream):
        stream.synchronize()
        t0 = time.perf_counter()
        cur = 0
        for i in range(e2e_steps):
            pin_in[0] = cur
            pin_in[1] = cfg["ctx"] - e2e_steps + i
            tok.copy_(pin_in[0:1], non_blocking=True)
            pos.copy_(pin_in[1:2], non_blocking=True)
            model.step(sh)
            pin_out.copy_(tok, non_blocking=True)
            stream.synchronize()
            cur = int(pin_out[0])
        e2e_sec = slowest(time.perf_counter() - t0, world, "cuda")
    e2e = {"value": job_rate(e2e_steps, world, e2e_sec), "unit": "tokens/s", "h2d_bytes_per_step": 8,
           "d2h_bytes_per_step": 4, "steps": e2e_steps}

    wbytes = recipes.weight_bytes_per_token(cfg)
    kv_mean = float(np.mean([recipes.kv_bytes_per_token(cfg, start_pos + args.warmup + i) for i in range(args.steps)]))
    peak, peak_kind = peaks()
    weight_gbs = wbytes * args.steps / sec / 1e9
    total_gbs = (wbytes + kv_mean) * args.steps / sec / 1e9

    line = {
        "metric": METRIC, "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if mode == q8.F32ACT_F64SUM else "i8", "data": "synthetic",
        "config": workload_config(cfg, mode, world),
        "positions": [start_pos + args.warmup, cfg["ctx"] - 1],
        "weight_stream": {"gbs": weight_gbs, "frac_of_peak": weight_gbs / peak, "bytes_per_token": wbytes,
                          "peak_gbs": peak, "peak_kind": peak_kind},
        "hbm_total_gbs": total_gbs,
        "gpu_launches": model.launches_per_step() * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }

    if rank == 0:
        dom_sec, dom_bytes = time_dominant_kernel(q8, cfg, dev, mode, reps=4, stream=sh)
        achieved = dom_bytes / dom_sec / 1e9
        line["roofline"] = {"bound": "hbm", "kernel": "moe_gate_up (8 experts x 2 x 768 rows of 2048)",
                            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                            "traffic": roofline_traffic(mode == q8.INT8ACT),
                            "traffic_source": ROOFLINE_TRAFFIC["profile"],
                            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                            "us_per_launch": dom_sec * 1e6, "algorithmic_bytes_per_launch": dom_bytes}
        if not args.no_secondary:
            names = {q8.F32ACT_F64SUM: "f32-activation/f64-sum", q8.INT8ACT: "int8-activation",
                     q8.INT8ACT2: "two-word int8-activation"}
            line["secondary"] = []
            for other in (q8.INT8ACT2, q8.F32ACT_F64SUM, q8.INT8ACT):
                if other == mode:
                    continue
                m2 = q8.Model(cfg, dev, other, tok, pos, logits)
                pos.fill_(cfg["ctx"] - total)
                with torch.cuda.stream(stream):
                    for _ in range(args.warmup):
                        m2.step(sh)
                    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a0.record(stream)
                    for _ in range(args.steps):
                        m2.step(sh)
                    a1.record(stream)
                    a1.synchronize()
                s2 = a0.elapsed_time(a1) / 1e3
                line["secondary"].append({"mode": names[other], "tokens_per_s": args.steps / s2,
                                          "weight_stream_gbs": wbytes * args.steps / s2 / 1e9,
                                          "frac_of_peak": wbytes * args.steps / s2 / 1e9 / peak})
                m2.check(sh)
                m2.close()
            # the same step in the other form (as one persistent launch for all layers, or as six launches a layer)
            if mode != q8.F32ACT_F64SUM:
                other_form = not model.persistent()
                q8.set_persistent_decode(other_form)
                try:
                    m3 = q8.Model(cfg, dev, mode, tok, pos, logits)
                    if m3.persistent() == other_form:
                        pos.fill_(cfg["ctx"] - total)
                        with torch.cuda.stream(stream):
                            for _ in range(args.warmup):
                                m3.step(sh)
                            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                            a0.record(stream)
                            for _ in range(args.steps):
                                m3.step(sh)
                            a1.record(stream)
                            a1.synchronize()
                        s3 = a0.elapsed_time(a1) / 1e3
                        line["secondary"].append({
                            "mode": names[mode] + (", all layers as one persistent launch" if other_form
                                                   else ", six launches a layer"),
                            "tokens_per_s": args.steps / s3, "weight_stream_gbs": wbytes * args.steps / s3 / 1e9,
                            "frac_of_peak": wbytes * args.steps / s3 / 1e9 / peak,
                            "launches_per_step": m3.launches_per_step()})
                        m3.check(sh)
                    m3.close()
                finally:
                    q8.set_persistent_decode(bool(args.persistent))
            line["batch"] = {"what": "the batch form: B sequences per step, every weight read once for all of them, "
                                     "one CUDA graph per step, int8 mode; the attention streamed from 8 sequences", "results": time_batch(q8, cfg, dev, sh, mode)}
            line["prefill"] = {"what": "prefill_chunk through all layers (plain launches), positions ctx-128-R ..",
                               "results": time_prefill(q8, model, cfg, tok, pos, sh)}
            line["chunks"] = {
                "what": "R-row chunks through the mixture block (int8: quantize, route + grouping, gate-up, "
                        "down-and-combine), another layer's experts per chunk, one CUDA graph of 8 chunks per R",
                "uncorrelated": time_chunks(q8, cfg, dev, sh, reps=max(2, min(args.steps, 8))),
                "correlated": time_chunks(q8, cfg, dev, sh, reps=max(2, min(args.steps, 8)), correlated=True,
                                          rows=(16, 32, 64))}
            line["configs"] = time_configs(q8, cfg, dev, sh, peak)
        if not args.no_cpu_baseline:
            cb, cores = cpu_baseline_oracle(cfg, host, int(mode), 0, cfg["ctx"] - 1)
            allc, one = cb["all_cores"], cb["single_thread"]
            line["cpu_baseline"] = {"value": allc["tokens_per_s"], "unit": "tokens/s", "cores": allc["threads"],
                                    "host_cores": cores, "kind": "oracle",
                                    "sample": f"one whole decode step (all {cfg['layers']} layers, LM head, greedy "
                                              f"token) at position 4095, f64 C oracle on {allc['threads']} threads, "
                                              f"median of {allc['runs']} steps of {allc['median_s']:.2f} s",
                                    "single_thread": {"value": one["tokens_per_s"], "unit": "tokens/s", "cores": 1,
                                                      "median_s": one["median_s"], "runs": one["runs"]},
                                    "weight_gbs_all_cores": wbytes * allc["tokens_per_s"] / 1e9}
        print(json.dumps(line), flush=True)
    model.close()
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
