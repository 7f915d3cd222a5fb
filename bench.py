#!/usr/bin/env python3
"""Benchmark of the GB300 quantized-weight linear projection.

Headline (the metric's first half, "Q2_0 GEMV weight GB/s vs HBM peak"): the fused
in_proj_qkvz decode projection, Q2_0 group-128 weight [16384 (QKV 10240 | Z 6144), 5120],
at m = 1 and m = 4.  One step runs that projection for L layers, each layer with its own
weight (L * 22.3 MB >> L2), first all layers at m = 1, then all at m = 4, so no weight is
ever re-read from L2.  The step is captured once in a CUDA graph and replayed K times
between CUDA events.  `value` = weight bytes streamed / elapsed time (GB/s).

Every other hot-path row is measured in the same run on its own workload (under "rows"):
the 1024x1024 GEMV, the packed-Q2 FFN decode chain (m = 2, 3, 8), q8_1 quantisation,
Q2_0 MMQ at m = 512/2048/4096 beside the dequant + cuBLAS route, Q4_K MMQ (FFN prefill),
and dequantisation.

--impl reference runs the CPU oracle (the only reference there is) on a bounded sample of
the same workload and prints the same line with "impl": "reference".

Multi-GPU: the projection has no exchange step; N > 1 runs N independent replicas (one
process per GPU under torchrun), value = total bytes of all ranks / max elapsed.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q2_0 GEMV weight GB/s vs HBM peak (m=1..8); Q2/Q4_K MMQ int8 TOPS"
N_QKVZ, K_HIDDEN, N_QKV, N_Z = 16384, 5120, 10240, 6144
WORKLOAD = "qkvz decode GEMV: Q2_0 g128 weight [16384 (QKV 10240 | Z 6144), 5120], m=1 and m=4"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- distributed
def _dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value, world):
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons every `period_ms` in the background."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id, period_ms=10):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-i", str(gpu_id),
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        parsed = []
        for ts, line in self.rows:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                parsed.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        inside = [p for p in parsed if t0 <= p[0] <= t1]
        note = "samples inside the timed region"
        if not inside and parsed:
            # region shorter than the sampling period: nearest samples, still under the load
            inside = sorted(parsed, key=lambda p: min(abs(p[0] - t0), abs(p[0] - t1)))[:3]
            note = "timed region shorter than the sampling period; nearest samples under the same load"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i, v in enumerate(p[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(p[1] for p in inside), "sm_max_mhz": max(p[2] for p in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


# ----------------------------------------------------------------------------- GPU helpers
def _bf(a, dev):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _graph(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _time_graph(g, reps, warm=2):
    import torch
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def _time_calls(fn, reps, warm=3):
    import torch
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def _traffic_record(kernel_src, name):
    """Per-launch DRAM traffic from a committed ncu summary, if it was taken on the current
    kernel source (sha256 match); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(name)
    if not rec:
        return None
    h = hashlib.sha256(open(os.path.join(ROOT, kernel_src), "rb").read()).hexdigest()
    return rec.get("bytes_per_launch") if rec.get("source_sha256") == h else None


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, local, world):
    import numpy as np
    import torch
    import bit_quantized_linear_q8_gb300 as B
    from bit_quantized_linear_q8_gb300 import build, synth

    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, bf16_sus, peak_src = _peaks()
    L = args.layers

    # ---- headline: L distinct qkvz weights, m = 1 and m = 4
    d = synth.qkvz_gemv()
    base = B.q2_pack(torch.from_numpy(d["codes"]).to(dev), _bf(d["scales"], dev))
    wbytes = B.q2_weight_bytes(N_QKVZ, K_HIDDEN)
    layers = [base] + [B.Q2Weight(base.data.clone(), N_QKVZ, K_HIDDEN) for _ in range(L - 1)]
    x_all = _bf(d["x"], dev)
    x1, x4 = x_all[:1].contiguous(), x_all[:4].contiguous()
    y1 = torch.empty((L, 1, N_QKVZ), dtype=torch.bfloat16, device=dev)
    y4 = torch.empty((L, 4, N_QKVZ), dtype=torch.bfloat16, device=dev)

    def step():
        for i in range(L):
            B.q2_gemv(x1, layers[i], out=y1[i])
        for i in range(L):
            B.q2_gemv_batchm(x4, layers[i], out=y4[i])

    g = _graph(step)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    gpu_id = torch.cuda.get_device_properties(dev).uuid if hasattr(torch.cuda.get_device_properties(dev), "uuid") else local
    sampler = ClockSampler("GPU-" + str(gpu_id) if not str(gpu_id).startswith("GPU-") else gpu_id) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    _barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    _barrier(world)
    elapsed = e0.elapsed_time(e1) / 1e3
    if sampler:
        time.sleep(0.1)
        sampler.stop()
    elapsed_max = reduce_max(elapsed, world)
    step_weight_bytes = 2 * L * wbytes
    total_bytes = reduce_sum(step_weight_bytes * args.steps, world)
    value = total_bytes / elapsed_max / 1e9
    launches_per_step = 2 * L
    per_launch = elapsed / (args.steps * launches_per_step)
    alg_bytes = wbytes + (K_HIDDEN * 2 + N_QKVZ * 2) * (1 + 4) / 2.0  # + x and y, averaged over m=1 and m=4
    achieved = alg_bytes / per_launch / 1e9

    # the public API called eagerly (no CUDA graph): host marshalling, the tensor-map cache
    # lookup and the launch, per call, against the same calls replayed from a graph
    eager = {}
    for m in (1, 4):
        xm, ym = (x1, y1) if m == 1 else (x4, y4)
        call = (lambda i: B.q2_gemv(xm, layers[i % L], out=ym[i % L])) if m == 1 else \
            (lambda i: B.q2_gemv_batchm(xm, layers[i % L], out=ym[i % L]))
        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        ncall = 400
        h0 = time.perf_counter()
        for i in range(ncall):
            call(i)
        h1 = time.perf_counter()
        torch.cuda.synchronize()
        h2 = time.perf_counter()
        eager["m%d" % m] = {"host_us_per_call": round((h1 - h0) / ncall * 1e6, 2),
                            "wall_us_per_call": round((h2 - h0) / ncall * 1e6, 2)}
    eager["note"] = ("eager calls through the Python binding and the C ABI (tensor maps from the library's "
                     "cache); host_us = time to issue a call, wall_us = issue to drain, per call")

    # per-m launch times: a graph of the L launches at one m, so host launch overhead is out
    kern = {}
    for m in (1, 4):
        gm = _graph(lambda: [(B.q2_gemv(x1, layers[i], out=y1[i]) if m == 1 else
                              B.q2_gemv_batchm(x4, layers[i], out=y4[i])) for i in range(L)])
        t = _time_graph(gm, max(3, args.steps // 4)) / L
        kern["m%d" % m] = {"us_per_launch": round(t * 1e6, 3), "weight_GBps": round(wbytes / t / 1e9, 1)}
        del gm

    # ---- e2e through the public API: x from pinned host memory, all outputs back to host
    x1h = x1.cpu().pin_memory()
    x4h = x4.cpu().pin_memory()
    yh1 = torch.empty((L, 1, N_QKVZ), dtype=torch.bfloat16).pin_memory()
    yh4 = torch.empty((L, 4, N_QKVZ), dtype=torch.bfloat16).pin_memory()
    xd1, xd4 = torch.empty_like(x1), torch.empty_like(x4)

    def e2e_step(_):
        xd1.copy_(x1h, non_blocking=True)
        xd4.copy_(x4h, non_blocking=True)
        for i in range(L):
            B.q2_gemv(xd1, layers[i], out=y1[i])
        for i in range(L):
            B.q2_gemv_batchm(xd4, layers[i], out=y4[i])
        yh1.copy_(y1, non_blocking=True)
        yh4.copy_(y4, non_blocking=True)
    # the step as a user would run it in a serving loop: one CUDA graph of the API calls,
    # the input copy from pinned host memory and the result copy back to pinned host memory
    e2e_graph = _graph(lambda: e2e_step(0))
    e2e_steps = max(3, min(args.steps, 100))
    t_e2e = _time_graph(e2e_graph, e2e_steps)
    e2e = {"value": reduce_sum(step_weight_bytes, world) / reduce_max(t_e2e, world) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": x1.numel() * 2 + x4.numel() * 2,
           "d2h_bytes_per_step": y1.numel() * 2 + y4.numel() * 2,
           "note": "public API calls captured with the per-step H2D (pinned) and D2H (pinned) copies in one "
                   "CUDA graph; %d steps" % e2e_steps}
    del e2e_graph

    clocks = sampler.summary(t0, t1) if sampler else None
    del layers, y1, y4
    torch.cuda.empty_cache()

    rows = {} if args.no_rows else measure_rows(args, dev, hbm_peak, bf16_peak)

    if rank != 0:
        return None
    traffic = _traffic_record("bit_quantized_linear_q8_gb300/csrc/gemv_hm.cu", "q2_gemv_qkvz")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_max / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers_per_step": L,
                   "l2": "inputs larger than L2: %d distinct layer weights (%.0f MB) per step" % (L, L * wbytes / 1e6),
                   "parallelism": "replicas x%d" % world, "graph": "one CUDA graph per step"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "kernel": "q2_gemv_hm_kernel", "peak_source": peak_src,
                     "note": "algorithmic bytes per launch (weight + x + y) / (graph elapsed / launches)"},
        "per_m": kern,
        "eager": eager,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "rows": rows,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def measure_rows(args, dev, hbm_peak, bf16_peak):
    rows = {}
    reps = max(5, min(args.steps, 50))
    groups = set(args.rows.split(","))
    if "gemv1024" in groups:
        _rows_gemv1024(rows, reps, dev, hbm_peak)
    if "ffn" in groups:
        _rows_ffn(rows, reps, dev, hbm_peak)
    if "prefill" in groups:
        _rows_prefill(rows, reps, dev, hbm_peak, bf16_peak)
    if "q4k" in groups:
        _rows_q4k(rows, reps, dev)
    if "nvfp4" in groups:
        _rows_nvfp4(rows, reps, dev, hbm_peak)
    return rows


def _rows_nvfp4(rows, reps, dev, hbm_peak):
    import torch
    import bit_quantized_linear_q8_gb300 as B
    from bit_quantized_linear_q8_gb300 import synth

    # NVFP4 -> BF16 dequantisation of the FFN gate weight [17408, 5120] (the step before the
    # Q4_K quantiser): reads k/2 + k/16 bytes per row, writes 2k
    d = synth.nvfp4_ffn_weight()
    n, k = d["n"], d["k"]
    packed = torch.from_numpy(d["packed"]).to(dev)
    scales = torch.from_numpy(d["scales"]).to(dev)
    out = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
    t = _time_calls(lambda i: B.dequant_nvfp4_to_bf16(packed, scales, d["scale2"], n, k, out=out), reps)
    nb = n * (k // 2) + n * (k // 16) + n * k * 2
    rows["a10_nvfp4_dequant_17408x5120"] = {"us": t * 1e6, "GBps": nb / t / 1e9, "frac_hbm": nb / t / 1e9 / hbm_peak}
    del packed, scales, out
    torch.cuda.empty_cache()


def _rows_gemv1024(rows, reps, dev, hbm_peak):
    import torch
    import bit_quantized_linear_q8_gb300 as B
    from bit_quantized_linear_q8_gb300 import synth

    # a1: 1024 x 1024 GEMV, m = 1 (latency-bound: 278,528 weight bytes)
    d = synth.q2_gemv_1024()
    w0 = B.q2_pack(torch.from_numpy(d["codes"]).to(dev), _bf(d["scales"], dev))
    copies = [w0] + [B.Q2Weight(w0.data.clone(), 1024, 1024) for _ in range(511)]
    x = _bf(d["x"], dev)
    y = torch.empty((1, 1024), dtype=torch.bfloat16, device=dev)
    g = _graph(lambda: [B.q2_gemv(x, c, out=y) for c in copies])
    t = _time_graph(g, max(2, reps // 10)) / len(copies)
    wb = B.q2_weight_bytes(1024, 1024)
    rows["a1_gemv_1024_m1"] = {"us": t * 1e6, "weight_GBps": wb / t / 1e9, "frac_hbm": wb / t / 1e9 / hbm_peak,
                               "note": "512 distinct copies (143 MB) per graph; per-launch time includes graph gaps"}
    del copies, g
    torch.cuda.empty_cache()


def _rows_ffn(rows, reps, dev, hbm_peak):
    import torch
    import bit_quantized_linear_q8_gb300 as B
    from bit_quantized_linear_q8_gb300 import synth

    # a2-a4: packed-Q2 FFN decode chain (gate/up [17408, 5120], down [5120, 17408])
    d = synth.ffn_q2_decode()
    hidden, inter = d["hidden"], d["inter"]
    ws = [B.q2_pack(torch.from_numpy(c).to(dev), _bf(s, dev)) for c, s in (d["gate"], d["up"], d["down"])]
    chain_bytes = sum(B.q2_weight_bytes(w.n, w.k) for w in ws)
    sets = [ws] + [[B.Q2Weight(w.data.clone(), w.n, w.k) for w in ws] for _ in range(3)]
    xf = _bf(d["x"], dev)
    for m in (2, 3, 8):
        xm = xf[:m].contiguous()
        gs = torch.empty((m, inter), dtype=torch.bfloat16, device=dev)
        us = torch.empty((m, inter), dtype=torch.bfloat16, device=dev)
        out = torch.empty((m, hidden), dtype=torch.bfloat16, device=dev)
        g = _graph(lambda: [B.ffn_q2_km(xm, *s, gate_scratch=gs, up_scratch=us, out=out)
                            for s in sets])
        t = _time_graph(g, reps) / len(sets)
        rows["a4_ffn_q2_m%d" % m] = {"us": t * 1e6, "weight_GBps": chain_bytes / t / 1e9,
                                     "frac_hbm": chain_bytes / t / 1e9 / hbm_peak,
                                     "launches": 2, "note": "gate+up in one launch (SiLU*mul in its store), then down"}
    # per-GEMV times inside the chain at m = 8 (gate, down) and SiLU*mul alone
    xm = xf.contiguous()
    gs = torch.empty((8, inter), dtype=torch.bfloat16, device=dev)
    us = torch.empty((8, inter), dtype=torch.bfloat16, device=dev)
    out = torch.empty((8, hidden), dtype=torch.bfloat16, device=dev)
    g = _graph(lambda: [B.q2_gemv_batchm(xm, s[0], out=gs) for s in sets])
    t = _time_graph(g, reps) / len(sets)
    rows["a2_gemv_gate_m8"] = {"us": t * 1e6, "weight_GBps": ws[0].data.numel() / t / 1e9}
    g = _graph(lambda: [B.q2_gemv_batchm(gs, s[2], out=out) for s in sets])
    t = _time_graph(g, reps) / len(sets)
    rows["a2_gemv_down_m8"] = {"us": t * 1e6, "weight_GBps": ws[2].data.numel() / t / 1e9}
    g = _graph(lambda: B.silu_mul_bf16(gs, us, out=gs))
    t = _time_graph(g, reps)
    rows["a3_silu_mul_m8"] = {"us": t * 1e6, "GBps": 3 * gs.numel() * 2 / t / 1e9}
    del sets, ws, g
    torch.cuda.empty_cache()


def _rows_prefill(rows, reps, dev, hbm_peak, bf16_peak):
    import torch
    import bit_quantized_linear_q8_gb300 as B
    from bit_quantized_linear_q8_gb300 import synth

    # a5, a6, a8, a9: Q2 prefill projection
    d = synth.q2_prefill_weight()
    w = B.q2_pack(torch.from_numpy(d["codes"]).to(dev), _bf(d["scales"], dev))
    n, k = d["n"], d["k"]
    wd = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
    t = _time_calls(lambda i: B.dequant_q2_to_bf16(w, out=wd), reps)
    dq_bytes = B.q2_weight_bytes(n, k) + n * k * 2
    rows["a8_dequant_16384x5120"] = {"us": t * 1e6, "GBps": dq_bytes / t / 1e9, "frac_hbm": dq_bytes / t / 1e9 / hbm_peak}
    for m in (512, 2048, 4096):
        x = _bf(synth.q2_prefill_x(m), dev)
        act = torch.empty(B.q8_1_bytes(m, k), dtype=torch.uint8, device=dev)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        qb = m * k * 2 + B.q8_1_bytes(m, k)
        # q8_1 rotates over copies of x and of its output that together exceed twice L2, so
        # every call reads and writes HBM
        nq = 2 * L2_BYTES // qb + 2
        xq = [x] + [x.clone() for _ in range(nq - 1)]
        aq = [act] + [torch.empty_like(act) for _ in range(nq - 1)]
        tq_eager = _time_calls(lambda i: B.quantize_act_q8_1(xq[i % nq], out=aq[i % nq]), reps)
        # the same calls replayed from a CUDA graph: the kernels back to back, without the
        # host's per-call marshalling (about 10 us, more than the kernel below m = 2048)
        gq = _graph(lambda: [B.quantize_act_q8_1(xq[i % nq], out=aq[i % nq]) for i in range(2 * nq)])
        tq = _time_graph(gq, max(3, reps // nq)) / (2 * nq)
        del xq, aq, gq
        tm = _time_calls(lambda i: B.q2_mmq_gemm(act, w, m, out=out), max(3, reps // 5))
        tg = _time_calls(lambda i: torch.matmul(x, wd.t(), out=out), max(3, reps // 5))
        to = _time_calls(lambda i: B.dense_gemm_bf16(x, wd, out=out), max(3, reps // 5))
        flops = 2.0 * m * n * k
        rows["a5_q8_1_m%d" % m] = {"us": tq * 1e6, "GBps": qb / tq / 1e9, "frac_hbm": qb / tq / 1e9 / hbm_peak,
                                   "us_eager": tq_eager * 1e6, "timing": "CUDA graph of back-to-back calls"}
        rows["a6_q2_mmq_m%d" % m] = {"us": tm * 1e6, "TOPS": flops / tm / 1e12,
                                     "frac_bf16_dense_peak": flops / tm / 1e12 / bf16_peak,
                                     "tensor_pipe_frac": 2 * flops / tm / 1e12 / bf16_peak,
                                     "pipe": "tcgen05.mma kind::f16 M128 N256 K16: exact BF16 weights d(c-2), q8_1 "
                                             "activations as a hi/lo BF16 pair (2 MMAs per K16; sm_103a has no "
                                             "tcgen05 int8)"}
        rows["a9_dequant_plus_gemm_m%d" % m] = {"us": (to + rows["a8_dequant_16384x5120"]["us"] / 1e6) * 1e6,
                                               "gemm_us": to * 1e6, "TFLOPS_gemm": flops / to / 1e12,
                                               "frac_bf16_dense_peak": flops / to / 1e12 / bf16_peak,
                                               "gemm": "dense_gemm_bf16 (this library's tcgen05 kernel)"}
        rows["a9_dequant_plus_cublas_m%d" % m] = {"us": (tg + rows["a8_dequant_16384x5120"]["us"] / 1e6) * 1e6,
                                                 "gemm_us": tg * 1e6, "TFLOPS_gemm": flops / tg / 1e12,
                                                 "gemm": "cuBLAS through torch.matmul (comparison only)"}
        del x, act, out
    del w, wd
    torch.cuda.empty_cache()


def _rows_q4k(rows, reps, dev):
    import torch
    import bit_quantized_linear_q8_gb300 as B
    from bit_quantized_linear_q8_gb300 import synth

    # a7: Q4_K MMQ FFN prefill (gate, up -> SiLU*mul -> down) at m = 2048
    try:
        d = synth.q4k_ffn_prefill()
        m, hidden, inter = d["m"], d["hidden"], d["inter"]
        wq = [B.quantize_weight_q4k(_bf(d[kk], dev)) for kk in ("w_gate", "w_up", "w_down")]
        x = _bf(d["x"], dev)
        a1 = torch.empty(B.q8_1_bytes(m, hidden), dtype=torch.uint8, device=dev)
        a2 = torch.empty(B.q8_1_bytes(m, inter), dtype=torch.uint8, device=dev)
        gt = torch.empty((m, inter), dtype=torch.bfloat16, device=dev)
        ut = torch.empty((m, inter), dtype=torch.bfloat16, device=dev)
        out = torch.empty((m, hidden), dtype=torch.bfloat16, device=dev)

        def chain(i):
            B.quantize_act_q8_1(x, out=a1)
            B.q4k_mmq_gemm(a1, wq[0], m, inter, hidden, out=gt)
            B.q4k_mmq_gemm(a1, wq[1], m, inter, hidden, out=ut)
            B.silu_mul_bf16(gt, ut, out=gt)
            B.quantize_act_q8_1(gt, out=a2)
            B.q4k_mmq_gemm(a2, wq[2], m, hidden, inter, out=out)
        t = _time_calls(chain, max(3, reps // 5))
        tg = _time_calls(lambda i: B.q4k_mmq_gemm(a1, wq[0], m, inter, hidden, out=gt), max(3, reps // 5))
        flops = 3 * 2.0 * m * hidden * inter
        rows["a7_q4k_ffn_prefill_m2048"] = {"us": t * 1e6, "TOPS_chain": flops / t / 1e12,
                                            "gate_gemm_us": tg * 1e6,
                                            "gate_TOPS": 2.0 * m * hidden * inter / tg / 1e12,
                                            "pipe": "tcgen05.mma kind::f16 M128 N256 K16: activations and Q4_K "
                                                    "weights as hi/lo BF16 pairs (3 MMAs per K16)"}
    except Exception as e:  # reported, not hidden
        rows["a7_q4k_ffn_prefill_m2048"] = {"error": str(e)[:200]}


# ----------------------------------------------------------------------------- CPU oracle
def cpu_baseline(seconds=10.0, rows_sample=1024):
    """The oracle, as it stands, on the host cores: GEMV m=1 and m=4 over a row sample of
    the qkvz weight, repeated until `seconds` elapse.  GB/s of weight bytes (the sample's
    share of the Q2_0 weight)."""
    import numpy as np
    import oracle as O
    from bit_quantized_linear_q8_gb300 import synth
    d = synth.qkvz_gemv()
    codes, scales = d["codes"][:rows_sample], d["scales"][:rows_sample]
    packed = O.q2_pack(codes, scales)
    x1, x4 = d["x"][:1], d["x"][:4]
    wbytes = packed.size
    done, t0 = 0, time.time()
    while True:
        O.q2_gemv(x1, packed, rows_sample, K_HIDDEN)
        O.q2_gemv(x4, packed, rows_sample, K_HIDDEN)
        done += 2
        if time.time() - t0 >= seconds:
            break
    el = time.time() - t0
    cores = O.num_threads()
    # the same sample on one core, for a quarter of the time
    O.set_num_threads(1)
    done1, t1 = 0, time.time()
    while True:
        O.q2_gemv(x1, packed, rows_sample, K_HIDDEN)
        O.q2_gemv(x4, packed, rows_sample, K_HIDDEN)
        done1 += 2
        if time.time() - t1 >= seconds / 4:
            break
    el1 = time.time() - t1
    O.set_num_threads(cores)
    return {"value": round(done * wbytes / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d of 16384 weight rows, GEMV m=1 and m=4, %d passes in %.1f s" % (rows_sample, done, el),
            "one_core": {"value": round(done1 * wbytes / el1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                         "sample": "%d passes in %.1f s" % (done1, el1)}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle as O
    from bit_quantized_linear_q8_gb300 import synth
    rows_sample = 256
    d = synth.qkvz_gemv()
    packed = O.q2_pack(d["codes"][:rows_sample], d["scales"][:rows_sample])
    x1, x4 = d["x"][:1], d["x"][:4]

    def step():
        O.q2_gemv(x1, packed, rows_sample, K_HIDDEN)
        O.q2_gemv(x4, packed, rows_sample, K_HIDDEN)
    for _ in range(args.warmup):
        step()
    t0 = time.time()
    for _ in range(args.steps):
        step()
    el = time.time() - t0
    value = 2 * packed.size * args.steps / el / 1e9
    sample = "%d of 16384 qkvz weight rows per step, GEMV m=1 and m=4" % rows_sample
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": O.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=64,
                    help="distinct qkvz layer weights per step (64: a step of about 1.7 ms, so that the clock "
                         "sampler sees the timed region even at 20 steps)")
    ap.add_argument("--no-rows", action="store_true", help="headline only")
    ap.add_argument("--rows", default="gemv1024,ffn,prefill,q4k,nvfp4",
                    help="row groups to measure: gemv1024 (a1), ffn (a2-a4), prefill (a5, a6, a8, a9), q4k (a7), "
                         "nvfp4 (NVFP4 -> BF16 weight preparation)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, local, world = _dist_init(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, local, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
