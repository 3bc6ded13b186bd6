"""Benchmark: one affinity-aware MoE layer forward per step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one whole layer forward (route + lookup/count + permute + grouped
FFN + shared FFN + combine) over one batch of synthetic tokens, inputs
resident in HBM.  Prints one JSON line (rank 0).  With N > 1 (torchrun) each
rank runs an independent replica of the layer: the path has no exchange step
on one device, so there is no collective on the data path ("weak" scaling).

``--impl reference`` times the CPU oracle (plain numpy, float64) on the host
cores on a bounded sample of the same workload, as the reference arm.
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s (route+permute+grouped FFN+combine), % of HBM/TC roofline"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 20 ms requested) while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = uuid if uuid.startswith("GPU-") else ("GPU-" + uuid)
        except Exception:
            sel = str(self.dev)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", sel], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)  # let the sampler start before the timed region
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _flops_bytes(spec, P, active_experts, fused_gather=False):
    """Algorithmic flops and bytes of each step for one layer forward.

    FFN bytes: the weights of every expert with at least one row, the rows in,
    the intermediate h written and read back, the rows out.  With the permute
    fused into GEMM1 (fused_gather) the permute writes index tables only and
    GEMM1's rows in are the T token rows of x, each read once."""
    s = 2 if spec.dtype == "bf16" else 4
    sr = 2 if spec.router_dtype == "bf16" else 4
    T, H, E, I, k = spec.T, spec.H, spec.E, spec.I, spec.k_max
    Is = spec.I_shared
    return {
        # an fp32 router weight times bf16 activations runs on the tensor cores as three
        # exact bf16 parts: three times the GEMM's flops executed (flops_executed)
        "route": dict(flops=2 * T * H * E, bytes=T * H * s + E * H * sr + T * k * 8,
                      flops_executed=(3 if spec.router_dtype == "f32" and spec.dtype == "bf16" else 1) * 2 * T * H * E),
        "permute": dict(bytes=4 * T * k * 2 + 4 * P + 4 * T * k + (0 if fused_gather else T * H * s + P * H * s)),
        "grouped_ffn": dict(flops=6 * H * I * P,
                            bytes=active_experts * 3 * H * I * s + (T if fused_gather else P) * H * s
                            + 2 * P * I * s + P * H * s),
        "shared_ffn": dict(flops=6 * H * Is * T, bytes=3 * H * Is * s + 2 * T * H * s + 2 * T * Is * s),
        "combine": dict(bytes=P * H * s + 8 * T * k + T * H * s * (2 if spec.I_shared else 1)),
    }


def _sources_hash(files):
    import hashlib
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(call: str, workload: str):
    """DRAM bytes per call from the committed ncu record (profiles/traffic.json),
    or None when that record is missing or the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(call, {}).get(workload)
    if not rec:
        return None
    try:
        if _sources_hash(rec["sources"]) != rec["sources_sha1"]:
            return None
    except OSError:
        return None
    return rec["dram_bytes"]


def cpu_oracle_rate(d, n_tokens: int, weights64=None):
    """Tokens/s of the CPU oracle on the first n_tokens of the workload."""
    import oracle
    spec = d["spec"]
    if weights64 is None:
        weights64 = _weights64(d)
    sl = slice(0, n_tokens)
    t0 = time.perf_counter()
    oracle.moe_layer(d["x"][sl], weights64["w_router"], d["token_ids"][sl], d["lut"], d["expert_rank"],
                     d["k_per_token"][sl], weights64["w13"], weights64["w2"], spec.R, spec.dtype,
                     spec.k_max, weights64["ws13"], weights64["ws2"])
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def _weights64(d):
    """float64 numpy copies of the weights (exact), made once outside any timing."""
    f = lambda t: None if t is None else t.to(torch.float64).numpy()  # noqa: E731
    return {k: f(d[k]) for k in ("w_router", "w13", "w2", "ws13", "ws2")}


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _blas_threads():
    """Threads numpy's BLAS runs with: asked of the loaded OpenBLAS itself,
    else the thread environment variables, else the usable cores."""
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ".so" in ln})
        for path in paths:
            lib = ctypes.CDLL(path)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                        "openblas_get_num_threads"):
                fn = getattr(lib, sym, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    return int(fn()), f"{os.path.basename(path)} {sym}()"
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var]), var
    return _cores(), "usable cores (BLAS default)"


def _cpu_desc(value, sample):
    threads, how = _blas_threads()
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample,
            "cpu_model": _cpu_model(), "host_cores": _cores(), "threads_from": how}


#: workloads the oracle is also timed on with one thread (tiny layer, decode)
SINGLE_THREAD_CONFIGS = ("tiny_fp32_T256_E8", "dsv2lite_decode_T64")


def oracle_single_thread():
    """Oracle tokens/s on the tiny and decode workloads with one BLAS thread.
    Runs in a child process started with the thread variables set to 1 (numpy
    reads them once, at import)."""
    out = {}
    for name in SINGLE_THREAD_CONFIGS:
        spec = wl.CONFIGS[name]
        d = wl.make_inputs(spec)
        rate, dt = cpu_oracle_rate(d, spec.T)
        out[name] = {"value": rate, "unit": "tokens/s", "s": dt, "tokens": spec.T}
    threads, how = _blas_threads()
    out["threads"] = threads
    out["threads_from"] = how
    return out


def _single_thread_baseline():
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-thread"],
                           capture_output=True, text=True, timeout=600, env=env)
        for ln in r.stdout.splitlines()[::-1]:
            if ln.startswith("{"):
                return json.loads(ln)
        return {"error": (r.stderr or r.stdout)[-300:]}
    except Exception as e:  # reported, never fatal to the benchmark line
        return {"error": repr(e)[:300]}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    spec = wl.CONFIGS[args.config]
    d = wl.make_inputs(spec)
    w64 = _weights64(d)
    n = args.ref_tokens
    for _ in range(args.warmup):
        cpu_oracle_rate(d, n, w64)
    times = []
    for _ in range(args.steps):
        _, dt = cpu_oracle_rate(d, n, w64)
        times.append(dt)
    total = sum(times)
    value = n * args.steps / total
    sample = f"first {n} of {spec.T} tokens of {spec.name} per step (float64 numpy oracle)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(spec),
        "cpu_baseline": _cpu_desc(value, sample),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(spec):
    return {"workload": spec.name, "T": spec.T, "H": spec.H, "E": spec.E, "top_k": spec.k_max,
            "I": spec.I, "I_shared": spec.I_shared, "R": spec.R, "dtype": spec.dtype,
            "router_dtype": spec.router_dtype,
            "l2": "inputs larger than L2: expert weights (>1 GB) are streamed every step",
            "parallelism": "replicas"}


def _time_around_layer(args, spec, d, layer, dev, stream):
    """Device time of the table-driven steps around the layer, on the same
    workload: Attention-DP request scheduling and the next-layer transition
    lookup (not part of the layer step above)."""
    from token_expert_routing_gb300 import _abi
    T, R, E, k_max = spec.T, spec.R, spec.E, spec.k_max
    i32 = dict(dtype=torch.int32, device=dev)
    pred = torch.empty(T, **i32)
    _abi.semmoe_affinity_lookup(d["token_ids"].to(dev), layer.lut, layer.V, R, T, pred, stream)
    off = d["req_offsets"].to(dev)
    n = off.shape[0] - 1
    bufs = [torch.empty(n, R, **i32), torch.empty(n, **i32), torch.empty(n, **i32), torch.empty(R + 1, **i32),
            torch.empty(n, **i32), torch.empty(T, **i32), torch.empty(T, **i32), torch.empty(R + 1, **i32)]
    res = layer.forward(d["x"].to(dev), d["token_ids"].to(dev),
                        d["k_per_token"].to(dev) if spec.k_choices else None,
                        None if spec.k_choices else spec.k, int(d["k_per_token"].sum()), stream=stream)
    trans = d["trans"].to(dev)
    kpt = d["k_per_token"].to(dev) if spec.k_choices else None
    nxt = torch.empty(T, **i32)
    calls = {
        "dp_schedule": (lambda: _abi.semmoe_dp_schedule(pred, off, T, n, R, *bufs),
                        4 * T + 4 * (n + 1) * 3 + 4 * n * R + 4 * n * 4 + 8 * T + 4 * T, f"{n} requests"),
        "transition_lookup": (lambda: _abi.semmoe_transition_lookup(res.topk_idx, kpt, 0 if kpt is not None else
                                                                   spec.k, trans, T, k_max, E, R, nxt),
                              4 * T * k_max + (4 * T if kpt is not None else 0) + 4 * E * R + 4 * T,
                              f"E={E} R={R} k_max={k_max}"),
    }
    if d.get("sub_logw") is not None:   # MoE-Prism layer: the hierarchical gate over the same tokens
        Ep = d["w_router_parent"].shape[0]
        wp = d["w_router_parent"].to(dev)
        slw = d["sub_logw"].to(dev)
        hidx = torch.empty(T, k_max, **i32)
        hw = torch.empty(T, k_max, dtype=torch.float32, device=dev)
        hws = torch.empty(max(_abi.semmoe_route_hier_workspace_size(T, spec.H, Ep, _abi.dtype_code(d["x"]),
                                                                     _abi.dtype_code(wp)), 256),
                          dtype=torch.uint8, device=dev)
        xd = d["x"].to(dev)
        calls["route_hier"] = (
            lambda: _abi.semmoe_route_hier(xd, wp, None, None, slw, E // Ep, kpt, 0 if kpt is not None else spec.k,
                                           T, spec.H, Ep, k_max, hidx, hw, hws),
            T * spec.H * 2 + Ep * spec.H * (2 if spec.router_dtype == "bf16" else 4) + 4 * E + T * k_max * 8,
            f"Ep={Ep} N={E // Ep} k_max={k_max} (parent router GEMM + hierarchical top-k)")
    out = {}
    n_it = max(args.steps, 20)
    for name, (fn, nbytes, what) in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        # n_it calls captured as one CUDA graph, so the device time is not the
        # host's per-call cost
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):            # calls go to the capture stream (current inside)
            for _ in range(n_it):
                fn()
        g.replay()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(b) * 1e3 / n_it
        out[name] = {"us": us, "algorithmic_bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9, "workload": what,
                     "bound": "latency (a few small kernels over kilobytes)",
                     "how": f"{n_it} calls in one CUDA graph, CUDA events around one replay"}
        del g
    _abi.semmoe_check_errors()
    return out


def _build_layers(spec, d, dev):
    """The layer as a user runs it (its steps spread over two streams), and the
    same layer with every step on one stream, whose per-step events give the
    stage times and the roofline of each kernel alone."""
    from token_expert_routing_gb300 import MoELayer
    layer = MoELayer(d["w_router"], d["w13"], d["w2"], d["expert_rank"], d["lut"], spec.R, spec.k_max,
                     d["ws13"], d["ws2"], device=dev)
    serial = MoELayer(d["w_router"], d["w13"], d["w2"], d["expert_rank"], d["lut"], spec.R, spec.k_max,
                      d["ws13"], d["ws2"], overlap=False, overlap_shared=False, device=dev)
    return layer, serial


def _time_eager(serial, inp, steps, warmup, world, dev, stream, local):
    """K one-stream forwards, inputs resident in HBM; per-step events give the stages."""
    from token_expert_routing_gb300 import _abi
    x, ids, kpt, k, P = inp

    def step(marks=None, side_marks=None):
        return serial.forward(x, ids, kpt, k, P, stream=stream, marks=marks, side_marks=side_marks)

    for _ in range(warmup):
        step()
    _abi.semmoe_check_errors()
    all_marks = [[] for _ in range(steps)]
    all_side = [[] for _ in range(steps)]
    launches0 = _abi.semmoe_kernel_launches()
    _barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        h0 = time.perf_counter()
        start.record(stream)
        for i in range(steps):
            step(all_marks[i], all_side[i])
        end.record(stream)
        host_ms = (time.perf_counter() - h0) * 1e3 / steps   # enqueue cost per step
        torch.cuda.synchronize(dev)
    _barrier(world)
    launches = _abi.semmoe_kernel_launches() - launches0
    _abi.semmoe_check_errors()
    ms_max = _max_over_ranks(world, start.elapsed_time(end))
    stage_ms = {}
    for marks in all_marks:
        for (_, a), (name, b) in zip(marks[:-1], marks[1:]):
            stage_ms.setdefault(name, []).append(a.elapsed_time(b))
    for side in all_side:  # steps run on the layer's second stream, beside the ones above
        for name, a, b in side:
            stage_ms.setdefault(name, []).append(a.elapsed_time(b))
    stage_avg = {n: sum(v) / len(v) for n, v in stage_ms.items()}
    per_step = sorted(m[0][1].elapsed_time(m[-1][1]) for m in all_marks)  # each step, first to last mark
    return dict(ms_max=ms_max, stage_avg=stage_avg, per_step=per_step, launches=launches, host_ms=host_ms,
                clocks=clocks.summary())


def _time_stages_graph(serial, inp, steps, warmup, dev):
    """Per-step device times of the one-stream forward captured as one CUDA
    graph: events between its steps are captured as event nodes, so every
    replay times each step without the gaps of separate launches from the host.
    Returns {step: mean ms} over the replays, or None if this torch cannot
    capture timing events."""
    x, ids, kpt, k, P = inp
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):            # workspaces and kernel attributes before capture
        for _ in range(2):
            serial.forward(x, ids, kpt, k, P, stream=side)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    marks = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        serial.forward(x, ids, kpt, k, P, stream=torch.cuda.current_stream(dev), marks=marks, mark_external=True)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    stage_ms = {}
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize(dev)
        for (_, a), (name, b) in zip(marks[:-1], marks[1:]):
            stage_ms.setdefault(name, []).append(a.elapsed_time(b))
    from token_expert_routing_gb300 import _abi
    _abi.semmoe_check_errors()
    del g
    return {n: sum(v) / len(v) for n, v in stage_ms.items()}


def _event_node_overhead(dev, n=20, replays=10):
    """What an event pair around one kernel adds to that kernel's time inside a
    CUDA graph (the event nodes and the kernel's launch after one): a small
    combine (T=64, H=2048, k=6, bf16) captured n times back to back with events
    only at the two ends, and n times between event pairs of its own.  Returns
    ms = mean event-pair time - back-to-back time per kernel, or None."""
    from token_expert_routing_gb300 import _abi
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None
    gen = torch.Generator().manual_seed(7)
    T, H, k = 64, 2048, 6
    P = T * k
    p2s = torch.randperm(P, generator=gen).to(torch.int32).to(dev)
    w = torch.rand(T, k, generator=gen).to(dev)
    y = torch.randn(P, H, generator=gen).to(torch.bfloat16).to(dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    _abi.semmoe_combine(y, p2s, w, None, T, H, k, P, out, side)
    torch.cuda.synchronize(dev)
    per_kernel = {}
    for mode in ("ends", "pairs"):
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * n)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(n):
                if mode == "pairs" or i == 0:
                    evs[2 * i].record(side)
                _abi.semmoe_combine(y, p2s, w, None, T, H, k, P, out, side)
                if mode == "pairs" or i == n - 1:
                    evs[2 * i + 1].record(side)
        vals = []
        for r in range(replays + 3):
            g.replay()
            torch.cuda.synchronize(dev)
            if r >= 3:
                vals.append(evs[0].elapsed_time(evs[2 * n - 1]) / n if mode == "ends" else
                            sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(n)) / n)
        per_kernel[mode] = sorted(vals)[len(vals) // 2]
        del g
    _abi.semmoe_check_errors()
    return max(0.0, per_kernel["pairs"] - per_kernel["ends"])


def _time_graph(layer, spec, d, inp, steps, warmup, world, dev, local):
    """The same forward as one CUDA-graph replay per step (static buffers)."""
    from token_expert_routing_gb300 import CapturedLayer, _abi
    x, ids, _, _, _ = inp
    per_token = bool(spec.k_choices)
    cap = CapturedLayer(layer, spec.T, None if per_token else spec.k, d["k_per_token"] if per_token else None)
    cap.x.copy_(x)
    cap.token_ids.copy_(ids)
    for _ in range(warmup):
        cap.replay()
    _barrier(world)
    torch.cuda.synchronize(dev)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(local) as clocks_graph:
        g0.record()
        rep_ev[0].record()
        for i in range(steps):
            cap.replay()
            rep_ev[i + 1].record()
        g1.record()
        torch.cuda.synchronize(dev)
    per_replay = sorted(a.elapsed_time(b) for a, b in zip(rep_ev[:-1], rep_ev[1:]))
    _barrier(world)
    g_ms = _max_over_ranks(world, g0.elapsed_time(g1))
    _abi.semmoe_check_errors()
    del cap
    return {"value": spec.T * steps * world / (g_ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": g_ms / steps,
            "how": "CapturedLayer: the whole forward (steps on two streams: bookkeeping and the shared "
                   "experts beside the permute and routed FFN) captured once as a CUDA graph, one replay "
                   "per step",
            "ms_median": per_replay[len(per_replay) // 2], "ms_min": per_replay[0], "ms_max": per_replay[-1],
            "clocks": clocks_graph.summary()}


def _roofline_and_stages(spec, P, active, fused_gather, stage_avg, peaks, event_ms=None):
    """The grouped FFN's roofline object and every stage's fraction of its bound.
    With event_ms (what the event pair around a step adds to it in graph
    replay), each stage also gets its time and fractions less that overhead
    (ms_net, frac_*_net)."""
    fb = _flops_bytes(spec, P, active, fused_gather)
    ffn_ms = stage_avg["grouped_ffn"]
    ffn = fb["grouped_ffn"]
    ffn_call = "semmoe_grouped_ffn_gather" if fused_gather else "semmoe_grouped_ffn"
    # the FFN's bound: whichever of its flops at the tensor peak and its bytes at
    # the HBM peak takes longer (weight streaming wins for small batches)
    t_tc = ffn["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = ffn["bytes"] / (peaks["hbm_gbs"] * 1e9)
    tflops = ffn["flops"] / (ffn_ms * 1e-3) / 1e12
    gbs = ffn["bytes"] / (ffn_ms * 1e-3) / 1e9
    if t_tc >= t_hbm:
        roofline = {
            "kernel": ffn_call + " (GEMM1+SwiGLU, GEMM2)",
            "bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tflops / peaks["bf16_tflops"], "traffic": _traffic(ffn_call, spec.name),
            "peak_source": f"{peaks['source']} bf16 burst (short timed region, SM clock at its maximum); "
                           f"sustained figure {peaks['bf16_tflops_sustained']} TFLOP/s",
            "frac_of_sustained": tflops / peaks["bf16_tflops_sustained"],
            "frac_hbm": gbs / peaks["hbm_gbs"],
            "algorithmic_flops": ffn["flops"], "ms": ffn_ms,
        }
    else:
        roofline = {
            "kernel": ffn_call + " (GEMM1+SwiGLU, GEMM2)",
            "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "traffic": _traffic(ffn_call, spec.name),
            "peak_source": f"{peaks['source']} HBM copy bandwidth",
            "algorithmic_bytes": ffn["bytes"], "active_experts": active,
            "frac_tensor": tflops / peaks["bf16_tflops"], "ms": ffn_ms,
        }
    stages = {}
    for name, avg in stage_avg.items():
        ent = {"ms": avg}
        f = fb.get(name, {})
        if "flops" in f:
            ent["tflops"] = f["flops"] / (avg * 1e-3) / 1e12
            ent["frac_tensor"] = ent["tflops"] / peaks["bf16_tflops"]
        if "bytes" in f:
            ent["gbs"] = f["bytes"] / (avg * 1e-3) / 1e9
            ent["frac_hbm"] = ent["gbs"] / peaks["hbm_gbs"]
        if "flops_executed" in f:
            ent["frac_tensor_executed"] = f["flops_executed"] / (avg * 1e-3) / 1e12 / peaks["bf16_tflops"]
        if event_ms is not None and avg > event_ms:
            net = avg - event_ms
            ent["ms_net"] = net
            if "flops" in f:
                ent["frac_tensor_net"] = f["flops"] / (net * 1e-3) / 1e12 / peaks["bf16_tflops"]
            if "bytes" in f:
                ent["frac_hbm_net"] = f["bytes"] / (net * 1e-3) / 1e9 / peaks["hbm_gbs"]
        stages[name] = ent
    return roofline, stages


def _inputs_on(spec, d, dev):
    per_token = bool(spec.k_choices)
    return (d["x"].to(dev), d["token_ids"].to(dev), d["k_per_token"].to(dev) if per_token else None,
            None if per_token else spec.k, int(d["k_per_token"].sum()))


def _other_workloads(args, world, dev, stream, local, peaks, event_ms=None):
    """The other large workloads, timed the same way with fewer steps: their
    graph-replay throughput, FFN roofline and the permute / combine / route
    fractions of HBM (the 70% HBM targets of the permute and combine apply on each)."""
    out = {}
    for name in [n for n in args.also.split(",") if n and n != args.config]:
        spec = wl.CONFIGS[name]
        d = wl.make_inputs(spec)
        layer, serial = _build_layers(spec, d, dev)
        inp = _inputs_on(spec, d, dev)
        steps = max(3, args.also_steps)
        ev = _time_eager(serial, inp, steps, args.warmup, world, dev, stream, local)
        gr = None if args.no_graph else _time_graph(layer, spec, d, inp, steps, args.warmup, world, dev, local)
        gst = None if args.no_graph else _time_stages_graph(serial, inp, steps, args.warmup, dev)
        res = layer.forward(*inp[:4], inp[4], stream=stream)
        active = int((res.expert_counts > 0).sum())
        roof, stages = _roofline_and_stages(spec, inp[4], active, serial.fused_gather, gst or ev["stage_avg"], peaks,
                                            event_ms if gst else None)
        eager_value = spec.T * steps * world / (ev["ms_max"] * 1e-3)
        best = gr if gr is not None and gr["ms_per_step"] < ev["ms_max"] / steps else None
        out[name] = {
            "value": best["value"] if best else eager_value, "unit": "tokens/s",
            "ms_per_step": best["ms_per_step"] if best else ev["ms_max"] / steps,
            "timed_path": "graph replay" if best else "eager, one stream", "steps": steps,
            "eager_ms_per_step": ev["ms_max"] / steps,
            "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "ms")},
            "stages": {k: {kk: round(vv, 5) for kk, vv in v.items()} for k, v in stages.items()},
            "stages_timed_in": "one-stream graph replay" if gst else "eager one-stream forwards",
            "clocks": (best or ev)["clocks"],
        }
        del layer, serial, res, d
        torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    from token_expert_routing_gb300 import _abi

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = wl.CONFIGS[args.config]
    d = wl.make_inputs(spec)
    layer, serial = _build_layers(spec, d, dev)
    inp = _inputs_on(spec, d, dev)
    x, ids, kpt, k, P = inp
    per_token = bool(spec.k_choices)
    stream = torch.cuda.current_stream(dev)

    ev = _time_eager(serial, inp, args.steps, args.warmup, world, dev, stream, local)
    ms_max, stage_avg, per_step = ev["ms_max"], ev["stage_avg"], ev["per_step"]
    graph = None if args.no_graph else _time_graph(layer, spec, d, inp, args.steps, args.warmup, world, dev, local)
    graph_stages = None if args.no_graph else _time_stages_graph(serial, inp, args.steps, args.warmup, dev)

    # end to end through the public API: pinned host inputs in, host output back,
    # every step (GraphPipeline: one graph replay per step; HostPipeline: eager)
    e2e = e2e_eager = None
    if not args.no_e2e:
        from token_expert_routing_gb300 import GraphPipeline, HostPipeline
        x_h = d["x"].pin_memory()
        ids_h = d["token_ids"].pin_memory()
        k_h = d["k_per_token"].pin_memory() if per_token else None
        outs = [torch.empty(spec.T, spec.H, dtype=d["x"].dtype).pin_memory() for _ in range(2)]
        h2d = x_h.numel() * x_h.element_size() + ids_h.numel() * 4 + (k_h.numel() * 4 if per_token else 0)
        d2h = outs[0].numel() * outs[0].element_size()

        def run_pipe(submit, sync):
            for i in range(args.warmup):
                submit(i)
            sync()
            _barrier(world)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()           # wall clock: the copies run on their own stream
            for i in range(args.steps):
                submit(i)
            sync()
            return _max_over_ranks(world, (time.perf_counter() - t0) * 1e3)

        pipe = HostPipeline(layer, stream=stream)
        ms_e = run_pipe(lambda i: pipe.submit(x_h, ids_h, outs[i % 2], k_h, k), pipe.synchronize)
        e2e_eager = {"value": spec.T * args.steps * world / (ms_e * 1e-3), "unit": "tokens/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "how": "HostPipeline.submit per step: eager forward, uploads and readbacks on a copy stream "
                            "overlapped with compute; host wall clock"}
        e2e = e2e_eager
        if not args.no_graph:
            gp = GraphPipeline(layer, spec.T, None if per_token else spec.k, d["k_per_token"] if per_token else None,
                               stream=stream)
            ms_g = run_pipe(lambda i: gp.submit(x_h, ids_h, outs[i % 2]), gp.synchronize)
            e2e = {"value": spec.T * args.steps * world / (ms_g * 1e-3), "unit": "tokens/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "how": "GraphPipeline.submit per step (pinned inputs in, output back): one graph replay per "
                          "step, uploads and readbacks on a copy stream overlapped with compute across steps; "
                          "host wall clock from the first submit to the last readback"}
            del gp

    around = None if args.no_around else _time_around_layer(args, spec, d, layer, dev, stream)

    peaks = _peaks()
    event_ms = None if args.no_graph else _event_node_overhead(dev)
    others = None if args.no_also else _other_workloads(args, world, dev, stream, local, peaks, event_ms)

    if rank != 0:
        return
    res = layer.forward(x, ids, kpt, k, P, stream=stream)
    active = int((res.expert_counts > 0).sum())
    counts = res.counts.cpu().numpy()
    roofline, stages = _roofline_and_stages(spec, P, active, serial.fused_gather, graph_stages or stage_avg, peaks,
                                            event_ms if graph_stages else None)
    _, stages_eager = _roofline_and_stages(spec, P, active, serial.fused_gather, stage_avg, peaks)
    roofline["timed_in"] = ("the one-stream forward captured as a CUDA graph, events between its steps (one "
                            "replay per step, mean over the replays)" if graph_stages else
                            "eager one-stream forwards, events between the steps")
    cpu = None
    if not args.no_cpu_baseline:
        n_cpu = min(args.cpu_tokens, spec.T)
        rate, dt = cpu_oracle_rate(d, n_cpu)
        cpu = _cpu_desc(rate, f"first {n_cpu} of {spec.T} tokens of {spec.name}, one pass "
                              f"({dt:.1f} s, float64 numpy oracle)")
        cpu["single_thread"] = _single_thread_baseline()

    total_tokens = spec.T * args.steps * world
    eager = {"value": total_tokens / (ms_max * 1e-3), "unit": "tokens/s", "ms_per_step": ms_max / args.steps,
             "ms_median": per_step[len(per_step) // 2], "ms_min": per_step[0], "ms_max": per_step[-1],
             "how": "MoELayer.forward per step, its steps serialised on one stream (one library call per step "
                    "of the layer; per-step events give the stages and the roofline)",
             "clocks": ev["clocks"]}
    best = graph if graph is not None and graph["ms_per_step"] < eager["ms_per_step"] else eager
    line = {
        "metric": METRIC, "value": best["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": best["ms_per_step"],
        "timed_path": best["how"], "eager": eager,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic", "config": _config(spec),
        "e2e": e2e,
        "e2e_eager": e2e_eager,
        "graph": graph,
        "gpu_launches": ev["launches"],
        "host_enqueue_ms_per_step": ev["host_ms"],
        "roofline": roofline,
        "stages": stages,
        "stages_eager": stages_eager,
        "stages_event_overhead_ms": event_ms,
        "stages_event_overhead_how": ("what an event pair adds to one kernel inside a CUDA graph: a small combine "
                                      "20x back to back against 20x each between its own event pair; ms_net and "
                                      "frac_*_net are the graph-timed stages less this"),
        "cpu_baseline": cpu,
        "clocks": best["clocks"],
        "local_activation_rate": float(np.trace(counts) / counts.sum()),
        "around_layer": around,
        "other_workloads": others,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=wl.BENCH_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=512,
                    help="tokens per step of the CPU oracle sample")
    ap.add_argument("--cpu-tokens", type=int, default=4096,
                    help="tokens of the one-pass CPU oracle baseline (capped at T)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) timing")
    ap.add_argument("--no-around", action="store_true",
                    help="skip timing the scheduling steps around the layer")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--also", default="dsv2lite_prefill_T4096,prism_subexpert_T8192",
                    help="other workloads timed in the same run (comma-separated; reported under other_workloads)")
    ap.add_argument("--also-steps", type=int, default=10)
    ap.add_argument("--no-also", action="store_true", help="time the --config workload only")
    ap.add_argument("--oracle-single-thread", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_single_thread:   # child process of the CPU baseline: one BLAS thread
        print(json.dumps(oracle_single_thread()), flush=True)
        return
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    world, rank, local = _dist()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
