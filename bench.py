"""Benchmark of the decode-step MoE block on GB300.

Headline: one step = one decode token (T = 1) through the 36-layer MoE stack
of the sharded-shape workload: H=2048, 256 experts, top-8, I=128 per expert,
shared expert I=128, fp16, weights ~N(0, 0.02), x ~N(0, 1).  Each layer has
its own weights (405 MB, 14.6 GB in all, far above the 129 MB L2) and each
step uses one of four pre-generated input sets, so routing differs from step
to step.  The 36 single-launch layer kernels of a step are captured in a CUDA
graph (chained with programmatic dependent launch) and replayed; every layer
still reads its input only after the previous layer's kernel has completed.
The timed region (K steps) is repeated and the median reported.  Beside it:
the same stack chained through the residual add (layer l+1 reads
x_l + MoE_l(x_l), written by layer l's kernel), and a ``workloads`` object
with every other seeded configuration (tiny, full-width decode, small-batch
T = 2..64, chunked prefill T = 512 / 4096), each timed the same way.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead
(single-threaded fp64) on K steps, each a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs an independent replica ("replicas
only": the T = 1 block does not shard); value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth  # noqa: E402

METRIC = "MoE decode layer µs & achieved HBM GB/s (% of GB300 peak) at T=1; tokens/s"
NX = 4  # input sets rotated across steps


def algorithmic_bytes(wl, T=1) -> int:
    """Bytes one T=1 layer must move: router, the k selected experts' W13 and W2
    rows, the shared expert (and gate vector), x in and out."""
    H, E, k, I, Is = wl.hidden, wl.n_experts, wl.top_k, wl.inter, wl.shared_inter
    n = E * H + k * 2 * I * H + k * H * I + 2 * Is * H + H * Is + (H if wl.has_shared_gate else 0)
    return 2 * n + 2 * T * H * 2


def code_lines(text):
    """The lines of a C++/CUDA source with // comments, trailing blanks and
    empty lines removed (a '//' after an odd number of quotes is inside a
    string and kept), so that comment-only edits keep the hash."""
    out = []
    for line in text.splitlines():
        i = line.find("//")
        while i >= 0 and line.count('"', 0, i) % 2 == 1:
            i = line.find("//", i + 2)
        code = (line[:i] if i >= 0 else line).rstrip()
        if code:
            out.append(code)
    return out


def kernel_source_hash(read=None) -> str:
    """Hash of the code (comments excluded) the single-launch decode kernel is
    built from."""
    import hashlib
    h = hashlib.sha256()
    for f in ("moe_decode.cu", "moe_common.cuh"):
        if read is None:
            with open(os.path.join(ROOT, "moe_decode_expert_gb300", "csrc", f)) as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update("\n".join(code_lines(text)).encode())
    return h.hexdigest()[:16]


def profiled_traffic(wl):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel changed since."""
    p = os.path.join(ROOT, "profiles", f"decode_fused_kernel_{wl.name}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        pj = json.load(f)
    if pj.get("kernel_source_hash") != kernel_source_hash():
        return None
    per_layer = pj.get("dram_bytes_per_launch")
    return per_layer


def cpu_info() -> dict:
    """Host CPU model and online core count (for the CPU-baseline records)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"cpu_model": model or platform.processor() or platform.machine(), "nproc": os.cpu_count()}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def reduce_max(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ oracle
def oracle_inputs(wl, layers, get_layer):
    """Host inputs of the CPU oracle for one token per layer: x, router, the
    selected experts only (the oracle routes on the host first) and the shared
    expert.  Prepared outside any timed region."""
    import oracle
    c = oracle.OracleCfg(wl.hidden, wl.n_experts, wl.top_k, wl.inter, wl.shared_inter, wl.dtype,
                         wl.norm_topk, wl.has_shared_gate)
    b = moe_synth.bits
    out = []
    for l in range(layers):
        g = get_layer(l)
        x, wr = b(g["x"]), b(g["router_w"])
        _, ids, _ = oracle.router(c, x[0], wr)
        w13 = {int(e): b(g["w13"][int(e)]) for e in ids}
        w2 = {int(e): b(g["w2"][int(e)]) for e in ids}
        out.append((x, wr, w13, w2, b(g["shared_w13"]), b(g["shared_w2"]), b(g["shared_gate_w"])))
        del g
    return c, out


def oracle_layer_tokens(c, inputs, n, start=0):
    """Run the oracle on n (layer, token) samples, cycling through the layers;
    returns the seconds spent."""
    import oracle
    t0 = time.perf_counter()
    for j in range(n):
        oracle.moe_forward(c, *inputs[(start + j) % len(inputs)])
    return time.perf_counter() - t0


def run_reference(args, wl, ws_, rank):
    """The oracle (single-threaded fp64, as it stands) as the reference arm:
    W untimed warm-up steps, then exactly K timed steps, each step one token
    through n_s of the 36 layers (n_s sized so the whole run stays within a
    few minutes); value = tokens/s scaled to the 36-layer stack."""
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    c, inputs = oracle_inputs(wl, wl.layers, lambda l: moe_synth.make_layer(wl, l, 1, device=dev))
    t1 = oracle_layer_tokens(c, inputs, 2) / 2  # calibration (untimed)
    budget = 90.0
    n_s = max(1, min(wl.layers, int(budget / max(1e-9, (args.steps + args.warmup) * t1))))
    for i in range(args.warmup):
        oracle_layer_tokens(c, inputs, n_s, i * n_s)
    spent = 0.0
    for i in range(args.steps):
        spent += oracle_layer_tokens(c, inputs, n_s, (args.warmup + i) * n_s)
    s_per_layer = spent / (args.steps * n_s)
    value = 1.0 / (s_per_layer * wl.layers)   # tokens/s through the 36-layer stack
    cpu = cpu_info()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", **cpu,
                         "sample": f"{args.steps} timed steps after {args.warmup} untimed ones; each step is "
                                   f"one token through {n_s} of the {wl.layers} layers (cycling), "
                                   f"{spent:.1f} s of oracle time in all; value scaled to the "
                                   f"{wl.layers}-layer stack"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl, T=None):
    return {"workload": f"{wl.name}: H={wl.hidden} E={wl.n_experts} top-{wl.top_k} I={wl.inter} "
                        f"shared I={wl.shared_inter}{' +sigmoid gate' if wl.has_shared_gate else ''} "
                        f"{'fp16' if wl.dtype == 1 else 'bf16'} T={wl.T if T is None else T}, "
                        f"{wl.layers} layers rotated",
            "T": 1, "layers": wl.layers, "global_batch": 1, "seq_len": 1,
            "parallelism": "replicas",
            "l2": f"inputs larger than L2: {wl.layers} layers x {wl.layer_bytes() / 1e6:.0f} MB of weights, "
                  f"{NX} input sets rotated per step"}


def timed_replays(graphs, stream, steps, repeats):
    """Median over ``repeats`` of the CUDA-event time (ms) of ``steps``
    replays (graph i % len(graphs) at step i), bracketed by synchronisation;
    returns (median, all)."""
    times = []
    for _ in range(repeats):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(steps):
                graphs[i % len(graphs)].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times), times


# -------------------------------------------------------------------- ours
def decode_stack(m, wl, dev, flags, steps, warmup, repeats, chained=False, nx=NX, layers_data=None):
    """Time a T = 1 stack of wl.layers decode layers as CUDA graphs (one per
    input set).  chained: layer l+1 reads layer l's output (MOE_FLAG_RESIDUAL:
    out = x + MoE(x)), starting from the step's input set.  Returns a dict with
    the median us per layer and what the caller needs for more measurements."""
    cfg = m.cfg_from_workload(wl, None, flags | (m.MOE_FLAG_RESIDUAL if chained else 0))
    L, H, k = wl.layers, wl.hidden, wl.top_k
    layers = layers_data or [moe_synth.make_layer(wl, l, 1, device=dev, weights_only=True) for l in range(L)]
    xs = [[moe_synth.make_x(wl, l, 1, dev, seed_base=7919 * s) for l in range(L)] for s in range(nx)]
    outs = torch.empty(L, 1, H, dtype=cfg.out_torch_dtype, device=dev)
    ids = torch.empty(L, 1, k, dtype=torch.int32, device=dev)
    wts = torch.empty(L, 1, k, dtype=torch.float32, device=dev)
    ws = m.alloc_workspace(cfg, 1, dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # inputs were generated on the default stream

    def step(s):
        for l in range(L):
            g = layers[l]
            x = (xs[s][0] if l == 0 else outs[l - 1]) if chained else xs[s][l]
            m.moe_decode_forward(cfg, x, g["router_w"], g["w13"], g["w2"], g["shared_w13"],
                                 g["shared_w2"], g["shared_gate_w"], ids[l], wts[l], outs[l], ws, stream)

    with torch.cuda.stream(stream):
        for s in range(nx):
            step(s)
    torch.cuda.synchronize()
    m.moe_query_status(ws, stream)
    graphs = []
    for s in range(nx):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            step(s)
        graphs.append(gph)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i % nx].replay()
    torch.cuda.synchronize()
    med, all_ms = timed_replays(graphs, stream, steps, repeats)
    m.moe_query_status(ws, stream)
    return {"ms": med, "ms_repeats": all_ms, "us_per_layer": med * 1e3 / (steps * L), "cfg": cfg,
            "layers": layers, "xs": xs, "outs": outs, "ids": ids, "wts": wts, "ws": ws, "stream": stream,
            "graphs": graphs, "step": step}


def hbm_entry(wl, us_layer, alg, peak, extra=None):
    gbs = alg / (us_layer * 1e-6) / 1e9
    d = {"us_per_layer": us_layer, "tokens_per_s": wl.T * 1e6 / us_layer, "algorithmic_bytes_per_layer": alg,
         "hbm_gbs": gbs, "hbm_frac": gbs / peak}
    d.update(extra or {})
    return d


def run_ours(args, wl, ws_n, rank, local):
    import moe_decode_expert_gb300 as m

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    # Fixed inference weights: nothing on the stream writes them, so each layer
    # kernel may start reading its routing-independent weights before it waits
    # for the previous layer (x is still read only after that wait).
    flags = 0 if args.no_static_weights else m.MOE_FLAG_STATIC_WEIGHTS
    L, H, k = wl.layers, wl.hidden, wl.top_k
    K, W = args.steps, args.warmup
    peak, peak_kind = measured_peaks()

    m.moe_reset_stats()
    st = decode_stack(m, wl, dev, flags, 1, 0, 1)  # build + first timing pass (discarded)
    # repeats of the K-step timed region: as asked, or enough for about a
    # second of timed work in all (a steady clock record), at least 5
    R = args.repeats or max(5, min(500, int(1.0 / max(1e-6, K * st["ms"] * 1e-3))))
    # NX eager steps and the NX captured ones went through the launch code
    launches_per_step = m.moe_get_stats()["kernels_launched"] // (2 * NX)
    graphs, stream, ws = st["graphs"], st["stream"], st["ws"]
    with torch.cuda.stream(stream):
        for i in range(W):
            graphs[i % NX].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier(ws_n)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    times = []
    for _ in range(R):
        barrier(ws_n)
        ms, _ = timed_replays(graphs, stream, K, 1)
        times.append(reduce_max(ms, ws_n))
    clk = clocks.stop()
    barrier(ws_n)
    ms_max = statistics.median(times)
    m.moe_query_status(ws, stream)

    # ----------------------------------------- the same stack, layers chained
    chain = decode_stack(m, wl, dev, flags, K, W, R, chained=True, layers_data=st["layers"])
    chain_us = chain["us_per_layer"]

    # ------------------------------------------------ end to end, host buffers
    # The 36 public-API calls of a step captured once in a CUDA graph (as a
    # decode server would); each step copies its inputs from pinned host memory,
    # replays the graph and copies the outputs back, then synchronises.
    cfg, layers, outs, ids, wts = st["cfg"], st["layers"], st["outs"], st["ids"], st["wts"]
    E2E_STEPS = max(20, min(1000, K // 3))
    xh = torch.empty(L, 1, H, dtype=cfg.torch_dtype, pin_memory=True)
    xh.copy_(torch.stack([st["xs"][0][l] for l in range(L)]).cpu())
    xd = torch.empty(L, 1, H, dtype=cfg.torch_dtype, device=dev)
    oh = torch.empty(L, 1, H, dtype=cfg.out_torch_dtype, pin_memory=True)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        for l in range(L):
            g = layers[l]
            m.moe_decode_forward(cfg, xd[l], g["router_w"], g["w13"], g["w2"], g["shared_w13"],
                                 g["shared_w2"], g["shared_gate_w"], ids[l], wts[l], outs[l], ws, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            xd.copy_(xh, non_blocking=True)
            ge.replay()
            oh.copy_(outs, non_blocking=True)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(ws_n)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(E2E_STEPS):
            xd.copy_(xh, non_blocking=True)
            ge.replay()
            oh.copy_(outs, non_blocking=True)
            stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, ws_n)
    m.moe_query_status(ws, stream)

    # ----------------------------------------------------------- CPU oracle
    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        c, inputs = oracle_inputs(wl, L, lambda l: {**layers[l], "x": st["xs"][0][l]})
        n = 0
        spent = 0.0
        while spent < args.cpu_seconds and n < 4 * L:
            spent += oracle_layer_tokens(c, inputs, 1, n)
            n += 1
        cpu = {"value": 1.0 / (spent / n * L), "unit": "tokens/s", "cores": 1, "kind": "oracle", **cpu_info(),
               "sample": f"{n} layer-tokens of the workload ({spent:.1f} s single-threaded fp64), "
                         f"scaled to the {L}-layer step"}
    del st, chain, ge
    torch.cuda.empty_cache()

    workloads = None
    if ws_n == 1 and not args.no_workloads and wl.name == "sharded_decode":
        workloads = run_workloads(args, m, dev, peak)

    if rank != 0:
        return
    tokens = K * ws_n
    value = tokens / (ms_max / 1e3)
    us_layer = ms_max * 1e3 / (K * L)
    alg = algorithmic_bytes(wl)
    achieved = alg / (us_layer * 1e-6) / 1e9
    traffic = profiled_traffic(wl)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_n, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if wl.dtype == 1 else "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) x)",
        "config": {**config_of(wl), "static_weights_flag": not args.no_static_weights},
        "repeats": R, "ms_per_step_repeats": [t / K for t in times],
        "us_per_layer": us_layer,
        "us_per_layer_chained_residual": chain_us,
        "hbm_gbs": achieved,
        "hbm_frac_of_peak": achieved / peak,
        "kernels_per_layer": launches_per_step // L,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "decode_fused_kernel",
                     "algorithmic_bytes_per_launch": alg, "peak_kind": f"{peak_kind} (hbm_gbs)"},
        "cpu_baseline": cpu,
        "e2e": {"value": E2E_STEPS * ws_n / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": L * H * 2, "d2h_bytes_per_step": L * H * outs.element_size(),
                "path": "36 moe_decode_forward calls captured once in a CUDA graph; per step: pinned H2D of x, "
                        "graph replay, D2H of out, stream synchronise"},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)
def grouped_bytes(wl, T, n_distinct):
    """Algorithmic bytes of one T-token grouped layer: router, each distinct
    selected expert's W13 and W2 once, the shared expert (+gate), x and out."""
    H, E, I, Is = wl.hidden, wl.n_experts, wl.inter, wl.shared_inter
    n = E * H + n_distinct * 3 * I * H + 3 * Is * H + (H if wl.has_shared_gate else 0)
    return 2 * n + 2 * 2 * T * H


def grouped_flops(wl, T):
    H, E, k, I, Is = wl.hidden, wl.n_experts, wl.top_k, wl.inter, wl.shared_inter
    return 2 * T * (E * H + k * 3 * I * H + 3 * Is * H)


GROUPED_PATH_FLAGS = {"auto": 0, "simt": 1, "tc": 2, "single": 16}  # MOE_FLAG_GROUPED_* bits


def grouped_stack(m, wl, T, layers, dev, steps, warmup, repeats, xs=None, flags=0):
    """Time one grouped forward of T tokens through every layer (a CUDA graph
    of len(layers) calls); returns (median ms per step, kernels per layer,
    path, mean distinct experts per layer)."""
    cfg = m.cfg_from_workload(wl, None, flags)
    L, H, k = len(layers), wl.hidden, wl.top_k
    xs = xs or [moe_synth.make_x(wl, l, T, dev) for l in range(L)]
    outs = torch.empty(L, T, H, dtype=cfg.out_torch_dtype, device=dev)
    ids = torch.empty(L, T, k, dtype=torch.int32, device=dev)
    wts = torch.empty(L, T, k, dtype=torch.float32, device=dev)
    ws = m.alloc_workspace(cfg, T, dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))

    def step():
        for l in range(L):
            g = layers[l]
            m.moe_grouped_forward(cfg, xs[l], g["router_w"], g["w13"], g["w2"], g["shared_w13"],
                                  g["shared_w2"], g["shared_gate_w"], ids[l], wts[l], outs[l], ws, stream)

    m.moe_reset_stats()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    m.moe_query_status(ws, stream)
    stats = m.moe_get_stats()
    gph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            gph.replay()
    torch.cuda.synchronize()
    med, _ = timed_replays([gph], stream, steps, repeats)
    m.moe_query_status(ws, stream)
    distinct = [int(torch.unique(ids[l]).numel()) for l in range(L)]
    kpl = stats["kernels_launched"] // L
    if stats["grouped_tc_calls"]:
        path = "tcgen05"
    elif stats["grouped_calls"]:
        path = "single-launch batch kernel" if kpl == 1 else "cuda-core"
    else:
        path = "decode"
    return med, kpl, path, distinct


def run_workloads(args, m, dev, peak):
    """Every other seeded configuration, each as a CUDA graph over its layers
    with inputs far larger than L2 (except the tiny one, which is L2-resident
    and reported as latency only): median of 3 timed repeats."""
    out = {}
    R = 3
    flags = m.MOE_FLAG_STATIC_WEIGHTS
    tc_peak, tc_sus = tensor_peak(), tensor_peak(sustained=True)

    # tiny: one layer (its selected weights, ~200 KB, sit in L2), launched 36
    # times in a chained graph so the figure is the per-layer latency, not the
    # cost of replaying a one-launch graph
    wl = moe_synth.workload("tiny", layers=36)
    tiny = [moe_synth.make_layer(wl, 0, 1, device=dev, weights_only=True)] * wl.layers
    st = decode_stack(m, wl, dev, flags, 200, 20, R, nx=NX, layers_data=tiny)
    out["tiny"] = {"us_per_layer": st["us_per_layer"], "tokens_per_s": 1e6 / st["us_per_layer"],
                   "l2_resident": True, "note": "one layer's weights launched 36 times per graph; latency only: "
                                                "the roofline fraction is not meaningful in L2"}
    del st, tiny

    # full-width decode, T = 1: 36 layers (1.62 GB each), independent and chained
    wl = moe_synth.workload("full_decode")
    layers = [moe_synth.make_layer(wl, l, 1, device=dev, weights_only=True) for l in range(wl.layers)]
    st = decode_stack(m, wl, dev, flags, 100, 10, R, layers_data=layers)
    ch = decode_stack(m, wl, dev, flags, 100, 10, R, chained=True, layers_data=layers)
    out["full_decode"] = hbm_entry(wl, st["us_per_layer"], algorithmic_bytes(wl), peak,
                                   {"us_per_layer_chained_residual": ch["us_per_layer"], "layers": wl.layers,
                                    "kernels_per_layer": 1})
    del st, ch

    # small batch, T = 2..64: the same 36 full-width weight sets (same shapes
    # and distribution), each layer with the Zipf-biased router and x of the
    # small-batch recipe
    wls = moe_synth.workload("small_batch")
    sb_layers = [{**layers[l], "router_w": moe_synth.make_router(wls, l, dev)} for l in range(wls.layers)]
    out["small_batch"] = {}
    for T in wls.t_values:
        steps = max(20, int(0.3e6 / (36 * (30 + 1.1 * T))))
        med, kpl, path, distinct = grouped_stack(m, wls, T, sb_layers, dev, steps, 5, R)
        us = med * 1e3 / (steps * wls.layers)
        alg = sum(grouped_bytes(wls, T, u) for u in distinct) / len(distinct)
        wlT = moe_synth.workload("small_batch", T=T)
        out["small_batch"][f"T={T}"] = hbm_entry(wlT, us, alg, peak, {
            "kernels_per_layer": kpl, "path": path, "mean_distinct_experts": sum(distinct) / len(distinct)})
    del sb_layers

    # chunked prefill, T = 512 / 4096: 4 layers (full-width weight sets 0-3)
    # with the prefill router (logits ~ N(0, 1))
    wlp = moe_synth.workload("chunked_prefill")
    cp_layers = [{**layers[l], "router_w": moe_synth.make_router(wlp, l, dev)} for l in range(wlp.layers)]
    del layers
    torch.cuda.empty_cache()
    out["chunked_prefill"] = {}
    for T in wlp.t_values:
        steps = max(10, int(0.3e6 / (4 * 1.3 * T)))
        med, kpl, path, distinct = grouped_stack(m, wlp, T, cp_layers, dev, steps, 3, R)
        us = med * 1e3 / (steps * wlp.layers)
        alg = sum(grouped_bytes(wlp, T, u) for u in distinct) / len(distinct)
        tfl = grouped_flops(wlp, T) / (us * 1e-6) / 1e12
        wlT = moe_synth.workload("chunked_prefill", T=T)
        out["chunked_prefill"][f"T={T}"] = hbm_entry(wlT, us, alg, peak, {
            "kernels_per_layer": kpl, "path": path, "tensor_tflops": tfl, "tensor_frac": tfl / tc_peak,
            "tensor_frac_of_sustained": tfl / tc_sus, "tensor_peak_tflops": tc_peak})
    del cp_layers
    torch.cuda.empty_cache()
    out["note"] = ("small_batch and chunked_prefill reuse the full-width layers' expert and shared weights (same "
                   "shapes and N(0, 0.02) recipe) with their own seeded routers and inputs; peak = measured "
                   "hbm_gbs and bf16_tflops (burst)")
    return out


def run_grouped(args, wl, ws_n, rank, local):
    """T > 1 workloads (small-batch decode, chunked prefill) on their own: one
    step = one grouped forward of T tokens through every layer."""
    import moe_decode_expert_gb300 as m

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    T = args.T or wl.T
    layers = [moe_synth.make_layer(wl, l, T, device=dev) for l in range(wl.layers)]
    xs = [g.pop("x") for g in layers]
    K, W = args.steps, args.warmup
    clocks = ClockSampler(local)
    barrier(ws_n)
    clocks.start()
    time.sleep(0.3)
    med, kpl, path, distinct = grouped_stack(m, wl, T, layers, dev, K, W, args.repeats or 5, xs=xs,
                                             flags=GROUPED_PATH_FLAGS[args.grouped_path])
    clk = clocks.stop()
    ms_max = reduce_max(med, ws_n)
    if rank != 0:
        return
    L = wl.layers
    alg = sum(grouped_bytes(wl, T, u) for u in distinct) / L
    us_layer = ms_max * 1e3 / (K * L)
    peak, peak_kind = measured_peaks()
    achieved = alg / (us_layer * 1e-6) / 1e9
    tflops = grouped_flops(wl, T) / (us_layer * 1e-6) / 1e12
    tc_peak = tensor_peak()
    line = {
        "metric": f"MoE grouped layer µs & achieved HBM GB/s at T={T}; tokens/s", "value": T * K * ws_n / (ms_max / 1e3),
        "unit": "tokens/s", "n_gpus": ws_n, "steps": K, "warmup": W, "ms_per_step": ms_max / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)", "config": {**config_of(wl, T), "T": T, "path": path,
                                                 "mean_distinct_experts": sum(distinct) / L},
        "us_per_layer": us_layer, "hbm_gbs": achieved, "hbm_frac_of_peak": achieved / peak,
        "kernels_per_layer": kpl,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "algorithmic_bytes_per_layer": alg, "peak_kind": f"{peak_kind} (hbm_gbs)",
                     "tensor_tflops": tflops, "tensor_peak_tflops": tc_peak, "tensor_frac": tflops / tc_peak},
        "gpu_launches": K * L * kpl, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def tensor_peak(sustained=False):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained" if sustained and "bf16_tflops_sustained" in d else "bf16_tflops"])
    return 1700.0 if sustained else 1900.0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sharded_decode",
                    choices=["sharded_decode", "full_decode", "tiny", "small_batch", "chunked_prefill"])
    ap.add_argument("--T", type=int, default=None, help="tokens per step for the T > 1 workloads")
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=0,
                    help="timed regions of K steps, the median reported (0: at least 5, about 1 s in all)")
    ap.add_argument("--no-workloads", action="store_true", help="headline workload only")
    ap.add_argument("--grouped-path", default="auto", choices=sorted(GROUPED_PATH_FLAGS),
                    help="T > 1 path of --workload small_batch / chunked_prefill (auto: the library's choice)")
    ap.add_argument("--no-static-weights", action="store_true",
                    help="T=1: do not let layer kernels read weights before the previous layer completes")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = moe_synth.workload(args.workload)
    if args.layers:
        wl = moe_synth.workload(args.workload, layers=args.layers)
    ws_n, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, wl, ws_n, rank)
    elif wl.T > 1:
        run_grouped(args, wl, ws_n, rank, local)
    else:
        run_ours(args, wl, ws_n, rank, local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
