"""Per-phase timeline of the single-launch decode kernels (T = 1, and the
batch kernel for 2 <= T <= 8 with ``--T``).

Builds the phase-trace variant of the library (the same kernels, compiled
with ``-DMOE_PHASE_TRACE``: thread 0 of every CTA stores the GPU global time
at fixed points), runs ``--layers`` layers of a workload as one CUDA graph of
chained launches (programmatic dependent launch, static weights, as in the
benchmark), replays it, and prints for every stamp its time after the
previous layer's last CTA wrote its output: the median CTA and the latest
CTA, each the median over the traced launches.

    python -m moe_decode_expert_gb300.trace_phases --workload sharded_decode
    python -m moe_decode_expert_gb300.trace_phases --workload small_batch --T 2
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

EVENTS = [
    "entry",
    "PDL wait released",
    "x staged",
    "phase-1 dot products summed",
    "phase-1 results published",
    "logits gathered (warp 0)",
    "ranked",
    "routing weights ready (warp 0)",
    "phase-3 work done (thread 0)",
    "5/8 of the CTAs counted in (thread 0)",
    "W2 copies landed",
    "activations gathered (warp 0)",
    "terms written (warp 0)",
    "combine steps done (warp 0)",
    "output written",
]
EVENTS_BATCH = [
    "entry",
    "PDL wait released",
    "x staged",
    "phase-1 dot products summed",
    "phase-1 results published",
    "logits gathered (warp 0)",
    "ranked, union formed",
    "phase-3 passes done",
    "activations published (flags in)",
    "terms written",
    "warp 0's units done",
    "thread 0's outputs written",
    "first pass's dot products done (thread 0)",
    "second pass done",
    "third pass done",
    "warp 0's top-k done",
    "every token ranked",
    "union formed (warp 0)",
    "warp 0's first W2 unit landed",
    "warp 0's first W2 unit computed",
]


def trace(workload: str, layers: int, replays: int, static_weights: bool = True, T: int = 1) -> dict:
    from moe_decode_expert_gb300 import _build
    import moe_decode_expert_gb300 as m
    import moe_synth

    m.use_library(_build.build(trace=True))
    lib = m.library()
    lib.moe_trace_reset.restype = ctypes.c_int
    lib.moe_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    lib.moe_trace_read.restype = ctypes.c_int
    geo = [ctypes.c_int() for _ in range(3)]
    lib.moe_trace_geometry(*[ctypes.byref(g) for g in geo])
    slots, nctas, ring = (g.value for g in geo)
    if layers > ring:
        raise ValueError(f"at most {ring} layers")

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = moe_synth.workload(workload, layers=layers)
    flags = (m.MOE_FLAG_STATIC_WEIGHTS if static_weights else 0) | (m.MOE_FLAG_GROUPED_SINGLE if T > 1 else 0)
    cfg = m.cfg_from_workload(wl, None, flags)
    H, k = wl.hidden, wl.top_k
    lay = [moe_synth.make_layer(wl, l, T, device=dev) for l in range(layers)]
    outs = torch.empty(layers, T, H, dtype=cfg.out_torch_dtype, device=dev)
    ids = torch.empty(layers, T, k, dtype=torch.int32, device=dev)
    wts = torch.empty(layers, T, k, dtype=torch.float32, device=dev)
    ws = m.alloc_workspace(cfg, T, dev)
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream(dev))

    def step():
        for l in range(layers):
            g = lay[l]
            fwd = m.moe_decode_forward if T == 1 else m.moe_grouped_forward
            fwd(cfg, g["x"], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                g["shared_gate_w"], ids[l], wts[l], outs[l], ws, st)

    with torch.cuda.stream(st):
        step()
    torch.cuda.synchronize()
    m.moe_query_status(ws, st)
    names = EVENTS if T == 1 else EVENTS_BATCH
    events = dict(enumerate(names))
    last = len(EVENTS) - 1 if T == 1 else 11  # "output written"
    if lib.moe_trace_reset() != 0:
        raise RuntimeError("moe_trace_reset failed")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        step()  # launch l records into ring entry l
    with torch.cuda.stream(st):
        for _ in range(replays):
            graph.replay()
    torch.cuda.synchronize()
    m.moe_query_status(ws, st)
    buf = np.zeros(ring * nctas * slots, np.uint64)
    if lib.moe_trace_read(buf.ctypes.data, buf.size) != 0:
        raise RuntimeError("moe_trace_read failed")
    rec = buf.reshape(ring, nctas, slots)[:layers].astype(np.int64)
    used = rec[0, :, 0] != 0
    rec = rec[:, used, :]
    rows = []
    per_launch = []
    for l in range(1, layers):
        ref = rec[l - 1, :, last].max()
        rel = np.where(rec[l] != 0, (rec[l] - ref) / 1e3, np.nan)  # us; nan where not stamped
        with np.errstate(all="ignore"):
            per_launch.append((np.nanmedian(rel, axis=0), np.nanmax(rel, axis=0)))
    with np.errstate(all="ignore"):
        med = np.nanmedian(np.stack([p[0] for p in per_launch]), axis=0)
        late = np.nanmedian(np.stack([p[1] for p in per_launch]), axis=0)
    for e, name in sorted(events.items()):
        have = rec[1:, :, e] != 0
        if not have.any():
            continue  # not stamped on this shape
        rows.append({"event": name, "median_cta_us": float(med[e]), "last_cta_us": float(late[e]),
                     "ctas": int(have[0].sum())})
    span = [float((rec[l, :, last].max() - rec[l - 1, :, last].max()) / 1e3) for l in range(1, layers)]
    return {"workload": workload, "T": T, "kernel": "decode_fused_kernel" if T == 1 else "decode_batch_kernel",
            "layers": layers, "replays": replays, "ctas": int(used.sum()),
            "static_weights": static_weights, "layer_us_median": float(np.median(span)), "events": rows}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="sharded_decode",
                    choices=["tiny", "sharded_decode", "full_decode", "small_batch"])
    ap.add_argument("--T", type=int, default=None, help="tokens (1, or 2..8 for the batch kernel)")
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--replays", type=int, default=20)
    ap.add_argument("--no-static-weights", action="store_true")
    ap.add_argument("--json", default=None, help="also write the result here")
    a = ap.parse_args()
    T = a.T if a.T is not None else (2 if a.workload == "small_batch" else 1)
    r = trace(a.workload, a.layers, a.replays, not a.no_static_weights, T)
    print(f"{r['workload']} T = {T} ({r['kernel']}): {r['ctas']} CTAs, {r['layers']} chained layers, median layer "
          f"{r['layer_us_median']:.2f} us (last output to last output)")
    print(f"{'us after the previous layer ends':>34} | {'median CTA':>10} | {'last CTA':>9} | CTAs")
    for e in r["events"]:
        print(f"{e['event']:>34} | {e['median_cta_us']:10.2f} | {e['last_cta_us']:9.2f} | {e['ctas']}")
    if a.json:
        with open(a.json, "w") as f:
            json.dump(r, f, indent=1)


if __name__ == "__main__":
    main()
