"""Host logic of bench.py: the bytes model, and the multi-rank aggregation
(barrier, max over ranks) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import moe_synth


def test_algorithmic_bytes_per_layer():
    assert bench.algorithmic_bytes(moe_synth.workload("sharded_decode")) == 15_212_544
    assert bench.algorithmic_bytes(moe_synth.workload("full_decode")) == 57_683_968


def test_layer_bytes_match_generated_tensors():
    wl = moe_synth.workload("tiny")
    d = moe_synth.make_layer(wl, 0, 1)
    n = sum(v.numel() * v.element_size() for k, v in d.items() if v is not None and k != "x")
    assert n == wl.layer_bytes()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    ws, r, local = bench.dist_setup()
    assert ws == world and r == rank
    bench.barrier(ws)
    m = bench.reduce_max(float(10 * (rank + 1)), ws)
    q.put((rank, m))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 20.0), (1, 20.0)]


def test_grouped_bytes_model():
    wl = moe_synth.workload("small_batch")
    # router + 10 distinct experts (W13 + W2) + shared (W13 + W2 + gate) + x and out for 4 tokens
    H, E, I, Is = 2048, 256, 512, 512
    expect = 2 * (E * H + 10 * 3 * I * H + 3 * Is * H + H) + 2 * 2 * 4 * H
    assert bench.grouped_bytes(wl, 4, 10) == expect
    assert bench.grouped_flops(wl, 1) == 2 * (E * H + 8 * 3 * I * H + 3 * Is * H)


def test_kernel_code_hash_ignores_comments_only():
    """The committed ncu traffic stays valid across comment edits of the
    kernel sources, and is dropped when their code changes."""
    src = 'int f() {  // first\n  return g("a//b");  // the string keeps its slashes\n}\n// trailing note\n'
    same = 'int f() {  // reworded\n\n  return g("a//b");\n}\n'
    changed = 'int f() {  // first\n  return g("a//c");\n}\n'
    h = lambda text: bench.kernel_source_hash(lambda f: text)
    assert bench.code_lines(src) == ['int f() {', '  return g("a//b");', '}']
    assert h(src) == h(same)
    assert h(src) != h(changed)


def test_reference_arm_times_exactly_the_steps_it_reports(capsys):
    """The reference arm (the oracle on the host cores) times K steps after W
    untimed ones and reports them; its per-step time times K stays within the
    oracle time it measured, and the record names the CPU it ran on."""
    import argparse
    import json
    args = argparse.Namespace(steps=3, warmup=1, gpus=1)
    wl = moe_synth.workload("tiny")
    bench.run_reference(args, wl, 1, 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 1
    cb = line["cpu_baseline"]
    assert cb["cores"] == 1 and cb["nproc"] >= 1 and cb["cpu_model"]
    assert "3 timed steps" in cb["sample"]
    assert line["value"] > 0 and line["ms_per_step"] > 0
