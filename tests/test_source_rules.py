"""Source-level checks of the ordering rule under programmatic dependent
launch (no GPU): every kernel of the library may be scheduled while the
previous kernel on the stream still runs, and reads what earlier kernels wrote
only after griddepcontrol.wait.  To the compiler that wait is inline asm, so
such reads must be loads it cannot move above it: no `const T* __restrict__`
kernel parameter (an invariant load to the compiler) and no non-volatile asm
load.  A load of the tile count scheduled above the wait once gave all-zero
outputs in the parity tests; these checks keep the rule from regressing."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "moe_decode_expert_gb300", "csrc")


def _sources():
    files = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")))
    assert files, CSRC
    return {os.path.basename(f): open(f).read() for f in files}


def _kernel_signatures(text):
    """(name, parameter list) of every __global__ function in a source."""
    out = []
    text = re.sub(r"__launch_bounds__\s*\([^)]*\)", "", text)
    for mt in re.finditer(r"__global__[^(]*?\b(\w+)\s*\(", text):
        depth, i = 1, mt.end()
        while depth:
            depth += {"(": 1, ")": -1}.get(text[i], 0)
            i += 1
        out.append((mt.group(1), text[mt.end():i - 1]))
    return out


def test_kernels_found():
    names = {n for src in _sources().values() for n, _ in _kernel_signatures(src)}
    for k in ("decode_fused_kernel", "route_group_kernel", "tc_w13_kernel", "tc_w2_kernel", "combine_kernel",
              "router_mma_kernel", "router_topk_kernel", "group_kernel", "tc_fill_kernel"):
        assert k in names, k


def test_no_const_restrict_kernel_parameters():
    bad = []
    for f, src in _sources().items():
        for name, params in _kernel_signatures(src):
            if re.search(r"\bconst\s+[\w:]+\s*\*\s*__restrict__", params):
                bad.append(f"{f}:{name}")
    assert not bad, f"const __restrict__ parameters may be read before griddepcontrol.wait: {bad}"


def test_asm_loads_are_volatile():
    bad = []
    for f, src in _sources().items():
        for mt in re.finditer(r"\basm\s*(volatile)?\s*\(\s*\"([^\"]*)", src):
            if not mt.group(1) and re.search(r"\bld\.", mt.group(2)):
                bad.append(f"{f}: {mt.group(2)[:40]}")
    assert not bad, f"non-volatile asm loads can be hoisted above griddepcontrol.wait: {bad}"
