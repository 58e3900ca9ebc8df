"""The committed ncu summaries against the bench's own byte accounting (host only).

Every profiles/<kernel>_<workload>.json states the fused kernel's algorithmic bytes
per launch and the DRAM bytes ncu measured.  The first must be what bench.py computes
for that workload's layout (the bench reports the second as roofline.traffic), and the
second must sit just under it: DRAM reads equal the algorithmic reads, and writes fall
short only by what is still dirty in L2 when the launch ends (at most the L2's 126 MB),
never above it (a re-read would show as more).  A summary of a workload too large for a
profiler capture holds the capture of a smaller case of the same layout class
(`scaled_from`) and that capture's bytes scaled by the ratio of logical parameters."""
import glob
import json
import os

import pytest
import torch

import bench
import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.json")))
L2_BYTES = 126 * 1024 * 1024


def test_there_are_profiles():
    assert PROFILES


def accounting(name):
    """(algorithmic bytes per launch, algorithmic reads, logical parameters) of the fused
    kernel on a workload, as bench.py counts them."""
    w = synth.workload(name)
    info = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode).info
    gb = 2 if w.grad_dtype == torch.bfloat16 else 4
    pb = 2 if w.param_dtype == torch.bfloat16 else 4
    ab = bench.algorithmic_bytes(w.N, info["numel"], info["shard_numel"], info["full_numel"], w.mode, gb, pb)
    reads = w.N * info["numel"] * gb + 12 * info["numel"]      # gradients + three state arrays
    return ab["rs_adamw"], reads, info["numel"], w


def check_capture(d, name):
    alg, reads, _, _ = accounting(name)
    assert d["algorithmic_bytes_per_launch"] == alg
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    # reads: the algorithmic reads, to within ncu's rounding
    assert abs(d["dram_bytes_read"] - reads) <= 0.002 * reads
    # writes: short of the algorithmic writes by at most one L2 of dirty lines, never over
    writes = alg - reads
    assert writes - L2_BYTES <= d["dram_bytes_write"] <= writes * 1.002


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_matches_the_bench_accounting(path):
    d = json.load(open(path))
    assert os.path.basename(path) == f"{d['kernel'].split('<')[0]}_{d['workload']}.json"
    assert len(d["kernel_src_sha256_16"]) == 16 and d["command"].startswith("ncu ")
    sf = d.get("scaled_from")
    if sf is None:
        check_capture(d, d["workload"])
        return
    # taken on a smaller case of the same layout class (same N, dtypes, mode) and scaled
    # by the ratio of logical parameters: the capture itself must pass the same checks
    check_capture(sf, sf["workload"])
    alg, _, P, w = accounting(d["workload"])
    _, _, p, ws = accounting(sf["workload"])
    assert (w.N, w.mode, w.grad_dtype, w.param_dtype) == (ws.N, ws.mode, ws.grad_dtype, ws.param_dtype)
    assert d["scale"] == pytest.approx(P / p, rel=1e-12)
    assert d["algorithmic_bytes_per_launch"] == alg
    for k in ("dram_bytes_read", "dram_bytes_write"):
        assert d[k] == round(sf[k] * P / p)
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    assert d["dram_bytes_per_launch"] <= alg * 1.002
