"""Library pins of the oracle: torch's own FSDP1 (FlatParameter) and FSDP2
(fully_shard, Shard(0)) on gloo CPU ranks compute the same layout, the same
reduce-scatter mean and, within a band, the same AdamW result as the oracle.

This is the pages' own check ("NCCL ZeRO/FSDP state sharding", section
全模式性能结果与限制: FSDP results equal the replicated run) and their way of
testing multi-rank behaviour without GPUs ("第18章 FSDP：ZeRO 风格的参数分片"
§18.8/§18.14: two gloo processes on one machine), with torch as the reference.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

WORKER = os.path.join(os.path.dirname(__file__), "fsdp_gloo_worker.py")
HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def run_torch_fsdp(tmp_path, mode, n, shapes, steps, seed=1):
    spec = ",".join("x".join(str(d) for d in s) if s else "scalar" for s in shapes)
    cmd = [sys.executable, WORKER, "--mode", mode, "--n", str(n), "--shapes", spec, "--steps", str(steps),
           "--seed", str(seed), "--port", str(free_port()), "--out", str(tmp_path)]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    return [torch.load(os.path.join(tmp_path, f"rank{k}.pt")) for k in range(n)]


def pack_full(L, tensors):
    full = np.zeros(L["F"], np.float32)
    for t, x in enumerate(tensors):
        x = x.detach().numpy().reshape(-1).astype(np.float32)
        full[L["t_full_off"][t]:L["t_full_off"][t] + x.size] = x
    return full


CASES = [
    ("flat", 3, [(5, 3), (4,)]),                  # P = 19: one padding element on rank 2
    ("flat", 4, [(7, 5), (3,), (9, 2)]),          # P = 56: divisible
    ("dim0", 3, [(5, 3), (7,), (2, 4), (1, 6)]),  # rows 5, 7, 2, 1 over 3 ranks
    ("dim0", 4, [(6, 2), (9,), (3, 3)]),          # 6 rows on 4 ranks: 2,2,2,0
]


@pytest.mark.parametrize("mode,n,shapes", CASES)
def test_torch_fsdp_matches_oracle(oracle_lib, tmp_path, mode, n, shapes):
    steps = 3
    outs = run_torch_fsdp(tmp_path, mode, n, shapes, steps)
    omode = oracle.FLAT if mode == "flat" else oracle.DIM0
    sh = oracle.Shapes(shapes)
    L = oracle.layout(sh, n, omode)
    stride = L["S"]

    # (1) layout: local shard sizes
    for r in range(n):
        fi = oracle.full_index(sh, n, omode, r, np.arange(L["S"]))
        if omode == oracle.FLAT:
            assert outs[r]["local_shapes"] == [(L["S"],)]
        else:
            for t, s in enumerate(shapes):
                inner = int(np.prod(s[1:])) if len(s) > 1 else 1
                j = np.arange(L["t_shard_off"][t], L["t_shard_off"][t] + L["t_slot"][t])
                owned_rows = int((fi[j] >= 0).sum()) // inner
                assert outs[r]["local_shapes"][t][0] == owned_rows, (r, t)

    # (2) oracle run on the same inputs
    full0 = pack_full(L, outs[0]["init"])
    master, _ = oracle.reshard(sh, n, omode, full0, stride, True, False)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    gout = np.zeros_like(master)
    for t in range(steps):
        grads = [pack_full(L, outs[r]["grads"][t][0]) for r in range(n)]
        oracle.rs_adamw(sh, n, omode, grads, stride, master, m, v, grad_out=gout, hp=HP, step=t + 1)
        # reduce-scatter result of every rank: torch may sum in another order and FSDP1
        # divides before and after the reduction (by 2 and 1.5 at world size 3), so
        # allow 1e-6 relative plus a few ulps of the ~1e-3 summands (cancellation)
        for r in range(n):
            row = gout[r * stride:(r + 1) * stride]
            if omode == oracle.FLAT:
                got = outs[r]["grad_shards"][t][0].numpy()
                assert got.shape == (L["S"],)
                assert np.allclose(got, row[:L["S"]], rtol=1e-6, atol=2e-10), (t, r)
            else:
                for k, s in enumerate(shapes):
                    got = outs[r]["grad_shards"][t][k].numpy().reshape(-1)
                    o = L["t_shard_off"][k]
                    assert np.allclose(got, row[o:o + got.size], rtol=1e-6, atol=2e-10), (t, r, k)

    # (3) parameters after the steps, all-gathered
    got_full = oracle.unshard(sh, n, omode, master, stride, L["F"])
    ref_full = pack_full(L, outs[0]["final"])
    logical = np.zeros(L["F"], bool)
    for t, s in enumerate(shapes):
        logical[L["t_full_off"][t]:L["t_full_off"][t] + int(np.prod(s) if s else 1)] = True
    err = np.abs(got_full - ref_full)[logical]
    assert (err <= 1e-5 * np.abs(ref_full[logical]) + 1e-8).all(), err.max()
