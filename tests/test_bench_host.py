"""Host-side parts of bench.py (CPU): the algorithmic byte model, the clock-log
parser, and the max-over-ranks timing reduction on two gloo ranks."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from fsdp_sharded_state_gb300 import synth  # noqa: E402
import fsdp_sharded_state_gb300 as fs  # noqa: E402


def step_bytes(w, n_unshard=2):
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    i = L.info
    gb = 2 if w.grad_dtype == torch.bfloat16 else 4
    pb = 2 if w.param_dtype == torch.bfloat16 else 4
    ab = bench.algorithmic_bytes(w.N, i["numel"], i["shard_numel"], i["full_numel"], w.mode, gb, pb)
    return ab, ab["rs_adamw"] + n_unshard * ab["unshard"], i["numel"]


def test_byte_model_per_element():
    # fp32 parameters and gradients, N = 4: the fused kernel moves 4N + 24 bytes per
    # parameter, an all-gather 8; a FULL_SHARD step 56 bytes per parameter.
    ab, tot, P = step_bytes(synth.mlp128m())
    assert ab["rs_adamw"] == 40 * P and tot == 56 * P
    # bf16 parameters and gradients, fp32 state, N = 8: 2N + 26 and 50 per step.
    ab, tot, P = step_bytes(synth.llama4())
    assert ab["rs_adamw"] == 42 * P and tot == 50 * P
    # SHARD_GRAD_OP: one all-gather fewer
    _, tot1, P = step_bytes(synth.llama4(), n_unshard=1)
    assert tot1 == 46 * P


def test_row_byte_model_per_parameter():
    # the rows' bytes per logical parameter (each array read or written once):
    #   clip:  N gradient replicas, the fp32 shard written, re-read, rewritten clipped,
    #          master/m/v read and written (+ the bf16 parameter written);
    #   accum: per replica the micro-batch read, the fp32 accumulator read and written;
    #   accum_step: per replica the accumulator and the micro-batch read; the state as
    #          in the step;
    #   hsdp:  R x N replicas; R copies of the state (+ R bf16 parameters);
    #   zero1: N replicas; the owner's m, v (and master, or its own fp32 replica); the
    #          updated parameter written into all N replicas.
    # The DRAM reads ncu measured equal the reads counted here: the accumulation on the
    # 128 MiB layout 1.074 GB (32 B per parameter), the fused last micro-batch 1.476 GB
    # (44 B), ZeRO-1 0.940 GB (28 B).
    m = synth.mlp128m()                     # fp32, N = 4
    P = 33554432
    assert bench.row_bytes("clip", m, P, 4) == 52 * P
    assert bench.row_bytes("accum", m, P, 4) == 48 * P
    assert bench.row_bytes("accum_step", m, P, 4) == 56 * P
    assert bench.row_bytes("hsdp", m, P, 4, R=2) == 80 * P
    assert bench.row_bytes("zero1", m, P, 4) == 52 * P
    l4 = synth.llama4()                     # bf16 parameters and gradients, N = 8
    P = 809533440
    assert bench.row_bytes("clip", l4, P, 8) == 54 * P
    assert bench.row_bytes("accum", l4, P, 8) == 80 * P
    assert bench.row_bytes("accum_step", l4, P, 8) == 74 * P
    assert bench.row_bytes("hsdp", l4, P, 8, R=2) == 84 * P
    assert bench.row_bytes("zero1", l4, P, 8) == 56 * P
    with pytest.raises(KeyError):
        bench.row_bytes("nope", m, P, 4)


def test_parse_clocks():
    csv = "\n".join([
        "0, 1965 MHz, 2070 MHz, 900.1 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1980 MHz, 2070 MHz, 910.0 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 345 MHz, 2070 MHz, 100.0 W, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active",
    ])
    c = bench.parse_clocks(csv)
    assert c["sm_max_mhz"] == 2070 and c["sm_mhz"] == pytest.approx(1972.5)
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.parse_clocks("")["samples"] == 0


def _agg_worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=2)
    v = bench.aggregate_max([3.5, 7.25][rank], 2, dist)
    q.put((rank, v))
    dist.destroy_process_group()


def test_aggregate_max_two_gloo_ranks():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    ps = [ctx.Process(target=_agg_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    assert got == [(0, 7.25), (1, 7.25)]
    assert bench.aggregate_max(5.0, 1, None) == 5.0


def test_launch_stats():
    import bench
    s = bench.launch_stats([1.0, 1.0, 1.0, 1.0])
    assert s["median_ms"] == 1.0 and s["p95_ms"] == 1.0 and s["cv"] == 0.0 and not s["cv_flag"]
    s = bench.launch_stats([1.0, 2.0, 3.0, 4.0, 100.0])
    assert s["median_ms"] == 3.0 and s["p95_ms"] == 100.0 and s["cv_flag"] and s["n"] == 5


def test_code_hash_ignores_comments():
    import bench
    a = "int f(int x) {  // comment\n  return x; /* block\n comment */ }\n"
    b = "int f(int x) { return x; }"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only("int a;") != bench.code_only("int b;")


def test_oracle_host_run_spawns_one_process_per_core():
    # the host-wide CPU baseline: spawned processes, each the unmodified oracle on one
    # unit of its own copy of the workload, timed together behind a barrier
    import oracle
    oracle.build()
    r = bench.oracle_host_run(synth.tiny_mlp(), "full_shard", procs=3, warmup=1, steps=2)
    assert r["cores"] == 3 and r["kind"] == "oracle" and r["value"] > 0
    assert "3 processes" in r["sample"] and "2-2 oracle steps" in r["sample"]


def test_unit_workload_steps_like_its_unit_of_the_whole():
    # A host-wide oracle process builds one unit's tensors only: its step must give that
    # unit's shard of the whole workload's step, bit for bit (a FLAT unit's layout and
    # arithmetic do not depend on the other units).
    import numpy as np
    import oracle
    oracle.build()
    w = synth.llama4(blocks=3, hidden=64, ffn=176, N=8)
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = oracle.layout(sh, w.N, w.mode)
    rng = np.random.default_rng(3)
    full = rng.normal(0, 0.02, O["F"]).astype(np.float32)
    grads = [oracle.bf16_rne(rng.normal(0, 1e-3, O["F"]).astype(np.float32)) for _ in range(w.N)]
    S = O["S"]
    master, param = oracle.reshard(sh, w.N, w.mode, full, S, True, True)
    m, v = np.zeros_like(master), np.zeros_like(master)
    oracle.rs_adamw(sh, w.N, w.mode, grads, S, master, m, v, param=param, hp=w.hp, step=1)
    for u in range(O["U"]):
        ws = bench.unit_workload(w, u)
        shu = oracle.Shapes(ws.shapes, ws.unit_ids)
        Ou = oracle.layout(shu, ws.N, ws.mode)
        a, n, f0 = int(O["u_shard_off"][u]), int(O["u_S"][u]), int(O["u_full_off"][u])
        assert Ou["U"] == 1 and Ou["S"] == n and Ou["F"] == w.N * n
        fu = full[f0:f0 + Ou["F"]].copy()
        gu = [g[f0:f0 + Ou["F"]].copy() for g in grads]
        mu, pu_ = oracle.reshard(shu, ws.N, ws.mode, fu, n, True, True)
        mm, vv = np.zeros_like(mu), np.zeros_like(mu)
        oracle.rs_adamw(shu, ws.N, ws.mode, gu, n, mu, mm, vv, param=pu_, hp=w.hp, step=1)
        for r in range(w.N):
            assert np.array_equal(mu[r * n:(r + 1) * n].view(np.uint32),
                                  master[r * S + a:r * S + a + n].view(np.uint32))
            assert np.array_equal(pu_[r * n:(r + 1) * n], param[r * S + a:r * S + a + n])


def test_oracle_host_run_failure_falls_back_to_one_process():
    # a child that fails (here: its workload name is unknown, so it cannot rebuild it) is
    # noticed at once; the bench then times the oracle in its own process and says why
    import time
    import oracle
    oracle.build()
    w = synth.tiny_mlp()
    w.name = "no_such_workload"
    t0 = time.time()
    with pytest.raises(RuntimeError):
        bench.oracle_host_run(w, "full_shard", procs=2, warmup=0, steps=1)
    assert time.time() - t0 < 120
    r = bench.oracle_host_or_one(w, "full_shard", procs=2, warmup=0, steps=2)
    assert r["cores"] == 1 and r["value"] > 0 and "KeyError" in r["host_run_failed"]
