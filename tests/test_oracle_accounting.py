"""Pins of the oracle's per-rank model-state accounting (CPU).

Against the measured table of "NCCL ZeRO/FSDP state sharding" (section 实测状态因子,
128 MiB fp32 on 4 ranks), its steady-memory table (section Steady 显存与 Peak 显存),
its per-rank formulas (section Canonical ZeRO 状态公式), and the memory arithmetic of
"第18章 FSDP：ZeRO 风格的参数分片" §18.1/§18.32 and the torchtitan FSDP2 article §2.3.
"""
import os

import pytest

import oracle

G = os.path.join(os.path.dirname(__file__), "golden")
MiB = 1 << 20


def rows(name):
    out = []
    for line in open(os.path.join(G, name), encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append([p.strip() for p in line.split("|")])
    return out


P2_SHAPES = [(2048, 2048)] * 8      # 8 Linear weights, one wrap unit each
P2_UNITS = list(range(8))


def per_rank(stage, rank=0, N=4, step_bytes=0, physical=True):
    sh = oracle.Shapes(P2_SHAPES, P2_UNITS)
    return oracle.state_bytes(sh, N, oracle.FLAT, stage, rank, physical, 4, 4, 8, step_bytes)


def test_measured_state_factors_128MiB_N4(oracle_lib):
    P = 8 * 2048 * 2048 * 4
    assert P == 128 * MiB
    for name, stage, pf, gf, of, maxrank, _steady in rows("state_factors_128MiB_N4.txt"):
        stage = int(stage)
        totals = [0, 0, 0]
        maxes = [0, 0, 0]
        for r in range(4):
            b = per_rank(stage, r)
            for k in range(3):
                totals[k] += b[k]
                maxes[k] = max(maxes[k], b[k])
        assert [t / P for t in totals] == [float(pf), float(gf), float(of)], name
        assert [m // MiB for m in maxes] == [int(x) for x in maxrank.split("/")], name


def test_step_scalar_adds_about_1e6_to_optimizer_factor(oracle_lib):
    # one fp32 step scalar per parameter tensor on every rank
    P = 128 * MiB
    tot = sum(per_rank(3, r, step_bytes=4)[2] for r in range(4))
    extra = tot / P - 2.0
    assert 5e-7 < extra < 2e-6


def test_steady_memory_differences(oracle_lib):
    # steady allocated = model state + a constant; the differences between rows are
    # the state differences: 528.25 - 336.25 = 192 MiB = 4P - (2P + 2P/N), and
    # 336.25 - 144.25 = 192 MiB = (2P + 2P/N) - 4P/N.
    steady = {r[0]: float(r[6]) for r in rows("state_factors_128MiB_N4.txt")}
    state = {name: sum(per_rank(int(stage))) / MiB for name, stage, *_ in rows("state_factors_128MiB_N4.txt")}
    assert steady["zero0_ddp"] - steady["zero1_zro"] == state["zero0_ddp"] - state["zero1_zro"] == 192
    assert steady["zero1_zro"] - steady["zero3_pre"] == state["zero1_zro"] - state["zero3_pre"] == 192
    # and the constant is the same for all rows
    offsets = {steady[k] - state[k] for k in steady}
    assert len(offsets) == 1


@pytest.mark.parametrize("N", [2, 3, 4, 8, 16])
def test_canonical_formulas(oracle_lib, N):
    # 4P, 2P + 2P/N, P + 3P/N, 4P/N per rank (bytes, fp32 Adam, P divisible by N)
    P = 4 * 2048 * 2048 * N          # logical fp32 bytes, divisible by 4N
    sh = oracle.Shapes([(P // 4,)])
    tot = [sum(oracle.state_bytes(sh, N, oracle.FLAT, s, 0, True, 4, 4, 8)) for s in range(4)]
    assert tot == [4 * P, 2 * P + 2 * P // N, P + 3 * P // N, 4 * P // N]


def test_logical_vs_physical_with_padding(oracle_lib):
    sh = oracle.Shapes([(5, 3), (4,)])         # P = 19 elements, N = 3, S = 7
    phys = [oracle.state_bytes(sh, 3, oracle.FLAT, 3, r, True, 1, 1, 1) for r in range(3)]
    logi = [oracle.state_bytes(sh, 3, oracle.FLAT, 3, r, False, 1, 1, 1) for r in range(3)]
    assert [p[0] for p in phys] == [7, 7, 7]
    assert [l[0] for l in logi] == [7, 7, 5]
    assert sum(l[0] for l in logi) == 19


@pytest.mark.parametrize("row", rows("memory_closed_forms.txt"), ids=lambda r: r[0])
def test_memory_closed_forms(oracle_lib, row):
    name, numel, N, bpe, expect, _src = row
    numel, N = int(float(numel)), int(N)
    pb, gb, ob = (int(x) for x in bpe.split("/"))
    sh = oracle.Shapes([(numel,)])
    stage = 0 if N == 1 else 3
    b = oracle.state_bytes(sh, N, oracle.FLAT, stage, 0, True, pb, gb, ob)
    exp = [float(x) for x in expect.split("/")]
    if len(exp) == 3:
        assert [x / 1e9 for x in b] == pytest.approx(exp, rel=1e-12)
    else:
        assert sum(b) / 1e9 == pytest.approx(exp[0], rel=1e-12)
