"""Pins of the oracle's per-rank model-state and collective-payload accounting (CPU).

Against the measured table of "NCCL ZeRO/FSDP state sharding" (section 实测状态因子,
128 MiB fp32 on 4 ranks), its steady-memory table (section Steady 显存与 Peak 显存),
its per-rank formulas (section Canonical ZeRO 状态公式), and the memory arithmetic of
"第18章 FSDP：ZeRO 风格的参数分片" §18.1/§18.32 and the torchtitan FSDP2 article §2.3.
"""
import os

import numpy as np

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


# ---------------------------------------------------------------------------
# Collective payload of one step (logical inputs, ring bus elements per rank)
PAYLOAD_STRATEGY = {"zero0_ddp": oracle.NO_SHARD, "zero1_zro": oracle.ZERO1_OPT,
                    "fsdp_shard_grad_op": oracle.SHARD_GRAD_OP, "fsdp_full_shard": oracle.FULL_SHARD}


@pytest.mark.parametrize("shapes,units,N", [(P2_SHAPES, P2_UNITS, 4), ([(37, 5), (3,), (11, 13)], [0, 1, 1], 3),
                                            ([(1000, 7)], [0], 8)])
def test_logical_payload_table(oracle_lib, shapes, units, N):
    # the page's table, row by row, in units of P, on the page's layout and on others
    sh = oracle.Shapes(shapes, units)
    P = oracle.layout(sh, N, oracle.FLAT)["P"]
    table = [r for r in rows("logical_payload_per_step.txt") if r[0] in PAYLOAD_STRATEGY]
    assert len(table) == 4
    for name, *units_of_p in table:
        elems, _ = oracle.collective_payload(sh, N, oracle.FLAT, PAYLOAD_STRATEGY[name])
        assert elems == [int(x) * P for x in units_of_p], name


def ring_sends(op, N, P):
    """Elements each rank sends in a ring all-reduce / all-gather / reduce-scatter of a
    P-element buffer (P divisible by N), simulated chunk by chunk; the result is checked."""
    rng = np.random.default_rng(N * 1000 + P)
    c = P // N
    data = [rng.integers(-1000, 1000, P).astype(np.int64) for _ in range(N)]
    sent = [0] * N
    if op in ("allreduce", "reducescatter"):
        buf = [d.copy() for d in data]
        for step in range(N - 1):                 # rank r passes chunk (r - step) mod N to r+1
            msgs = []
            for r in range(N):
                k = (r - step) % N
                msgs.append((r, k, buf[r][k * c:(k + 1) * c].copy()))
                sent[r] += c
            for r, k, x in msgs:
                buf[(r + 1) % N][k * c:(k + 1) * c] += x
        total = sum(data)
        for r in range(N):                        # rank r now owns chunk (r + 1) mod N, fully reduced
            k = (r + 1) % N
            assert np.array_equal(buf[r][k * c:(k + 1) * c], total[k * c:(k + 1) * c])
        if op == "reducescatter":
            return sent
        own = [(r + 1) % N for r in range(N)]
        data = buf
    else:
        own = list(range(N))                      # all-gather: rank r starts with its chunk r
        full = np.concatenate([data[r][r * c:(r + 1) * c] for r in range(N)])
        data = [d.copy() for d in data]
        total = full
    have = [{own[r]} for r in range(N)]
    for step in range(N - 1):                     # pass the newest chunk on around the ring
        msgs = []
        for r in range(N):
            k = (own[r] - step) % N
            msgs.append((r, k, data[r][k * c:(k + 1) * c].copy()))
            sent[r] += c
        for r, k, x in msgs:
            data[(r + 1) % N][k * c:(k + 1) * c] = x
            have[(r + 1) % N].add(k)
    for r in range(N):
        assert len(have[r]) == N and np.array_equal(data[r], total)
    return sent


@pytest.mark.parametrize("N", [2, 3, 4, 8])
def test_bus_elements_equal_simulated_ring_traffic(oracle_lib, N):
    # brute force: the per-rank sends of simulated ring collectives (which must also
    # produce the right result) against the oracle's bus elements, per strategy
    P = 24 * N
    sh = oracle.Shapes([(P,)], [0])
    ar = ring_sends("allreduce", N, P)
    ag = ring_sends("allgather", N, P)
    rs = ring_sends("reducescatter", N, P)
    assert len(set(ar)) == len(set(ag)) == len(set(rs)) == 1      # every rank sends the same
    expect = {oracle.NO_SHARD: ar[0], oracle.SHARD_GRAD_OP: ag[0] + rs[0], oracle.FULL_SHARD: 2 * ag[0] + rs[0],
              oracle.ZERO1_OPT: ar[0] + ag[0]}                    # broadcast: each rank receives what others own
    for strategy, sends in expect.items():
        _, bus = oracle.collective_payload(sh, N, oracle.FLAT, strategy)
        assert bus == pytest.approx(sends, rel=0, abs=1e-9), strategy
    for R in (1, 2, 3):                           # HSDP: FULL_SHARD in the group, all-reduce of the shard over R
        _, bus = oracle.collective_payload(sh, N, oracle.FLAT, oracle.HYBRID_SHARD, R)
        S = P // N
        across = ring_sends("allreduce", R, S)[0] if R > 1 else 0      # the S-element shard over R groups
        assert bus == pytest.approx(2 * ag[0] + rs[0] + across, abs=1e-9)


def test_communication_volume_in_psi(oracle_lib):
    # "第18章 FSDP" §18.2: DDP about 2 Psi, ZeRO-2 still 2 Psi, ZeRO-3 about 3 Psi, 1.5 x DDP;
    # the ratios hold for every N, the Psi multiples in the limit of many ranks
    vol = {r[0]: float(r[1]) for r in rows("logical_payload_per_step.txt") if r[0].startswith("volume_")}
    sh = oracle.Shapes([(4096, 64)], [0])
    for N in (2, 4, 8, 64, 1024):
        P = oracle.layout(sh, N, oracle.FLAT)["P"]
        ddp = oracle.collective_payload(sh, N, oracle.FLAT, oracle.NO_SHARD)[1]
        sgo = oracle.collective_payload(sh, N, oracle.FLAT, oracle.SHARD_GRAD_OP)[1]
        full = oracle.collective_payload(sh, N, oracle.FLAT, oracle.FULL_SHARD)[1]
        assert ddp == pytest.approx(2 * (N - 1) / N * P)             # the all-reduce bus factor
        assert sgo / ddp == pytest.approx(vol["volume_zero2"] / vol["volume_ddp"])
        assert full / ddp == pytest.approx(vol["volume_zero3"] / vol["volume_ddp"])
    assert ddp / P == pytest.approx(vol["volume_ddp"], rel=2e-3)       # N = 1024
    assert full / P == pytest.approx(vol["volume_zero3"], rel=2e-3)


def test_payload_special_cases(oracle_lib):
    sh = oracle.Shapes([(37, 5), (3,), (11, 13)], [0, 1, 1])
    for s in (oracle.NO_SHARD, oracle.ZERO1_OPT, oracle.SHARD_GRAD_OP, oracle.FULL_SHARD):
        assert oracle.collective_payload(sh, 1, oracle.FLAT, s)[1] == 0.0          # one rank moves nothing
    for N in (2, 5):
        full = oracle.collective_payload(sh, N, oracle.FLAT, oracle.FULL_SHARD)
        h1 = oracle.collective_payload(sh, N, oracle.FLAT, oracle.HYBRID_SHARD, 1)
        assert h1[1] == pytest.approx(full[1]) and h1[0][1:] == full[0][1:]          # one group = FULL_SHARD
    P = oracle.layout(sh, 1, oracle.FLAT)["P"]
    for R in (2, 3, 7):                                                             # one rank per group = DDP over R
        assert oracle.collective_payload(sh, 1, oracle.FLAT, oracle.HYBRID_SHARD, R)[1] == pytest.approx(
            2 * (R - 1) / R * P)
    with pytest.raises(ValueError):
        oracle.collective_payload(sh, 2, oracle.FLAT, oracle.FULL_SHARD, 2)         # groups only with HSDP
    with pytest.raises(ValueError):
        oracle.collective_payload(sh, 2, oracle.FLAT, 5)
