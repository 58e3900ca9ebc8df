"""Pins of the oracle's flatten/pad/shard layout (CPU).

Pinned against (a) the worked examples the pages print (tests/golden/page_examples.txt),
(b) a brute-force construction written independently of the oracle: element ids are
laid out, the FLAT unit is padded to the smallest multiple of N and split into N
equal chunks; a DIM0 tensor is split with torch.chunk along dim 0 (how FSDP2's
Shard(0) places rows), each rank's slot padded to the first chunk's row count.
"""
import itertools
import os
import random

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_examples.txt")


def golden_rows(kind):
    rows = []
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = [p.strip() for p in line.split("|")]
        if parts[0] == kind:
            rows.append(parts)
    assert rows, kind
    return rows


def parse_shapes(s):
    return [tuple(int(d) for d in piece.split("x")) for piece in s.split("=")[1].split(";")]


def test_flatparameter_worked_example(oracle_lib):
    # [768,768] + [768] + [768] flattened and concatenated -> 591,360 elements.
    for _, inp, exp, _src in golden_rows("flat_numel"):
        sh = oracle.Shapes(parse_shapes(inp))
        for N in (1, 2, 4, 8):
            L = oracle.layout(sh, N, oracle.FLAT)
            assert L["P"] == int(exp)
            assert L["u_numel"][0] == int(exp)
    for _, inp, exp, _src in golden_rows("flat_piece"):
        sh = oracle.Shapes(parse_shapes(inp))
        assert oracle.layout(sh, 1, oracle.FLAT)["P"] == int(exp)


def test_dim0_local_shapes(oracle_lib):
    # [8,8] on 2 ranks -> local [4,8]; [4096,4096] on 8 ranks -> [512,4096].
    for _, inp, exp, _src in golden_rows("dim0_local"):
        shape_s, n_s = inp.split()
        shape = tuple(int(d) for d in shape_s.split("=")[1].split("x"))
        N = int(n_s.split("=")[1])
        rows, inner = (int(x) for x in exp.split("x"))
        L = oracle.layout(oracle.Shapes([shape]), N, oracle.DIM0)
        assert L["t_rows"][0] == rows
        assert L["t_slot"][0] == rows * inner
        assert L["S"] == rows * inner and L["N"] * L["S"] == L["P"]   # divisible: no padding


def test_padding_formula_example(oracle_lib):
    for _, inp, exp, _src in golden_rows("pad_formula"):
        P = int(inp.split()[0].split("=")[1])
        N = int(inp.split()[1].split("=")[1])
        L = oracle.layout(oracle.Shapes([(P,)]), N, oracle.FLAT)
        assert L["N"] * L["S"] == int(exp) == L["F"]          # padded flat numel
        assert L["F"] == L["S"] * N                            # padded numel == shard numel * N


# ---------------------------------------------------------------------------
# brute force
# ---------------------------------------------------------------------------
def brute_layout(shapes, units, N, mode):
    """{(rank, j): full index or -1}, built without the oracle's formulas."""
    owner = {}
    numels = [int(np.prod(s)) if len(s) else 1 for s in shapes]
    if mode == oracle.FLAT:
        full_pos = 0
        shard_base = 0
        for u in sorted(set(units)):
            ids = []
            for t, (s, uu) in enumerate(zip(shapes, units)):
                if uu == u:
                    ids.extend(range(full_pos + len(ids), full_pos + len(ids) + numels[t]))
            P_u = len(ids)
            padded = list(ids)
            while len(padded) % N:          # smallest multiple of N at or above P_u
                padded.append(-1)
            if not padded:
                padded = []
            chunk = len(padded) // N
            for r in range(N):
                piece = padded[r * chunk:(r + 1) * chunk]
                for k, fid in enumerate(piece):
                    owner[(r, shard_base + k)] = fid
            shard_base += chunk
            full_pos += len(padded)
        return owner, shard_base, full_pos
    # DIM0
    full_pos = 0
    shard_base = 0
    for t, s in enumerate(shapes):
        shape = tuple(s) if len(s) else (1,)
        ids = torch.arange(full_pos, full_pos + numels[t]).reshape(shape)
        chunks = list(torch.chunk(ids, N, dim=0)) if shape[0] > 0 else []
        rows = chunks[0].shape[0] if chunks else 0
        inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
        for r in range(N):
            mine = chunks[r].reshape(-1).tolist() if r < len(chunks) else []
            for k in range(rows * inner):
                owner[(r, shard_base + k)] = mine[k] if k < len(mine) else -1
        shard_base += rows * inner
        full_pos += numels[t]
    return owner, shard_base, full_pos


def random_cases(n, seed=7):
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        T = rng.randint(1, 3)
        shapes = []
        for _t in range(T):
            nd = rng.randint(0, 3)
            shapes.append(tuple(rng.randint(0, 5) for _ in range(nd)))
        units = [0]
        for _t in range(1, T):
            units.append(units[-1] + rng.randint(0, 1))
        cases.append((shapes, units, rng.randint(1, 9), rng.choice([oracle.FLAT, oracle.DIM0])))
    return cases


EDGE_CASES = [
    ([(5, 3), (4,)], [0, 0], 3, oracle.FLAT),        # P = 19, N = 3: one padding element
    ([(5, 3)], [0], 4, oracle.DIM0),                 # 5 rows on 4 ranks: 2,2,1,0
    ([(1, 7)], [0], 5, oracle.DIM0),                 # d0 < N: four ranks own nothing
    ([(0, 4), (3,)], [0, 1], 2, oracle.DIM0),        # empty tensor
    ([(), (2,)], [0, 0], 2, oracle.FLAT),            # scalar
    ([(7,)], [0], 1, oracle.FLAT),                   # N = 1: identity
    ([(2, 2), (3,), (1,)], [0, 1, 2], 4, oracle.FLAT),   # every unit padded
]


@pytest.mark.parametrize("case", EDGE_CASES + random_cases(250))
def test_layout_brute_force(oracle_lib, case):
    shapes, units, N, mode = case
    sh = oracle.Shapes(shapes, units)
    L = oracle.layout(sh, N, mode)
    owner, S_bf, F_bf = brute_layout(shapes, units, N, mode)
    assert L["S"] == S_bf
    assert L["F"] == F_bf
    numels = [int(np.prod(s)) if len(s) else 1 for s in shapes]
    assert L["P"] == sum(numels)
    seen = {}
    for r in range(N):
        j = np.arange(L["S"], dtype=np.int64)
        got = oracle.full_index(sh, N, mode, r, j)
        exp = np.array([owner[(r, int(x))] for x in j], dtype=np.int64)
        assert np.array_equal(got, exp), (r, got, exp)
        for x in got:
            if x >= 0:
                assert x not in seen
                seen[int(x)] = r
    # every logical element is owned exactly once; the padding count is N*S - P
    assert len(seen) == L["P"]
    pad = sum(int((oracle.full_index(sh, N, mode, r, np.arange(L["S"])) < 0).sum()) for r in range(N))
    assert pad == N * L["S"] - L["P"]


def test_flat_rank_views_may_be_empty(oracle_lib):
    # A rank's view of an original parameter can be a 1-D piece or empty.
    sh = oracle.Shapes([(2,), (10,)], [0, 0])
    N = 4                               # S = 3: rank 0 holds [a0 a1 b0], ranks 1..3 only b
    L = oracle.layout(sh, N, oracle.FLAT)
    assert L["S"] == 3
    idx = [oracle.full_index(sh, N, oracle.FLAT, r, np.arange(3)) for r in range(N)]
    holders_of_a = [r for r in range(N) if ((idx[r] >= 0) & (idx[r] < 2)).any()]
    assert holders_of_a == [0]


def test_llama_and_dim0_config_layouts(oracle_lib):
    # Survey of the workloads: 4 Llama blocks, one FLAT unit each, N = 8 ...
    from fsdp_sharded_state_gb300 import synth
    w = synth.llama4()
    L = oracle.layout(oracle.Shapes(w.shapes, w.unit_ids), w.N, w.mode)
    assert L["P"] == 809_533_440
    assert list(L["u_S"]) == [25_297_920] * 4 and L["N"] * L["S"] == L["P"]
    # ... and FSDP2 dim-0 sharding with N = 6 (not dividing 32000, 4096, 11008).
    w = synth.dim0_n6()
    L = oracle.layout(oracle.Shapes(w.shapes, w.unit_ids), w.N, w.mode)
    assert list(L["t_rows"]) == [5334, 683, 683, 683, 683, 1835, 683]
    assert L["S"] == 40_555_179 and L["P"] == 243_273_728 and 6 * L["S"] - L["P"] == 57_346
    Lf = oracle.layout(oracle.Shapes(w.shapes, w.unit_ids), w.N, oracle.FLAT)
    assert Lf["S"] == 40_545_622 and 6 * Lf["S"] - Lf["P"] == 4
