"""CUDA path vs oracle on the five workloads (GPU).

Small layouts, and the one-unit sweep up to 2^26+1 parameters (bf16 and fp32
parameters), are compared element by element over the whole state after every
step; the full-size 4-block Llama (809.5M parameters, N=8) and the FSDP2 dim-0
group (243M, N=6) are run at full size and compared on sampled positions that the
oracle tracks across the steps: every element of each tile touching a unit, tensor,
rank or padding boundary, every element of a seeded 1 % of all tiles, and random
positions; every padding element of every state array is checked for +0.  Most runs also request the reduced-gradient output; the last
tests run the configurations bench.py times (no such output, so the kernel
instance the bench launches) at full size.
"""
import pytest
import torch

from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


def test_tiny_mlp_flat_fp32(oracle_lib):
    _, ulps = pu.run_full_parity(synth.tiny_mlp(), strategy="full_shard")
    print("tiny_mlp ulps per step", ulps)


def test_tiny_mlp_dim0_bf16(oracle_lib):
    w = synth.tiny_mlp(mode=synth.DIM0)
    w.param_dtype = torch.bfloat16
    w.grad_dtype = torch.bfloat16
    pu.run_full_parity(w, strategy="shard_grad_op")


def test_mlp128m_10_steps(oracle_lib):
    _, ulps = pu.run_full_parity(synth.mlp128m(), check_unshard=True)
    assert len(ulps) == 10
    print("mlp128m ulps per step", ulps)


def test_llama_block_reduced_full_compare(oracle_lib):
    # one Llama-style block with small hidden sizes, every element compared
    w = synth.llama4(blocks=2, hidden=256, ffn=688, N=8)
    pu.run_full_parity(w)


def test_llama4_full_size_sampled(oracle_lib):
    _, ulps = pu.run_sampled_parity(synth.llama4())
    print("llama4 ulps per step", ulps)


def test_dim0_reduced_full_compare(oracle_lib):
    w = synth.dim0_n6(vocab=320, hidden=64, ffn=176, N=6)
    pu.run_full_parity(w)


def test_dim0_n6_full_size_sampled(oracle_lib):
    _, ulps = pu.run_sampled_parity(synth.dim0_n6())
    print("dim0_n6 ulps per step", ulps)


@pytest.mark.parametrize("N", [2, 4, 8, 16, 32])
@pytest.mark.parametrize("P", [1 << 20, (1 << 20) + 1])
def test_sweep_small_full_compare(oracle_lib, P, N):
    w = synth.sweep(P, N)
    pu.run_full_parity(w, strategy="full_shard" if P % 2 else "shard_grad_op")


@pytest.mark.parametrize("N", [2, 8, 32])
@pytest.mark.parametrize("P", [(1 << 22) + 1, (1 << 24) + 1, (1 << 26) + 1])
def test_sweep_full_compare_to_2_26(oracle_lib, P, N):
    # the sweep compared over the whole state up to 2^26+1 parameters (odd sizes:
    # padding in the last rank, views off their 16-byte congruence)
    pu.run_full_parity(synth.sweep(P, N), strategy="full_shard")


@pytest.mark.parametrize("N", [2, 4, 8, 16, 32])
@pytest.mark.parametrize("P", [(1 << 20) + 1, (1 << 24) + 1])
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32], ids=["bf16grad", "f32grad"])
def test_sweep_fp32_params_full_compare(oracle_lib, P, N, grad_dtype):
    # fp32 parameters (the master is the parameter, no bf16 copy); fp32 gradients
    # beyond N = 8 and bf16 ones beyond N = 16 are staged in replica groups
    w = synth.sweep(P, N, param_dtype=torch.float32, grad_dtype=grad_dtype)
    pu.run_full_parity(w, strategy="full_shard" if N % 4 else "shard_grad_op")


@pytest.mark.parametrize("P,N", [((1 << 22) + 1, 64), ((1 << 22) + 1, 1)])
def test_rank_count_extremes_full_compare(oracle_lib, P, N):
    # the largest N the layout takes (64: three replica groups of 22 per tile) and a single
    # rank, each large enough for the CTAs to claim their tiles, over the whole state
    pu.run_full_parity(synth.sweep(P, N), strategy="full_shard")


@pytest.mark.parametrize("P,N", [((1 << 26) + 1, 8), ((1 << 29) + 1, 32), (1 << 29, 2)])
def test_sweep_large_sampled(oracle_lib, P, N):
    pu.run_sampled_parity(synth.sweep(P, N), n_random=100_000)


# ---------------------------------------------------------------------------
# The configurations bench.py times: no reduced-gradient output (the kernel instance
# without it), the default kernel choice, FULL_SHARD.
def test_mlp128m_bench_config(oracle_lib):
    w = synth.mlp128m()
    _, ulps = pu.run_full_parity(w, steps=3, with_grad_out=False)
    print("mlp128m (bench configuration) ulps per step", ulps)


@pytest.mark.parametrize("name", ["llama4", "dim0_n6", "sweep_P268435457_N8", "sweep_P67108865_N32"])
def test_bench_config_full_size_sampled(oracle_lib, name):
    w = synth.workload(name)
    _, ulps = pu.run_sampled_parity(w, steps=min(w.steps, 2), n_random=100_000, with_grad_out=False)
    print(name, "(bench configuration) ulps per step", ulps)
