"""Pipeline launches that claim their work units from a counter (GPU).

A launch with enough units per CTA takes a counter pair from the device's ring and its
CTAs claim units from it; a slot is reused only after the launch that used it has
completed, and the kernel leaves the pair at zero.  The checks count: the accumulation
adds an exact integer per call, so a unit skipped or done twice changes the count.
  - 1,200 calls queued without a synchronisation (more than the ring's 1,024 slots, so
    that calls find no free slot and split their units statically while the GPU catches
    up);
  - calls on two streams at once, each with its own accumulators;
  - the fused step with claims against its static form (CUDA graph capture) bit for bit
    lives in tests/test_gpu_graph.py, and against the no-allocation entry point in
    tests/test_zz_no_alloc.py.
"""
import pytest
import torch

import fsdp_sharded_state_gb300 as fs

pytestmark = pytest.mark.gpu

# 1 FLAT unit of 2^23 elements: 4,096 tiles of the full layout, well above the 8 units
# per CTA from which a launch claims
SHAPES, UNITS, N = [(1 << 23,)], [0], 2


def _layout():
    L = fs.Layout(SHAPES, UNITS, N, fs.FSDP_FLAT)
    L.prepare()
    return L


def test_queued_calls_count_exactly():
    L = _layout()
    F = L.info["full_numel"]
    acc = [torch.zeros(F, dtype=torch.float32, device="cuda") for _ in range(N)]
    ones = [torch.ones(F, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    for k in range(1200):
        fs.fsdp_accumulate_grads(L, 0, L.n_units, acc, ones, first=(k == 0))
    torch.cuda.synchronize()
    fs.fsdp_check_status()
    for q in range(N):
        assert torch.equal(acc[q], torch.full_like(acc[q], 1200.0))


def test_two_streams_count_exactly():
    L = _layout()
    F = L.info["full_numel"]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    accs = [[torch.zeros(F, dtype=torch.float32, device="cuda") for _ in range(N)] for _ in streams]
    ones = [torch.ones(F, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    torch.cuda.synchronize()
    for k in range(40):
        for s, acc in zip(streams, accs):
            with torch.cuda.stream(s):
                fs.fsdp_accumulate_grads(L, 0, L.n_units, acc, ones, first=False, stream=s)
    torch.cuda.synchronize()
    fs.fsdp_check_status()
    for acc in accs:
        for q in range(N):
            assert torch.equal(acc[q], torch.full_like(acc[q], 40.0))
