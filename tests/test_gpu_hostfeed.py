"""HostFeed (GPU): steps fed from pinned host memory, with the copies overlapped
across steps, end in the same state, bit for bit, as the same steps fed from
device memory, and every step's parameters come back to the host."""
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [synth.tiny_mlp(), synth.llama4(blocks=1, hidden=256, ffn=688, N=8),
                               synth.dim0_n6(vocab=320, hidden=64, ffn=176, N=6)],
                         ids=["tiny_mlp", "llama_small", "dim0_small"])
@pytest.mark.parametrize("strategy", ["full_shard", "shard_grad_op"])
def test_hostfeed_equals_device_fed_steps(w, strategy):
    O = pu.oracle_offsets(w)
    full = synth.full_params(w, O["F"], O["t_full_off"], device="cuda")
    a, b = pu.make_state(w), pu.make_state(w)
    a.init_from_full(full)
    b.init_from_full(full)
    steps = 4
    grads = [synth.grad_replicas(w, O["F"], t, device="cuda") for t in range(1, steps + 1)]
    host = [[g.cpu().pin_memory() for g in gs] for gs in grads]
    outs = [torch.empty(b.param_shards.shape, dtype=b.param_shards.dtype).pin_memory() for _ in range(steps)]
    for t in range(steps):
        a.step(grads[t], w.hp, strategy=strategy)
    feed = fs.HostFeed(b, w.grad_dtype)
    for t in range(steps):
        feed.step(host[t], outs[t], w.hp, strategy)
    feed.finish()
    torch.cuda.synchronize()
    for name in ("master", "exp_avg", "exp_avg_sq"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.param_shards.cpu().view(torch.int16 if w.param_dtype == torch.bfloat16 else torch.int32),
                       outs[-1].view(torch.int16 if w.param_dtype == torch.bfloat16 else torch.int32))
    # every step's result came back: step 1's shards differ from step 4's
    assert not torch.equal(outs[0], outs[-1])


def test_hostfeed_checks_replica_count():
    w = synth.tiny_mlp()
    st = pu.make_state(w)
    feed = fs.HostFeed(st, w.grad_dtype)
    out = torch.empty(st.param_shards.shape, dtype=st.param_shards.dtype).pin_memory()
    with pytest.raises(ValueError):
        feed.step([torch.zeros(st.F).pin_memory()] * (w.N - 1), out, w.hp)
