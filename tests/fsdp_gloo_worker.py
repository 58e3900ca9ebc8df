"""Runs torch's own FSDP on gloo CPU ranks and records what it computes.

Used by tests/test_oracle_torch_fsdp.py as an independent pin of the oracle:
  --mode flat  FSDP1 FullyShardedDataParallel, one FlatParameter (use_orig_params=False)
  --mode dim0  FSDP2 fully_shard (per-parameter Shard(0))
Each rank r feeds its own gradient G[t][r] (loss = sum(p * G)), so after backward
FSDP holds the reduce-scattered mean of the G's; torch.optim.AdamW then steps the
local shards.  Saved per rank: local gradient shards, local parameter shapes, and
(rank 0) the initial and final full parameters.
"""
import argparse
import os
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


class Holder(torch.nn.Module):
    def __init__(self, shapes, seed):
        super().__init__()
        g = torch.Generator().manual_seed(seed)
        self.ps = torch.nn.ParameterList(
            [torch.nn.Parameter(torch.randn(*s, generator=g) * 0.02) for s in shapes])

    def forward(self, grads):
        return sum((p * g).sum() for p, g in zip(self.ps, grads))


def grad_for(shapes, seed, t, r):
    g = torch.Generator().manual_seed(seed * 1000 + 100 * t + r)
    return [torch.randn(*s, generator=g) * 1e-3 for s in shapes]


def worker(rank, a):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(a.port)
    dist.init_process_group("gloo", rank=rank, world_size=a.n)
    shapes = [tuple(int(d) for d in s.split("x")) if s != "scalar" else () for s in a.shapes.split(",")]
    model = Holder(shapes, a.seed)
    init = [p.detach().clone() for p in model.ps]
    if a.mode == "dim0":
        from torch.distributed.device_mesh import init_device_mesh
        from torch.distributed.fsdp import fully_shard
        fully_shard(model, mesh=init_device_mesh("cpu", (a.n,)))
        params = list(model.ps)
    else:
        from torch.distributed.fsdp import FullyShardedDataParallel as FSDP
        from torch.distributed.fsdp import ShardingStrategy
        model = FSDP(model, device_id=torch.device("cpu"), sharding_strategy=ShardingStrategy.FULL_SHARD,
                     use_orig_params=False)
        params = [p for p in model.parameters()]
    lr, b1, b2, eps, wd = (float(torch.tensor(x, dtype=torch.float32)) for x in (1e-3, 0.9, 0.999, 1e-8, 0.01))
    opt = torch.optim.AdamW(params, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    out = {"local_shapes": [], "grad_shards": []}
    if a.mode == "dim0":
        out["local_shapes"] = [tuple(p.to_local().shape) for p in params]
    else:
        out["local_shapes"] = [tuple(p.shape) for p in params]
    for t in range(1, a.steps + 1):
        opt.zero_grad(set_to_none=True)
        loss = model(grad_for(shapes, a.seed, t, rank))
        loss.backward()
        if a.mode == "dim0":
            out["grad_shards"].append([p.grad.to_local().detach().clone() for p in params])
        else:
            out["grad_shards"].append([p.grad.detach().clone() for p in params])
        opt.step()
    if a.mode == "dim0":
        final = [p.full_tensor().detach().clone() for p in params]
    else:
        from torch.distributed.fsdp import FullyShardedDataParallel as FSDP
        with FSDP.summon_full_params(model, writeback=False):
            final = [p.detach().clone() for p in model.module.ps]
    out["init"] = init
    out["final"] = final
    out["grads"] = [grad_for(shapes, a.seed, t, rank) for t in range(1, a.steps + 1)]
    torch.save(out, os.path.join(a.out, f"rank{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    p = argparse.ArgumentParser()
    p.add_argument("--mode", choices=["flat", "dim0"], required=True)
    p.add_argument("--n", type=int, required=True)
    p.add_argument("--shapes", required=True)      # e.g. 5x3,7,2x4
    p.add_argument("--steps", type=int, default=3)
    p.add_argument("--seed", type=int, default=1)
    p.add_argument("--port", type=int, default=29561)
    p.add_argument("--out", required=True)
    a = p.parse_args()
    mp.spawn(worker, args=(a,), nprocs=a.n, join=True)
    sys.exit(0)
