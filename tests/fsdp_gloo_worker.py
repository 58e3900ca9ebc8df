"""Runs torch's own FSDP / ZeRO on gloo CPU ranks and records what it computes.

Used by the oracle pin tests as an independent reference:
  --mode flat   FSDP1 FullyShardedDataParallel, one FlatParameter (use_orig_params=False)
  --mode dim0   FSDP2 fully_shard (per-parameter Shard(0))
  --mode hsdp   FSDP2 fully_shard on a 2-D mesh (--R replica groups x N shard ranks)
  --mode zero1  ZeroRedundancyOptimizer(AdamW) with the gradients all-reduced (mean)
Options: --clip MAX (clip_grad_norm_ after backward), --accum M (M micro-batches,
the first M-1 without gradient sync: FSDP1 no_sync / FSDP2 set_requires_gradient_sync).
Each rank r feeds its own gradient G[t][m][r] (loss = sum(p * G)).  Saved per rank:
local gradient shards, local parameter shapes, clip norms, ZeRO owners and (rank 0)
the initial and final full parameters.
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


def grad_for(shapes, seed, t, r, micro=0, scale=1e-3):
    g = torch.Generator().manual_seed(seed * 100000 + 1000 * micro + 100 * t + r)
    return [torch.randn(*s, generator=g) * scale for s in shapes]


def hparams():
    return tuple(float(torch.tensor(x, dtype=torch.float32)) for x in (1e-3, 0.9, 0.999, 1e-8, 0.01))


def worker(rank, a):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(a.port)
    world = a.n * a.R
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shapes = [tuple(int(d) for d in s.split("x")) if s != "scalar" else () for s in a.shapes.split(",")]
    model = Holder(shapes, a.seed)
    init = [p.detach().clone() for p in model.ps]
    lr, b1, b2, eps, wd = hparams()
    out = {"local_shapes": [], "grad_shards": [], "norms": [], "owners": None}
    fsdp1 = None
    if a.mode in ("dim0", "hsdp"):
        from torch.distributed.device_mesh import init_device_mesh
        from torch.distributed.fsdp import fully_shard
        mesh = init_device_mesh("cpu", (a.n,)) if a.mode == "dim0" else \
            init_device_mesh("cpu", (a.R, a.n), mesh_dim_names=("replicate", "shard"))
        fully_shard(model, mesh=mesh)
        params = list(model.ps)
        out["local_shapes"] = [tuple(p.to_local().shape) for p in params]
        opt = torch.optim.AdamW(params, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    elif a.mode == "flat":
        from torch.distributed.fsdp import FullyShardedDataParallel as FSDP
        from torch.distributed.fsdp import ShardingStrategy
        fsdp1 = FSDP(model, device_id=torch.device("cpu"), sharding_strategy=ShardingStrategy.FULL_SHARD,
                     use_orig_params=False)
        model = fsdp1
        params = [p for p in model.parameters()]
        out["local_shapes"] = [tuple(p.shape) for p in params]
        opt = torch.optim.AdamW(params, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    else:   # zero1
        from torch.distributed.optim import ZeroRedundancyOptimizer
        params = list(model.ps)
        opt = ZeroRedundancyOptimizer(params, optimizer_class=torch.optim.AdamW, lr=lr, betas=(b1, b2), eps=eps,
                                      weight_decay=wd, foreach=False)
        owned = {id(p) for g in opt.optim.param_groups for p in g["params"]}
        out["owners_mine"] = [id(p) in owned for p in params]

    for t in range(1, a.steps + 1):
        opt.zero_grad(set_to_none=True)
        for mi in range(a.accum):
            last = mi == a.accum - 1
            grads = grad_for(shapes, a.seed, t, rank, micro=mi)
            if a.mode == "flat" and not last:
                with fsdp1.no_sync():
                    model(grads).backward()
            else:
                if a.mode in ("dim0", "hsdp") and a.accum > 1:
                    model.set_requires_gradient_sync(last)
                model(grads).backward()
        if a.mode == "zero1":
            for p in params:
                dist.all_reduce(p.grad, op=dist.ReduceOp.SUM)
                p.grad /= world
        if a.clip > 0:
            if fsdp1 is not None:
                n = fsdp1.clip_grad_norm_(a.clip)
            else:
                n = torch.nn.utils.clip_grad_norm_(params, a.clip)
            out["norms"].append(float(n.full_tensor() if hasattr(n, "full_tensor") else n))
        if a.mode in ("dim0", "hsdp"):
            out["grad_shards"].append([p.grad.to_local().detach().clone() for p in params])
        else:
            out["grad_shards"].append([p.grad.detach().clone() for p in params])
        opt.step()
    if a.mode in ("dim0", "hsdp"):
        final = [p.full_tensor().detach().clone() for p in params]
    elif a.mode == "flat":
        from torch.distributed.fsdp import FullyShardedDataParallel as FSDP
        with FSDP.summon_full_params(model, writeback=False):
            final = [p.detach().clone() for p in model.module.ps]
    else:
        final = [p.detach().clone() for p in params]
    out["init"] = init
    out["final"] = final
    out["grads"] = [[grad_for(shapes, a.seed, t, rank, micro=mi) for mi in range(a.accum)]
                    for t in range(1, a.steps + 1)]
    torch.save(out, os.path.join(a.out, f"rank{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    p = argparse.ArgumentParser()
    p.add_argument("--mode", choices=["flat", "dim0", "hsdp", "zero1"], required=True)
    p.add_argument("--n", type=int, required=True)          # shard ranks (world size except HSDP)
    p.add_argument("--R", type=int, default=1)              # HSDP replica groups
    p.add_argument("--shapes", required=True)               # e.g. 5x3,7,2x4
    p.add_argument("--steps", type=int, default=3)
    p.add_argument("--seed", type=int, default=1)
    p.add_argument("--clip", type=float, default=0.0)
    p.add_argument("--accum", type=int, default=1)
    p.add_argument("--port", type=int, default=29561)
    p.add_argument("--out", required=True)
    a = p.parse_args()
    mp.spawn(worker, args=(a,), nprocs=a.n * a.R, join=True)
    sys.exit(0)
