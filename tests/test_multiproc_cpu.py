"""Multi-process host logic on the CPU (gloo, world size 2):

* the cross-shard exchange the vocabulary-parallel entry points rely on: each
  rank holds a vocabulary shard, computes its per-row LSE and target logit
  (by definition, in fp64), and the all-reduces (MAX, then SUM of
  exp(lse_s - max), SUM of target logits) reproduce the unsharded oracle's
  LSE and loss;
* the benchmark's whole-job throughput: tokens of all ranks over the slowest
  rank's time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
        import synthetic_inputs as si
        from oracle import flce_oracle as O
        import bench

        n, v = 64, 1000
        logits, t = si.make_ce_logits(n, v, 12, std=2.0, dtype="fp32", ignore_frac=0.1)
        cuts = [0, 430, v]
        a, b = cuts[rank], cuts[rank + 1]
        z = logits[:, a:b].astype(np.float64)
        m = z.max(axis=1)
        lse_s = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        tl = t - a
        here = (t != -100) & (tl >= 0) & (tl < b - a)
        zt_s = np.zeros(n)
        zt_s[here] = z[here, tl[here]]
        mx = torch.tensor(lse_s)
        dist.all_reduce(mx, op=dist.ReduceOp.MAX)
        se = torch.tensor(np.exp(lse_s - mx.numpy()))
        dist.all_reduce(se, op=dist.ReduceOp.SUM)
        zt = torch.tensor(zt_s)
        dist.all_reduce(zt, op=dist.ReduceOp.SUM)
        lse = mx.numpy() + np.log(se.numpy())
        ref = O.ce_reference(logits, t, reduction="mean")
        valid = t != -100
        loss = np.where(valid, lse - zt.numpy(), 0.0).sum() / valid.sum()

        def all_reduce_max(x):
            tt = torch.tensor([x], dtype=torch.float64)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            return float(tt.item())

        value, ms = bench.aggregate_tokens_per_s(10.0 + 5.0 * rank, 1000, world, all_reduce_max)
        out[rank] = (float(np.abs(lse - ref["lse"]).max()), abs(loss - ref["loss"]), value, ms)
    finally:
        dist.destroy_process_group()


def test_vocab_shard_exchange_and_throughput_aggregation():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        lse_err, loss_err, value, ms = out[r]
        assert lse_err < 1e-12 and loss_err < 1e-12
        assert ms == 15.0 and abs(value - 2000 / 0.015) < 1e-6
