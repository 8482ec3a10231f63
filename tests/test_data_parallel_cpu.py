"""Multi-rank host logic on CPU: world_size-2 gloo process groups.

The shard + exchange of a data-parallel step (each rank the unscaled sums of
its tokens, then one all-reduce and a 1/n_valid rescale) must equal the
unsplit mean; the replica timing takes the max over ranks.  The per-rank
compute here is the fp64 oracle (no GPU is involved)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from linear_cross_entropy_ce_gb300 import dist as fdist


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    from linear_cross_entropy_ce_gb300 import workloads as wl
    from oracle import flce_oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = wl.random_problem(203, 24, 77, seed=5, ignore_frac=0.3)
        sl = fdist.shard_rows(203, rank, world)
        o = flce_oracle(p["hidden"][sl], p["weight"], p["targets"][sl], reduction="sum")
        gw = torch.from_numpy(o["grad_weight"].copy())
        loss, n, scale = fdist.exchange_sums(o["loss"], o["n_valid"], gw)
        gh = o["grad_hidden"] * scale
        t = fdist.max_over_ranks(10.0 + rank)
        q.put((rank, loss, n, gw.numpy(), gh, sl.start, sl.stop, t))
    finally:
        dist.destroy_process_group()


def _vp_worker(rank, world, port, q):
    import torch.distributed as dist
    from linear_cross_entropy_ce_gb300 import workloads as wl
    from oracle import decode_bf16
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = wl.random_problem(40, 16, 101, seed=6, ignore_frac=0.2)
        bounds = [0, 37, 101]                      # uneven vocabulary shards
        a, b = bounds[rank], bounds[rank + 1]
        X = decode_bf16(p["hidden"])
        W = decode_bf16(p["weight"])[a:b]
        t = p["targets"].astype(np.int64)
        z = X @ W.T                                # this rank's logits (fp64)
        m = torch.from_numpy(z.max(axis=1).copy())
        d = torch.from_numpy(np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1))
        inside = (t >= a) & (t < b)
        zt = torch.from_numpy(np.where(inside, z[np.arange(40), np.clip(t - a, 0, b - a - 1)], 0.0))

        def rescale(lm, gm, s):
            s.mul_(torch.exp(lm - gm))
        fdist.vocab_merge(m, d, zt, rescale)
        q.put((rank, (m + torch.log(d)).numpy(), zt.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_rank_vocab_merge_matches_oracle():
    from linear_cross_entropy_ce_gb300 import workloads as wl
    from oracle import flce_oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_vp_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=180) for _ in range(2)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    p = wl.random_problem(40, 16, 101, seed=6, ignore_frac=0.2)
    full = flce_oracle(p["hidden"], p["weight"], p["targets"])
    valid = p["targets"] != -100
    for rank, lse, zt in res:
        np.testing.assert_allclose(lse[valid], full["lse"][valid], rtol=1e-13)
        np.testing.assert_allclose((lse - zt)[valid], full["row_loss"][valid], rtol=1e-11, atol=1e-13)


def test_shard_rows_partition():
    for N in (1, 7, 203, 4096):
        for world in (1, 2, 3, 8):
            parts = [fdist.shard_rows(N, r, world) for r in range(world)]
            assert parts[0].start == 0 and parts[-1].stop == N
            for a, b in zip(parts, parts[1:]):
                assert a.stop == b.start
            sizes = [s.stop - s.start for s in parts]
            assert max(sizes) - min(sizes) <= 1
    assert fdist.replica_seed(3, 0) == 3 and fdist.replica_seed(3, 2) == 2003
    assert fdist.max_over_ranks(1.5) == 1.5


def test_two_rank_exchange_matches_unsplit():
    from linear_cross_entropy_ce_gb300 import workloads as wl
    from oracle import flce_oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = sorted([q.get(timeout=180) for _ in range(2)], key=lambda x: x[0])
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    p = wl.random_problem(203, 24, 77, seed=5, ignore_frac=0.3)
    full = flce_oracle(p["hidden"], p["weight"], p["targets"])
    for rank, loss, n, gw, gh, a, b, t in res:
        assert n == full["n_valid"]
        assert abs(loss - full["loss"]) <= 1e-12 * abs(full["loss"])
        np.testing.assert_allclose(gw, full["grad_weight"], rtol=1e-10, atol=1e-15)
        np.testing.assert_allclose(gh, full["grad_hidden"][a:b], rtol=1e-10, atol=1e-15)
        assert t == 11.0          # max over ranks of 10 + rank
