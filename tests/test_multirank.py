"""Replica sharding across ranks (world size 2, gloo, CPU): each rank takes its
contiguous share of independent requests, runs the cycle on its share, and
the gathered results equal the single-process run.  There is no collective
on the data path -- only the test gathers results to compare them."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import spec_oracle as O
        from speculative_decoding_draft_04_gb300 import workloads as W
        w = W.make_workload(W.config("C2", B=10, V=512, r=32), trial=3)
        rows = W.shard_rows(w.B, rank, world)
        sub = w.subset(rows)
        res = O.cycle(sub.f64("target"), sub.f64("U"), sub.f64("W1"), sub.f64("W2"), sub.anchor,
                      sub.temperature.astype(np.float64), sub.u_draft.astype(np.float64),
                      sub.verify_len, sub.u_accept.astype(np.float64),
                      sub.u_final.astype(np.float64))
        mine = torch.tensor(np.concatenate([rows[:, None], res.out_tokens(),
                                            res.accept_len()[:, None]], axis=1), dtype=torch.int64)
        n = torch.tensor([mine.shape[0]])
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, n)
        pad = torch.full((int(max(s.item() for s in sizes)), mine.shape[1]), -9, dtype=torch.int64)
        pad[: mine.shape[0]] = mine
        got = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(got, pad)
        if rank == 0:
            allrows = torch.cat([g[: int(s.item())] for g, s in zip(got, sizes)]).numpy()
            q.put(allrows)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_match_single_process():
    from oracle import spec_oracle as O
    from speculative_decoding_draft_04_gb300 import workloads as W
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = W.make_workload(W.config("C2", B=10, V=512, r=32), trial=3)
    ref = O.cycle(w.f64("target"), w.f64("U"), w.f64("W1"), w.f64("W2"), w.anchor,
                  w.temperature.astype(np.float64), w.u_draft.astype(np.float64), w.verify_len,
                  w.u_accept.astype(np.float64), w.u_final.astype(np.float64))
    order = np.argsort(got[:, 0])
    np.testing.assert_array_equal(got[order, 0], np.arange(w.B))
    np.testing.assert_array_equal(got[order, 1:-1], ref.out_tokens())
    np.testing.assert_array_equal(got[order, -1], ref.accept_len())
