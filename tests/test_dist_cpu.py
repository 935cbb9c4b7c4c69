"""Multi-process paths on CPU with gloo, world size 2.

1. Sharding by whole sequences (how the estimator splits across GPUs): each
   rank estimates GW from its own sequences with the oracle (the scan never
   crosses a sequence and the hash uses global token indices), one all-reduce
   sums the shards, and the sum equals the unsharded estimate.
2. Sharding by draws (the split the pages' eight GPUs use): rank r owns a
   range of absolute draw indices (draw_begin), the loss changes are centred
   once over all K draws, and each shard's estimate, scaled by its share of
   the draws, sums to the unsharded centred estimate.
3. The benchmark's whole-job aggregation: the max over ranks of the timed
   region and units summed over ranks.
"""
import os
import socket

import numpy as np
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import sys
    import torch
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import oracle
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(0)
    lengths = [30, 50, 20, 40]
    so = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, d_in, d_out, K = int(so[-1]), 6, 9, 4
    X = rng.standard_normal((T, d_in))
    delta = rng.standard_normal((K, T))
    # rank r owns sequences [2r, 2r+2)
    Xs = np.zeros_like(X)
    lo, hi = so[2 * rank], so[2 * rank + 2]
    Xs[lo:hi] = X[lo:hi]
    part = oracle.estimate_gW(Xs, delta, d_out, so, 5, 1, 0, 0.01, 0.9, 1.0, oracle.CENTER)
    t = torch.from_numpy(part)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    # draws [2r, 2r + 2) on rank r, centred over all K beforehand (CENTER off)
    centred = delta - delta.mean(axis=0, keepdims=True)
    d0, d1 = 2 * rank, 2 * rank + 2
    dpart = oracle.estimate_gW(X, centred[d0:d1], d_out, so, 5, 1, d0, 0.01, 0.9,
                               (d1 - d0) / K, 0)
    td = torch.from_numpy(dpart)
    dist.all_reduce(td, op=dist.ReduceOp.SUM)

    def max_over_ranks(x):
        v = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(v, op=dist.ReduceOp.MAX)
        return float(v.item())

    ms_local = 100.0 + 50.0 * rank  # rank 1 is the slow one
    value, ms_per_step = bench.aggregate(1000.0, ms_local, 10, world, max_over_ranks)
    if rank == 0:
        full = oracle.estimate_gW(X, delta, d_out, so, 5, 1, 0, 0.01, 0.9, 1.0, oracle.CENTER)
        np.save(os.path.join(out_dir, "sum.npy"), t.numpy())
        np.save(os.path.join(out_dir, "dsum.npy"), td.numpy())
        np.save(os.path.join(out_dir, "full.npy"), full)
        np.save(os.path.join(out_dir, "agg.npy"), np.array([value, ms_per_step]))
    dist.barrier()
    dist.destroy_process_group()


def test_sequence_sharded_estimate_and_bench_aggregation(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    s = np.load(tmp_path / "sum.npy")
    f = np.load(tmp_path / "full.npy")
    assert np.allclose(s, f, rtol=1e-12, atol=1e-12 * np.abs(f).max())
    ds = np.load(tmp_path / "dsum.npy")
    assert np.allclose(ds, f, rtol=1e-10, atol=1e-10 * np.abs(f).max())
    value, ms_per_step = np.load(tmp_path / "agg.npy")
    assert ms_per_step == pytest.approx(15.0)          # max over ranks: 150 ms / 10 steps
    assert value == pytest.approx(2 * 1000.0 * 10 / 0.150)
