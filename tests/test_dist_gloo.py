"""Data-parallel decomposition over whole pairs, two gloo ranks on CPU.

Each rank takes its block of pairs (orpo_preference_loss_gb300.dp), runs the
float64 oracle on its rows with its own pair count, rescales loss and
cotangent by P_rank / P, and all-reduces the loss, metric sums and dW.  The
result must equal the single-process oracle on the whole batch.  The bench's
max-over-ranks timing reduction runs through the same process group."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads
from orpo_preference_loss_gb300 import dp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        w = workloads.make("small", M=400, d=16, V=96)
        h, W = oracle.bf16_bits_to_f64(w.h), oracle.bf16_bits_to_f64(w.W)
        rows, local_seq, P_loc, scale = dp.shard_pairs(w.seq_id, w.n_pairs, rank, WORLD)
        logp, lse, res, dh, dW = oracle.full_chain(h[rows], W, w.targets[rows], w.mask[rows], local_seq, P_loc,
                                                    w.lam, w.softcap)
        # rescale so that the sum over ranks is the global mean over pairs
        dh *= scale
        dW *= scale
        sums = torch.tensor(res.metrics() * scale, dtype=torch.float64)
        dW_t = torch.from_numpy(dW)
        dist.all_reduce(sums)
        dist.all_reduce(dW_t)
        # the bench's timing reduction: max over ranks
        t = torch.tensor([10.0 + rank], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                {"sums": sums.numpy(), "dW": dW_t.numpy(), "rows": rows, "dh": dh, "tmax": float(t.item())},
                allow_pickle=True)
    finally:
        dist.destroy_process_group()


def test_pairs_split_across_two_ranks_reproduce_the_global_step(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(port, str(tmp_path)), nprocs=WORLD, start_method="spawn")
    w = workloads.make("small", M=400, d=16, V=96)
    h, W = oracle.bf16_bits_to_f64(w.h), oracle.bf16_bits_to_f64(w.W)
    _, _, res, dh, dW = oracle.full_chain(h, W, w.targets, w.mask, w.seq_id, w.n_pairs, w.lam, w.softcap)
    outs = [np.load(os.path.join(tmp_path, f"rank{r}.npy"), allow_pickle=True).item() for r in range(WORLD)]
    for o in outs:
        assert np.allclose(o["sums"][[0, 1, 2, 4]], res.metrics()[[0, 1, 2, 4]], rtol=1e-12, atol=1e-14)
        assert np.allclose(o["sums"][3], res.accuracy)   # accuracy: mean of per-pair indicators
        assert np.allclose(o["dW"], dW, rtol=1e-10, atol=1e-16)
        assert o["tmax"] == 11.0
    # every row's dh lives on exactly one rank and equals the global one
    got = np.zeros_like(dh)
    seen = np.zeros(w.M, dtype=int)
    for o in outs:
        got[o["rows"]] = o["dh"]
        seen[o["rows"]] += 1
    assert np.all(seen[w.seq_id >= 0] == 1)
    assert np.allclose(got, dh, rtol=1e-10, atol=1e-16)


def test_shard_pairs_partitions_the_pairs():
    seq = np.array([0, 0, 1, -1, 2, 3, 3, 4, 5, -1, 6, 7])
    r0 = dp.shard_pairs(seq, 4, 0, 2)
    r1 = dp.shard_pairs(seq, 4, 1, 2)
    assert list(r0[0]) == [0, 1, 2, 4, 5, 6] and list(r0[1]) == [0, 0, 1, 2, 3, 3]
    assert list(r1[0]) == [7, 8, 10, 11] and list(r1[1]) == [0, 1, 2, 3]
    assert r0[2] == 2 and r1[2] == 2 and r0[3] == 0.5
    with pytest.raises(ValueError):
        dp.shard_pairs(seq, 1, 0, 2)
