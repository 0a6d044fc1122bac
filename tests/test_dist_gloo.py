"""Multi-rank host logic on CPU: world_size 2, gloo backend, 127.0.0.1.

* shard_range splits heads / batch rows into disjoint covering slices;
* max_over_ranks returns the slowest rank's time (bench's job time);
* batch-sharded training: each rank runs the fp64 oracle's BPTT on its batch
  shard, allreduce_weight_grads sums dR and db, and the result equals the
  full-batch gradients (dR, db are sums over batch rows).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sequential_rnn_gb300.dist import allreduce_weight_grads, max_over_ranks, shard_range


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import rnn_oracle as O
        from synth import make_inputs
        d = make_inputs("lstm", "f32", 6, 5, 2, 4, seed=3, bias="normal", states="random",
                        backward=True)
        lo, hi = shard_range(d["B"], rank, world)
        g = O.lstm_backward(d["Wx"][:, lo:hi], d["R"], d["b"], d["h0"][lo:hi], d["c0"][lo:hi],
                            dh_seq=d["dh"][:, lo:hi])
        dR = torch.from_numpy(g["dR"].copy())
        db = torch.from_numpy(g["db"].copy())
        allreduce_weight_grads(dR, db)
        tmax = max_over_ranks(1.5 + rank)
        out[rank] = (dR.numpy(), db.numpy(), tmax, (lo, hi))
    finally:
        dist.destroy_process_group()


def test_shard_range_covers_disjointly():
    for n in (0, 1, 5, 12, 13):
        for world in (1, 2, 3, 8):
            parts = [shard_range(n, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_range(4, 2, 2)


def test_two_rank_gloo_batch_sharded_gradients():
    from oracle import rnn_oracle as O
    from synth import make_inputs
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    d = make_inputs("lstm", "f32", 6, 5, 2, 4, seed=3, bias="normal", states="random",
                    backward=True)
    full = O.lstm_backward(d["Wx"], d["R"], d["b"], d["h0"], d["c0"], dh_seq=d["dh"])
    for rank in (0, 1):
        dR, db, tmax, _ = res[rank]
        np.testing.assert_allclose(dR, full["dR"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(db, full["db"], rtol=0, atol=1e-12)
        assert tmax == 2.5
    assert res[0][3] == (0, 3) and res[1][3] == (3, 5)
