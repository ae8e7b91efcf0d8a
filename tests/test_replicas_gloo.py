"""The N>1 path on CPU: two gloo ranks run independent replicas of the layer.

Each rank draws its own batch (seed + rank), runs the whole layer on it with
no collective on the data path, then takes part in the two host-side steps
the bench uses (barrier, max over the ranks' times). The test checks that a
rank's output equals the single-process layer on that rank's batch, that the
ranks really processed different batches, and that the aggregate throughput
is all ranks' tokens over the slowest rank's time.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from mxfp4_latent_moe_gb300 import replicas, synth

WL = synth.shape("replica", T=6, d=128, E=10, k=3, I=64)
STEPS = 3


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer_output(seed):
    import oracle
    L = synth.make_layer(WL, seed=seed)
    W = [L[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s")]
    return oracle.moe_forward(synth.bf16_bits(L["x"]), L["logits"].numpy(), WL.k, *W)["y"]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = replicas.dist_env()
        assert (r, w, local) == (rank, world, rank)
        y = _layer_output(replicas.replica_seed(0, rank))
        replicas.barrier()
        my_ms = 10.0 * (rank + 1)
        max_ms = replicas.max_over_ranks(my_ms)
        rate = replicas.aggregate_rate(WL.T, world, STEPS, max_ms)
        np.save(os.path.join(outdir, "y%d.npy" % rank), y)
        np.save(os.path.join(outdir, "t%d.npy" % rank), np.array([max_ms, rate]))
        replicas.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_replicas(orc):
    world = 2
    with tempfile.TemporaryDirectory() as outdir:
        mp.start_processes(_rank_main, args=(world, _free_port(), outdir), nprocs=world,
                           join=True, start_method="spawn")
        ys = [np.load(os.path.join(outdir, "y%d.npy" % r)) for r in range(world)]
        ts = [np.load(os.path.join(outdir, "t%d.npy" % r)) for r in range(world)]
    for r in range(world):
        np.testing.assert_array_equal(ys[r], _layer_output(replicas.replica_seed(0, r)))
        assert ts[r][0] == 20.0                                  # slowest rank's 20 ms
        assert ts[r][1] == pytest.approx(world * WL.T * STEPS / 0.020)
    assert not np.array_equal(ys[0], ys[1]), "replicas must process different batches"


def test_single_process_identity():
    assert not torch.distributed.is_initialized()
    assert replicas.max_over_ranks(3.5) == 3.5
    replicas.barrier()
    assert replicas.aggregate_rate(64, 1, 10, 100.0) == pytest.approx(6400.0)
    with pytest.raises(ValueError):
        replicas.aggregate_rate(64, 1, 10, 0.0)
