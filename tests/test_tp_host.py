"""Tensor-parallel vocabulary sharding, host side (CPU, gloo, world size 2): the vocabulary
split and the all-gather of per-rank shard statistics, merged here with the oracle and checked
against whole-row statistics."""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_vocab_range_partitions_the_vocabulary():
    sys.path.insert(0, ROOT)
    from diffusion_decoding_gb300.tp import vocab_range
    for V in (1, 7, 126464, 126465):
        for world in (1, 2, 3, 8):
            if world > V:
                continue
            spans = [vocab_range(V, world, k) for k in range(world)]
            assert spans[0][0] == 0
            for (a, n), (b, _) in zip(spans, spans[1:]):
                assert a + n == b
            assert spans[-1][0] + spans[-1][1] == V
            assert max(n for _, n in spans) - min(n for _, n in spans) <= 1


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist
    import oracle
    from diffusion_decoding_gb300.tp import all_gather_shard_stats, vocab_range
    dist.init_process_group("gloo", rank=rank, world_size=world)
    V, R = 1001, 12
    rng = np.random.default_rng(5)                       # same full logits on every rank
    x = rng.normal(0, 2, size=(R, V)).astype(np.float32)
    x[3, 10] = x[3, 900] = 11.0                          # a tie across the two ranks' shards
    masked = (rng.random(R) < 0.8).astype(np.uint8)
    first, n = vocab_range(V, world, rank)
    local = oracle.stats(np.ascontiguousarray(x[:, first:first + n]), masked)

    class Local:
        row_max = torch.from_numpy(local.row_max.astype(np.float32))
        lse = torch.from_numpy(local.lse.astype(np.float32))
        argmax = torch.from_numpy(local.argmax)

    gathered = all_gather_shard_stats(Local)
    shards = []
    for g in gathered:
        s = oracle.Stats(R)
        s.row_max[:] = g.row_max.numpy()
        s.lse[:] = g.lse.numpy()
        s.argmax[:] = g.argmax.numpy()
        shards.append(s)
    merged = oracle.merge_shard_stats(shards, [vocab_range(V, world, k)[0] for k in range(world)])
    full = oracle.stats(x, masked)
    act = masked.astype(bool)
    out[rank] = (bool(np.array_equal(merged.argmax, full.argmax)),
                 float(np.max(np.abs(merged.lse[act] - full.lse[act]) / np.abs(full.lse[act]))),
                 bool(np.array_equal(merged.row_max.astype(np.float32),
                                     full.row_max.astype(np.float32))))
    dist.destroy_process_group()


def test_two_ranks_gather_shard_statistics_and_merge_to_the_whole_row():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        argmax_ok, lse_rel, max_ok = out[r]
        assert argmax_ok and max_ok
        assert lse_rel < 1e-6   # the shard statistics crossed the wire as float32
