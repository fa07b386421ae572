"""bench.py's multi-rank pieces on CPU with gloo, world size 2: whole-job
throughput uses every rank's units over the slowest rank's time, and ranks
draw distinct token batches on the same tables."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from synth.configs import CONFIGS, make_tokens


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [10.0, 25.0][rank]  # rank 1 is the slow one
    rate, ms_max = bench.job_rate(local_ms, 5, 1000, world, torch.device("cpu"))
    out[rank] = (rate, ms_max)
    dist.barrier()
    dist.destroy_process_group()


def test_job_rate_is_max_over_ranks_gloo():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        rate, ms_max = res[r]
        assert ms_max == 25.0
        assert abs(rate - 2 * 1000 / (25e-3 / 5)) < 1e-6


def test_rank_batches_differ_but_tables_do_not():
    base = CONFIGS["tiny"]
    c0, c1 = bench.rank_config(base, 0), bench.rank_config(base, 1)
    assert c0 == base and c1.seed != base.seed
    assert (c0.V, c0.R, c0.d, c0.seq_lens) == (c1.V, c1.R, c1.d, c1.seq_lens)
    t0, _ = make_tokens(c0)
    t1, _ = make_tokens(c1)
    assert not np.array_equal(t0, t1)
