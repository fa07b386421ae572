"""Row-sharded tables on CPU ranks (gloo, world size 2): the partition of the
tables and the exchange of the partial module sums, checked against the
oracle on the whole tables.  Each rank's partial sums are taken with the
oracle over the rows its shard holds; the CUDA kernel that computes them on
a GPU is checked in test_gpu_shard.py."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from engram_gram_hash_gb300 import shard
from synth import host
from synth.configs import CONFIGS, default_seeds, make_tokens

CFG = CONFIGS["tiny"].with_(seq_lens=(90, 1, 37), R=4093, seed=13)  # prime R: shards of unequal size


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _partial_mem(rank, world, tables, scales, idx):
    """Oracle sums over the rows this rank's shard holds (others add nothing)."""
    rows_per = -(-CFG.R // world)
    t_sh, s_sh = shard.shard_tables(torch.from_numpy(tables), torch.from_numpy(scales), rank, world, rows_per)
    owner, local = shard.row_owner(idx, world)
    mine = owner == rank
    jj = np.broadcast_to(np.arange(48), idx.shape)
    rows = t_sh.numpy()[jj, np.where(mine, local, 0)]
    sc = np.where(mine, s_sh.numpy()[jj, np.where(mine, local, 0)], 0.0).astype(np.float32)
    rows = np.where(mine[:, :, None], rows, 0).astype(np.uint8)
    return oracle.gather_reduce_rows(rows, sc)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    tok, offs = make_tokens(CFG)
    tables, scales = host.full_tables(CFG.seed, CFG.R)
    idx = oracle.hash_tokens(tok, offs, 0, CFG.V, CFG.R, default_seeds())
    mem = torch.from_numpy(_partial_mem(rank, world, tables, scales, idx))
    shard.reduce_partials(mem)
    out[rank] = mem.numpy().tobytes()
    dist.barrier()
    dist.destroy_process_group()


def test_row_shards_sum_to_the_whole_gather_gloo():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = {r: np.frombuffer(out[r], dtype=np.float64).reshape(-1, 512) for r in (0, 1)}
    tok, offs = make_tokens(CFG)
    tables, scales = host.full_tables(CFG.seed, CFG.R)
    idx = oracle.hash_tokens(tok, offs, 0, CFG.V, CFG.R, default_seeds())
    whole = oracle.gather_reduce(tables, scales, idx)
    # the oracle's sums are exact (every term a multiple of 2^-33 below 2^10),
    # so the exchanged partial sums equal the whole sums bit for bit
    assert np.array_equal(res[0], whole) and np.array_equal(res[1], whole)


def test_row_owner_and_shard_tables_partition_every_row():
    """Every global row is held by exactly one shard, at its local row."""
    R, G = 4093, 3
    tables = torch.arange(2 * R * 16, dtype=torch.int64).reshape(2, R, 16).to(torch.uint8)
    scales = torch.arange(2 * R, dtype=torch.float32).reshape(2, R)
    rows_per = -(-R // G)
    shards = [shard.shard_tables(tables, scales, s, G, rows_per) for s in range(G)]
    r = np.arange(R)
    owner, local = shard.row_owner(r, G)
    for j in range(2):
        for s in range(G):
            sel = owner == s
            assert torch.equal(shards[s][0][j, local[sel]], tables[j, r[sel]])
            assert torch.equal(shards[s][1][j, local[sel]], scales[j, r[sel]])
    assert sum(int((owner == s).sum()) for s in range(G)) == R
    assert all(t.shape[1] == rows_per for t, _ in shards)
