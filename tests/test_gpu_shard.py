"""Row-sharded tables on the GPU: every shard's partial gather through the C
ABI, run one after another on one GPU, against the oracle (needs a GB300).
The shards' sum stands in for the all-reduce of the multi-GPU form."""

import numpy as np
import pytest
import torch

import oracle
from engram_gram_hash_gb300 import shard
from synth import host
from synth.configs import CONFIGS
from workload import Workload, check_h, check_mem, sample_queries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


CASES = {
    # prime R: shards of unequal size; ragged sequences with the pad
    "ragged_prime_g3": (CONFIGS["tiny"].with_(seq_lens=(300, 1, 2, 140, 77), R=4093, seed=5), 3),
    # d = 4096, several tiles, repeated spans; four shards
    "prefill_small_g4": (CONFIGS["prefill"].with_(seq_lens=(640, 421), R=1 << 16, seed=6), 4),
}


@pytest.mark.parametrize("name", list(CASES))
def test_row_shards_partial_and_total(eg, name):
    cfg, G = CASES[name]
    w = Workload(cfg)
    nq = cfg.tq
    rows_per = eg.engram_shard_rows(w.c, G)
    assert rows_per == -(-cfg.R // G)
    parts = []
    for s in range(G):
        t_s, sc_s = shard.shard_tables(w.tables, w.scales, s, G, rows_per)
        parts.append(eg.engram_gather_reduce_shard(w.c, s, G, w.tokens, w.seq_offsets, t_s, sc_s,
                                                   last_n=cfg.last_n))
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    q = np.arange(nq) if nq <= 2048 else sample_queries(cfg, w.offs, 300)
    idx, mem_ref, bound, h_ref, _ = w.ref_for(q)
    # each shard: the oracle's sums over the rows it owns
    owner, _ = shard.row_owner(idx, G)
    jj = np.tile(np.arange(48), len(q))
    rows = host.table_rows(cfg.seed, jj, idx.reshape(-1)).reshape(len(q), 48, 256)
    sc = host.scales(cfg.seed, jj, idx.reshape(-1)).reshape(len(q), 48)
    qt = torch.from_numpy(q).cuda()
    for s in range(G):
        mine = owner == s
        ref_s = oracle.gather_reduce_rows(np.where(mine[:, :, None], rows, 0).astype(np.uint8),
                                          np.where(mine, sc, 0).astype(np.float32))
        check_mem(parts[s][qt].cpu().numpy(), ref_s, bound)
    # the exchange (the shards' sum) then the projection
    total = parts[0].clone()
    for s in range(1, G):
        total += parts[s]
    check_mem(total[qt].cpu().numpy(), mem_ref, bound)
    h = w.fresh_h()
    eg.engram_fuse(w.c, total, w.W, w.g, h)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    check_h(h[qt], h_ref)


def test_one_shard_is_the_whole_gather(eg):
    """n_shards = 1: the shard is the whole table and the partial sums are
    engram_gather_reduce's bits."""
    cfg = CASES["ragged_prime_g3"][0]
    w = Workload(cfg)
    a = eg.engram_gather_reduce_shard(w.c, 0, 1, w.tokens, w.seq_offsets, w.tables, w.scales)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    b = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(a, b)
