"""Row-sharded Engram tables across ranks, with one exchange of the module
sums per call (rohitghumare.com "guides/deepseek-v4-1-flash", section
"Engram: the table that is never multiplied": SGLang splits the tables by
row across tensor-parallel GPUs and pays one all-reduce per Engram layer).

Row r of every table belongs to rank r mod G and is stored there as local row
r // G.  Each rank gathers only the rows it owns for every query token
(``engram_gather_reduce_shard``, CUDA), the partial fp32 sums [T, 512] are
summed over ranks by one all-reduce (torch.distributed: NCCL between GPUs),
and every rank then applies the gated projection to its copy of h
(``engram_fuse``).  The all-reduce moves 2 KB per token, less than reducing
the d-wide projection output would (2 d bytes per token in bf16).
"""

import torch

from . import engram_fuse, engram_gather_reduce_shard, engram_shard_rows


def row_owner(rows, n_shards):
    """(owning rank, local row) of global row indices under the mod-G split."""
    return rows % n_shards, rows // n_shards


def shard_tables(tables, scales, rank, n_shards, rows_per_shard):
    """This rank's rows of every table: rows rank, rank + G, rank + 2G, ...,
    as [48, rows_per_shard, row_bytes] (and [48, rows_per_shard] scales, or
    None for rows that carry their scale), padded with zero rows at the end;
    on the device of `tables`."""
    mine = tables[:, rank::n_shards]
    out = torch.zeros((tables.shape[0], rows_per_shard, tables.shape[2]), dtype=tables.dtype, device=tables.device)
    out[:, :mine.shape[1]] = mine
    sc = None
    if scales is not None:
        sm = scales[:, rank::n_shards]
        sc = torch.zeros((scales.shape[0], rows_per_shard), dtype=scales.dtype, device=scales.device)
        sc[:, :sm.shape[1]] = sm
    return out, sc


def reduce_partials(mem, group=None):
    """The one exchange: sum the ranks' partial module sums in place."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(mem, op=dist.ReduceOp.SUM, group=group)
    return mem


def forward_row_sharded(cfg, rank, n_shards, tokens, seq_offsets, tables_shard, scales_shard, W_out, g, h, last_n=0,
                        n_query=None, mem=None, group=None, stream=None):
    """Steps 1-5 with row-sharded tables: partial gather, all-reduce of the
    module sums, gated projection into this rank's h (in place)."""
    assert tables_shard.shape[1] == engram_shard_rows(cfg, n_shards)
    mem = engram_gather_reduce_shard(cfg, rank, n_shards, tokens, seq_offsets, tables_shard, scales_shard,
                                     last_n=last_n, n_query=n_query, mem=mem, stream=stream)
    reduce_partials(mem, group)
    engram_fuse(cfg, mem, W_out, g, h, stream=stream)
    return h
