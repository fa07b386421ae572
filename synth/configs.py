"""The five synthetic workloads and their seeded input recipes.

Sizes follow the Engram description on the DeepSeek-V4.1-Flash pages
(2/3/4-grams x 8 heads x 2 modules = 48 rows of 256 FP8 values per token;
"What makes up the 511 GB of weights?" and "Engram: the table that is never
multiplied"), with vocabulary, row counts, token mixes and d_model fixed by
the workload definitions below.
"""

from dataclasses import dataclass, replace

import numpy as np

# Philox stream ids (key word 1); key word 0 is the workload seed.
STREAM_TABLE = 0x100  # + table j: one u32 per e4m3 code, word = row*256 + c
STREAM_SCALE = 0x200  # + table j: one u32 per row, word = row
STREAM_H = 0x300  # word = t*d + c
STREAM_W = 0x301  # word = k*d + c
STREAM_G = 0x302  # word = c
STREAM_MX = 0x400  # + table j: eight u32 per row (one per E8M0 block scale), word = row*8 + b
STREAM_WQ = 0x500  # + layer m: per-row gate query weights W_q [d][256], word = i*256 + c
STREAM_WK = 0x510  # + layer m: per-row gate key weights W_k [256][256], word = i*256 + c
STREAM_WM = 0x520  # + layer m: layer projection W_m [256][d], word = c*d + n

N_TABLES = 48
ROW_BYTES = 256
K_MEM = 512  # 2 modules x 256


def splitmix64(state, n):
    """First n outputs of SplitMix64 (Steele, Lea & Flood, OOPSLA 2014)."""
    mask = (1 << 64) - 1
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & mask
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        out.append(z ^ (z >> 31))
    return out


def default_seeds():
    """Per-table hash seeds: SplitMix64 from state 0, in table order j."""
    return np.array(splitmix64(0, N_TABLES), dtype=np.uint64)


@dataclass(frozen=True)
class EngramConfig:
    name: str
    V: int  # vocabulary size; V itself is the pad id
    R: int  # rows per table
    seq_lens: tuple  # tokens per sequence
    last_n: int  # 0: query every position; k: the last k of each sequence
    zipf_s: float  # 0.0 means uniform ids
    span_frac: float  # fraction of each sequence overwritten by one repeated span
    span_len: int
    d: int  # d_model
    seed: int
    host_tables: bool = False
    rms_eps: float = 1e-6

    @property
    def n_seqs(self):
        return len(self.seq_lens)

    @property
    def t_all(self):
        return int(sum(self.seq_lens))

    @property
    def tq(self):
        if self.last_n == 0:
            return self.t_all
        return self.n_seqs * self.last_n

    @property
    def table_bytes(self):
        return N_TABLES * self.R * ROW_BYTES

    def with_(self, **kw):
        return replace(self, **kw)


CONFIGS = {
    "tiny": EngramConfig("tiny", 1024, 4096, (512,), 0, 1.1, 0.0, 64, 256, 0),
    "decode": EngramConfig("decode", 129280, 1 << 20, (4,) * 64, 1, 1.1, 0.0, 64, 4096, 1),
    "prefill": EngramConfig("prefill", 129280, 1 << 21, (32768,) * 8, 0, 1.05, 0.2, 64, 4096, 2),
    "large": EngramConfig("large", 129280, 1 << 23, (131072,), 0, 0.0, 0.0, 64, 4096, 3),
    "host": EngramConfig("host", 129280, 1 << 22, (65536,), 0, 1.1, 0.0, 64, 4096, 4, host_tables=True),
}


def zipf_ids(rng, V, s, n):
    """n ids with P(id = k-1) proportional to k^-s for ranks k in [1, V]."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    u = rng.random(n) * cdf[-1]
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int32)


def make_tokens(cfg):
    """Token stream int32 [t_all] and seq_offsets int64 [n_seqs+1]."""
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 0x746F6B]))
    parts = []
    for L in cfg.seq_lens:
        if cfg.zipf_s > 0.0:
            x = zipf_ids(rng, cfg.V, cfg.zipf_s, L)
        else:
            x = rng.integers(0, cfg.V, size=L, dtype=np.int64).astype(np.int32)
        if cfg.span_frac > 0.0:
            span = zipf_ids(rng, cfg.V, cfg.zipf_s, cfg.span_len) if cfg.zipf_s > 0 else rng.integers(
                0, cfg.V, size=cfg.span_len
            ).astype(np.int32)
            n_slots = L // cfg.span_len
            n_copy = int(np.floor(cfg.span_frac * L / cfg.span_len))
            slots = rng.choice(n_slots, size=n_copy, replace=False)
            for s in slots:
                x[s * cfg.span_len : (s + 1) * cfg.span_len] = span
        parts.append(x)
    tokens = np.concatenate(parts).astype(np.int32)
    offs = np.zeros(cfg.n_seqs + 1, dtype=np.int64)
    offs[1:] = np.cumsum(cfg.seq_lens)
    return tokens, offs


def span_info(cfg):
    """(span start positions, span_len) of the repeated-span copies, per make_tokens."""
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 0x746F6B]))
    out = []
    base = 0
    for L in cfg.seq_lens:
        if cfg.zipf_s > 0.0:
            zipf_ids(rng, cfg.V, cfg.zipf_s, L)
        else:
            rng.integers(0, cfg.V, size=L, dtype=np.int64)
        if cfg.span_frac > 0.0:
            if cfg.zipf_s > 0:
                zipf_ids(rng, cfg.V, cfg.zipf_s, cfg.span_len)
            else:
                rng.integers(0, cfg.V, size=cfg.span_len)
            n_slots = L // cfg.span_len
            n_copy = int(np.floor(cfg.span_frac * L / cfg.span_len))
            slots = rng.choice(n_slots, size=n_copy, replace=False)
            out.extend(base + int(s) * cfg.span_len for s in slots)
        base += L
    return np.array(sorted(out), dtype=np.int64), cfg.span_len


def query_positions(cfg, offs):
    """Global positions of the query tokens, in query order."""
    if cfg.last_n == 0:
        return np.arange(int(offs[-1]), dtype=np.int64)
    out = []
    for s in range(cfg.n_seqs):
        lo, hi = int(offs[s]), int(offs[s + 1])
        assert hi - lo >= cfg.last_n, "every sequence must hold at least last_n tokens"
        out.extend(range(hi - cfg.last_n, hi))
    return np.array(out, dtype=np.int64)
