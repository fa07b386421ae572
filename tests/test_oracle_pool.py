"""The all-token checker (tests/oracle_pool.py) on CPU: spawned workers rebuild
inputs from the host twins and run the oracle; results that match pass, and a
planted error in either output is counted."""

import numpy as np

import oracle
import oracle_pool
from oracle_pool import check_layer_all_tokens
from synth import host
from synth.configs import CONFIGS, default_seeds, make_tokens, query_positions


def _setup():
    cfg = CONFIGS["tiny"]
    seeds = default_seeds()
    tok, offs = make_tokens(cfg)
    qpos = query_positions(cfg, offs)
    oracle_pool._init(cfg.seed, cfg.d, cfg.rms_eps, cfg.V, cfg.R, seeds, tok, offs, qpos)
    mem, _, hn = oracle_pool.reference(np.arange(cfg.tq))
    return cfg, seeds, tok, offs, qpos, mem.astype(np.float32), hn


def test_all_tokens_match_and_planted_errors_are_counted():
    cfg, seeds, tok, offs, qpos, mem, h = _setup()
    s = oracle_pool.check_all_tokens(cfg, seeds, tok, offs, qpos, mem, h, chunk=128, procs=2)
    assert s["tokens"] == cfg.tq and s["mem_bad"] == 0 and s["h_bad"] == 0, s
    mem2, h2 = mem.copy(), h.copy()
    mem2[300, 7] += 1.0                 # far outside 1e-5 x sum|term|
    r = oracle_pool._bf16_f64(h2[5, 3:4])[0]
    h2[5, 3] = np.uint16(((np.float32(r + 4.0 * max(1.0, abs(r)))).view(np.uint32) >> 16))
    s2 = oracle_pool.check_all_tokens(cfg, seeds, tok, offs, qpos, mem2, h2, chunk=128, procs=2)
    assert s2["mem_bad"] == 1 and s2["h_bad"] == 1, s2


def test_layer_pool_checker_counts_planted_errors():
    """The every-token checker of the per-layer form: the oracle's own outputs
    pass; a flipped exponent bit in one h element and a wrong X element are
    each counted once."""
    import torch

    cfg = CONFIGS["tiny"].with_(seq_lens=(40, 9), R=4096)
    tok, offs = make_tokens(cfg)
    qpos = query_positions(cfg, offs)
    seeds = default_seeds()
    m = 1
    idx = oracle.hash_positions(tok, offs, cfg.V, cfg.R, seeds, qpos)
    jj = np.tile(np.arange(24 * m, 24 * m + 24), cfg.tq)
    r = idx[:, 24 * m:24 * m + 24].reshape(-1)
    codes = host.table_rows(cfg.seed, jj, r).reshape(cfg.tq, 24, 256)
    sc = host.scales(cfg.seed, jj, r).reshape(cfg.tq, 24)
    wq, wk, wm = host.layer_weights(cfg.seed, cfg.d, m)
    h0 = host.h_rows(cfg.seed, cfg.d, np.arange(cfg.tq))
    hn, _, e = oracle.layer_gated(codes, sc, wq, wk, wm, h0, cfg.rms_eps)
    x = torch.from_numpy(e).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ok = check_layer_all_tokens(cfg, seeds, tok, offs, qpos, m, h0, hn, x, chunk=16, procs=2)
    assert ok["tokens"] == cfg.tq and ok["h_bad"] == 0 and ok["x_bad"] == 0
    hb, xb = hn.copy(), x.copy()
    hb[3, 5] ^= 0x4000
    xb[7, 9] ^= 0x4000
    bad = check_layer_all_tokens(cfg, seeds, tok, offs, qpos, m, h0, hb, xb, chunk=16, procs=2)
    assert bad["h_bad"] == 1 and bad["x_bad"] == 1
