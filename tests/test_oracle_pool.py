"""The all-token checker (tests/oracle_pool.py) on CPU: spawned workers rebuild
inputs from the host twins and run the oracle; results that match pass, and a
planted error in either output is counted."""

import numpy as np

import oracle_pool
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
