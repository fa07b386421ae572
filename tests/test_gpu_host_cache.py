"""The host-table path with a cache of staged rows across calls (needs a
GB300): every call's h equals the HBM path's bit for bit, whatever mix of
cache hits, misses and overflow rows served it; a repeated batch is served
from the cache."""

import numpy as np
import pytest
import torch

from synth.configs import CONFIGS, make_tokens
from workload import Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


CFG = CONFIGS["host"].with_(seq_lens=(700, 555), R=1 << 15, seed=9)


def _batch(cfg, seed):
    """Tokens of another batch drawn over the same vocabulary (tables unchanged)."""
    tok, offs = make_tokens(cfg.with_(seed=seed))
    return torch.from_numpy(tok).cuda(), torch.from_numpy(offs).cuda()


def _hbm_h(eg, w, dev_tables, dev_scales, tokens, offs):
    h = w.fresh_h()
    eg.engram_forward(w.c, tokens, offs, dev_tables, dev_scales, w.W, w.g, h)
    return h


@pytest.mark.parametrize("slots", [1 << 20, 64])
def test_cached_calls_match_hbm_path(eg, slots):
    """Three calls on one cache: batch A cold, batch A again, batch B.  A large
    cache serves the repeat almost wholly from HBM; a 64-slot cache sends most
    rows to the overflow area; the bits never change."""
    w = Workload(CFG, host_tables=True)
    cap = CFG.tq * 48
    cache = eg.engram_host_cache_new(w.c, slots, cap)
    dev_t, dev_s = w.tables.cuda(), w.scales.cuda()
    side = torch.cuda.Stream()
    batches = [(w.tokens, w.seq_offsets), (w.tokens, w.seq_offsets), _batch(CFG, 77)]
    stats = []
    for k, (tk, of) in enumerate(batches):
        h = w.fresh_h()
        st = eg.engram_forward_host_cached(w.c, tk, of, w.tables, w.scales, w.W, w.g, h, cache, slots, cap,
                                           stamp=k + 1, side_stream=side)
        ref = _hbm_h(eg, w, dev_t, dev_s, tk, of)
        torch.cuda.synchronize()
        assert eg.engram_last_error() == 0
        assert torch.equal(h.view(torch.int16), ref.view(torch.int16)), f"call {k}"
        stats.append(st.cpu().numpy().copy())
    U, hits, staged, over = stats[0]
    assert hits == 0 and staged == U and 0 <= over <= U
    U1, hits1, staged1, over1 = stats[1]
    assert U1 == U and hits1 + staged1 == U1
    if slots >= 1 << 20:
        assert hits1 >= 0.9 * U1  # the repeated batch comes from the cache
    else:
        assert over1 >= U1 - slots  # at most one row per slot and call
    assert stats[2][1] + stats[2][2] == stats[2][0]


def test_cached_capacity_overflow_leaves_h(eg):
    w = Workload(CFG, host_tables=True)
    cache = eg.engram_host_cache_new(w.c, 1 << 10, 100)
    h0, h = w.fresh_h(), w.fresh_h()
    eg.engram_forward_host_cached(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, cache, 1 << 10, 100,
                                  stamp=1, side_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 4  # ENGRAM_ECAPACITY
    assert torch.equal(h.view(torch.int16), h0.view(torch.int16))


def test_cached_call_in_cuda_graph(eg):
    """A call captured in a CUDA graph replays its stamp.  The first replay
    (a newer stamp than the eager call before it) is served from the rows
    that call cached; the second finds every slot already claimed at its own
    stamp and stages every row into the overflow area (no hits).  h equals the
    HBM path's bits after every call."""
    w = Workload(CFG, host_tables=True)
    cap, slots = CFG.tq * 48, 1 << 20
    cache = eg.engram_host_cache_new(w.c, slots, cap)
    dev_t, dev_s = w.tables.cuda(), w.scales.cuda()
    side, s = torch.cuda.Stream(), torch.cuda.Stream()
    ws = torch.empty(eg.engram_forward_host_cached_workspace_bytes(w.c, CFG.tq, cap), dtype=torch.uint8,
                     device="cuda")
    stats = torch.zeros(4, dtype=torch.int64, device="cuda")
    evs = [torch.cuda.Event(), torch.cuda.Event()]

    def call(h, stamp):
        eg.engram_forward_host_cached(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, cache, slots,
                                      cap, stamp=stamp, workspace=ws, stats=stats, stream=s, side_stream=side,
                                      ev_dedup=evs[0], ev_staged=evs[1])

    h, ref = w.fresh_h(), w.fresh_h()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        call(h, 1)
    for _ in range(3):
        eg.engram_forward(w.c, w.tokens, w.seq_offsets, dev_t, dev_s, w.W, w.g, ref)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call(h, 2)
    graph.replay()
    torch.cuda.synchronize()
    st1 = stats.cpu().numpy().copy()
    graph.replay()
    torch.cuda.synchronize()
    st2 = stats.cpu().numpy().copy()
    assert eg.engram_last_error() == 0
    assert torch.equal(h.view(torch.int16), ref.view(torch.int16))
    U = st1[0]
    assert st1[1] >= 0.9 * U and st1[1] + st1[2] == U
    assert st2[0] == U and st2[1] == 0 and st2[2] == U and st2[3] == U
