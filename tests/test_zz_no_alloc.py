"""engram_forward_no_workspace: the entry point for callers that cannot
allocate device memory (for example code inside an engine whose allocator
owns all device memory).  Its scratch is the library's own device array; the
test checks it against engram_forward on two calls in a row, the second with
a different and smaller batch, so stale scratch contents from the first call
would show.  Collected last on purpose (file name)."""

import ctypes

import numpy as np
import pytest
import torch

from synth.configs import CONFIGS
from workload import Workload, check_h

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


def _call_no_workspace(eg, w, h):
    """Through the C ABI directly (ctypes), on the current stream."""
    lib = eg.lib()
    cfg = w.cfg
    nq = cfg.tq
    st = lib.engram_forward_no_workspace(
        ctypes.byref(w.c), ctypes.c_void_p(w.tokens.data_ptr()), ctypes.c_void_p(w.seq_offsets.data_ptr()),
        cfg.n_seqs, cfg.last_n, nq, ctypes.c_void_p(w.tables.data_ptr()), ctypes.c_void_p(w.scales.data_ptr()),
        ctypes.c_void_p(w.W.data_ptr()), ctypes.c_void_p(w.g.data_ptr()), ctypes.c_void_p(h.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_no_workspace_matches_forward_on_two_calls(eg):
    first = Workload(CONFIGS["prefill"].with_(seq_lens=(2000, 1071), R=1 << 16, seed=11))  # 3,071 queries, 24 tiles
    second = Workload(CONFIGS["decode"].with_(R=1 << 16, seed=12))  # 64 queries (last of each sequence)
    for w in (first, second):
        ref = w.fresh_h()
        eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, ref, last_n=w.cfg.last_n)
        got = w.fresh_h()
        assert _call_no_workspace(eg, w, got) == 0
        torch.cuda.synchronize()
        assert eg.engram_last_error() == 0
        # same tolerance as the other parity tests, with engram_forward's h as the reference
        check_h(got, ref.view(torch.int16).cpu().numpy().view(np.uint16))
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))  # same kernels, same bits


def test_no_workspace_rejects_too_many_queries(eg):
    cfg = CONFIGS["tiny"].with_(seq_lens=(eg.NO_WORKSPACE_MAX_QUERY + 1,), R=1 << 10, seed=13)
    w = Workload(cfg)
    h = w.fresh_h()
    before = h.clone()
    assert _call_no_workspace(eg, w, h) == 6  # ENGRAM_ENOMEM, nothing enqueued
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), before.view(torch.int16))
