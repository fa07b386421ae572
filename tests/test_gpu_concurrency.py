"""Calls on several streams at once (needs a GB300): each call reads only its
own arguments, so batches of different shapes run concurrently on separate
streams, each with its own workspace and h, give the bits of the same calls
run one after another, and the oracle's values."""

import numpy as np
import pytest
import torch

from synth.configs import CONFIGS
from workload import Workload, check_h

pytestmark = pytest.mark.gpu

CASES = {
    # 1 tile: gates beside the gather, then the d-split projection
    "decode": CONFIGS["decode"].with_(R=1 << 16),
    # 9 tiles: the cluster projection
    "prefill": CONFIGS["prefill"].with_(seq_lens=(640, 421), R=1 << 16, seed=6),
    # d = 256, 4 tiles
    "tiny": CONFIGS["tiny"],
}
REPS = 3


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


def _forward(eg, w, h, ws, stream):
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, last_n=w.cfg.last_n,
                      n_query=w.cfg.tq, workspace=ws, stream=stream)


def _split(eg, w, h, X, stream):
    eg.engram_gather_x(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, last_n=w.cfg.last_n, n_query=w.cfg.tq,
                       X=X, stream=stream)
    eg.engram_fuse_x(w.c, X, w.W, w.g, h, stream=stream)


def test_streams_run_concurrently_with_serial_bits(eg):
    ws = {k: Workload(cfg) for k, cfg in CASES.items()}
    work = {k: torch.empty(eg.engram_forward_workspace_bytes(w.c, w.cfg.tq), dtype=torch.uint8, device="cuda")
            for k, w in ws.items()}
    xbuf = {k: torch.empty((w.cfg.tq, 512), dtype=torch.bfloat16, device="cuda") for k, w in ws.items()}

    # one after another on one stream: REPS forward calls per batch (h is
    # updated in place each time), and the split form on a second h
    s0 = torch.cuda.Stream()
    ref_f = {k: w.fresh_h() for k, w in ws.items()}
    ref_s = {k: w.fresh_h() for k, w in ws.items()}
    torch.cuda.synchronize()
    for k, w in ws.items():
        for _ in range(REPS):
            _forward(eg, w, ref_f[k], work[k], s0)
        for _ in range(REPS):
            _split(eg, w, ref_s[k], xbuf[k], s0)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0

    # the same calls, each batch's forward and split form on streams of
    # their own, enqueued round-robin so that they overlap on the device
    work2 = {k: torch.empty_like(v) for k, v in work.items()}
    xbuf2 = {k: torch.empty_like(v) for k, v in xbuf.items()}
    h_f = {k: w.fresh_h() for k, w in ws.items()}
    h_s = {k: w.fresh_h() for k, w in ws.items()}
    streams = {(k, form): torch.cuda.Stream() for k in ws for form in ("f", "s")}
    torch.cuda.synchronize()
    for _ in range(REPS):
        for k, w in ws.items():
            _forward(eg, w, h_f[k], work2[k], streams[(k, "f")])
            _split(eg, w, h_s[k], xbuf2[k], streams[(k, "s")])
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0

    for k, w in ws.items():
        assert torch.equal(h_f[k].view(torch.int16), ref_f[k].view(torch.int16)), k
        assert torch.equal(h_s[k].view(torch.int16), ref_s[k].view(torch.int16)), k
        assert torch.equal(h_f[k].view(torch.int16), h_s[k].view(torch.int16)), k

    # and the first of the REPS calls against the oracle, on a fresh h
    for k, w in ws.items():
        h1 = w.fresh_h()  # filled on the current stream: finish before another stream reads it
        torch.cuda.synchronize()
        _forward(eg, w, h1, work[k], streams[(k, "f")])
        torch.cuda.synchronize()
        _, _, _, ref_h, _ = w.ref_for(np.arange(w.cfg.tq))
        check_h(h1, ref_h)
