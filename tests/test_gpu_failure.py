"""Failure detection on the GPU without a fault: a bounded device wait that
nothing satisfies runs out, the kernel reports ENGRAM_ETIMEOUT through the
sticky error word and returns, and the device keeps working (needs a GB300)."""

import time

import numpy as np
import pytest
import torch

from synth.configs import CONFIGS
from workload import Workload, check_h

pytestmark = pytest.mark.gpu

ETIMEOUT = 5


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


def test_bounded_wait_runs_out_and_reports_timeout(eg):
    eg.engram_last_error()  # start from a clear word
    t0 = time.perf_counter()
    eg.engram_wait_selftest(50_000_000)  # 50 ms of device time
    status = eg.engram_last_error()  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == ETIMEOUT
    assert 0.04 < elapsed < 5.0  # it waited about its limit, then gave up
    assert eg.engram_last_error() == 0  # reading cleared the word


def test_device_stays_usable_after_a_timeout(eg):
    eg.engram_wait_selftest(1_000_000)
    assert eg.engram_last_error() == ETIMEOUT
    w = Workload(CONFIGS["tiny"])
    h = w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, last_n=w.cfg.last_n)
    assert eg.engram_last_error() == 0
    _, _, _, ref_h, _ = w.ref_for(np.arange(w.cfg.tq))
    check_h(h, ref_h)
