"""The host-table path: dedup, staging from pinned host memory, and its
output against the HBM path (bit-identical) and the oracle (needs a GB300)."""

import numpy as np
import pytest
import torch

from synth.configs import CONFIGS
from workload import Workload, check_h, sample_queries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


SMALL_HOST = CONFIGS["host"].with_(seq_lens=(700, 555), R=1 << 15, seed=9)


def _unique_ref(idx, R):
    flat = (np.arange(48)[None, :] * R + idx).reshape(-1)
    return np.unique(flat)


def test_dedup_matches_brute_force(eg):
    w = Workload(SMALL_HOST, tables=False)
    cfg = w.cfg
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    cap = cfg.tq * 48
    unique, idx_staged, n_unique = eg.engram_dedup(w.c, idx, cap)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    ref_idx = w.ref_idx_all()
    ref = _unique_ref(ref_idx, cfg.R)
    U = int(n_unique.item())
    assert U == len(ref)
    assert np.array_equal(unique[:U].cpu().numpy(), ref)  # sorted by (table, row)
    # every query's slot points back at its own (table, row)
    back = unique[idx_staged.long()].cpu().numpy()
    assert np.array_equal(back, np.arange(48)[None, :] * cfg.R + ref_idx)


def test_dedup_capacity_overflow_is_reported(eg):
    w = Workload(SMALL_HOST, tables=False)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    unique, idx_staged, n_unique = eg.engram_dedup(w.c, idx, 100)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 4
    assert int(n_unique.item()) > 100
    assert bool((idx_staged == -1).all())  # no query points at a slot


def test_capacity_overflow_stages_nothing_and_leaves_h(eg):
    """More distinct rows than the staging capacity: ENGRAM_ECAPACITY, the
    stage copies nothing (staging buffers keep their contents), and the
    host-table forward leaves h bit for bit as it was."""
    w = Workload(SMALL_HOST, host_tables=True)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    cap = 100
    unique, idx_staged, n_unique = eg.engram_dedup(w.c, idx, cap)
    rows = torch.full((cap, 256), 0xA5, dtype=torch.uint8, device="cuda")
    scs = torch.full((cap,), -3.0, dtype=torch.float32, device="cuda")
    eg.engram_stage(w.c, w.tables, w.scales, unique, n_unique, cap, rows, scs)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 4
    assert bool((rows == 0xA5).all()) and bool((scs == -3.0).all())
    h0 = w.fresh_h()
    h = w.fresh_h()
    eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, capacity=cap,
                           side_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 4
    assert torch.equal(h.view(torch.int16), h0.view(torch.int16))


def test_stage_copies_rows_byte_exact(eg):
    w = Workload(SMALL_HOST, host_tables=True)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    cap = w.cfg.tq * 48
    unique, idx_staged, n_unique = eg.engram_dedup(w.c, idx, cap)
    rows, scales = eg.engram_stage(w.c, w.tables, w.scales, unique, n_unique, cap)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    U = int(n_unique.item())
    u = unique[:U].cpu()
    assert torch.equal(rows[:U].cpu(), w.tables.view(-1, 256)[u])
    assert torch.equal(scales[:U].cpu(), w.scales.view(-1)[u])


def test_host_path_bit_identical_to_hbm_path(eg):
    """Same tables in pinned host memory and in HBM: the host-table forward
    gives the same h bits as the HBM forward (the host-table mode is
    documented as bitwise identical), and both match the oracle."""
    w = Workload(SMALL_HOST, host_tables=True)
    cfg = w.cfg
    h_host = w.fresh_h()
    side = torch.cuda.Stream()
    n_unique = eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h_host,
                                      capacity=cfg.tq * 48, side_stream=side)
    dev_tables = w.tables.cuda()
    dev_scales = w.scales.cuda()
    h_hbm = w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, dev_tables, dev_scales, w.W, w.g, h_hbm)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_host.view(torch.int16), h_hbm.view(torch.int16))
    assert int(n_unique.item()) == len(_unique_ref(w.ref_idx_all(), cfg.R))
    q = sample_queries(cfg, w.offs, 200)
    _, _, _, ref_h, _ = w.ref_for(q)
    check_h(h_host[torch.from_numpy(q).cuda()], ref_h)


def test_host_tables_with_scales_in_hbm(eg):
    """Host tables with the fp32 scale array in device memory (read through
    its unified address): the same h bits as with pinned host scales."""
    w = Workload(SMALL_HOST, host_tables=True)
    cfg = w.cfg
    side = torch.cuda.Stream()
    h_pinned, h_dev = w.fresh_h(), w.fresh_h()
    eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h_pinned,
                           capacity=cfg.tq * 48, side_stream=side)
    eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, w.tables, w.scales.cuda(), w.W, w.g, h_dev,
                           capacity=cfg.tq * 48, side_stream=side)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_pinned.view(torch.int16), h_dev.view(torch.int16))


@pytest.mark.parametrize("cfg", [CONFIGS["decode"].with_(R=1 << 15, seed=12), SMALL_HOST],
                         ids=["decode_64", "two_seqs_1255"])
def test_forward_reads_pinned_host_tables_in_place(eg, cfg):
    """engram_forward with the tables (and scales) in pinned host memory reads
    the rows in place over unified addressing: the same h bits as with the
    tables in HBM, scales pinned or in HBM."""
    w = Workload(cfg, host_tables=True)
    h_host, h_host_dsc, h_hbm = w.fresh_h(), w.fresh_h(), w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h_host, last_n=cfg.last_n)
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales.cuda(), w.W, w.g, h_host_dsc,
                      last_n=cfg.last_n)
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables.cuda(), w.scales.cuda(), w.W, w.g, h_hbm,
                      last_n=cfg.last_n)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_host.view(torch.int16), h_hbm.view(torch.int16))
    assert torch.equal(h_host_dsc.view(torch.int16), h_hbm.view(torch.int16))


def test_host_path_record_layout(eg):
    """Host tables as 272-byte records (scale inside the row): same h bits as
    the HBM path with separate scales."""
    a = Workload(SMALL_HOST)
    b = Workload(SMALL_HOST, host_tables=True, layout="record")
    ha, hb = a.fresh_h(), b.fresh_h()
    eg.engram_forward(a.c, a.tokens, a.seq_offsets, a.tables, a.scales, a.W, a.g, ha)
    eg.engram_forward_host(b.c, b.tokens, b.seq_offsets, b.tables, None, b.W, b.g, hb, capacity=b.cfg.tq * 48)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(ha.view(torch.int16), hb.view(torch.int16))


def test_host_path_mx_layout(eg):
    """MXFP8-style rows in pinned host memory: staged whole (byte-exact), the
    staged gather equals the HBM gather, and the host-table forward gives the
    HBM forward's bits and matches the oracle."""
    a = Workload(SMALL_HOST, layout="mx")
    b = Workload(SMALL_HOST, host_tables=True, layout="mx")
    cap = b.cfg.tq * 48
    idx = eg.engram_hash(b.c, b.tokens, b.seq_offsets)
    unique, idx_staged, n_unique = eg.engram_dedup(b.c, idx, cap)
    rows, sc = eg.engram_stage(b.c, b.tables, None, unique, n_unique, cap)
    assert sc is None and rows.shape == (cap, 272)
    mem_staged = eg.engram_gather_reduce_staged(b.c, rows, None, idx_staged)
    mem_hbm = eg.engram_gather_reduce(a.c, a.tables, None, idx)
    ha, hb = a.fresh_h(), b.fresh_h()
    eg.engram_forward(a.c, a.tokens, a.seq_offsets, a.tables, None, a.W, a.g, ha)
    eg.engram_forward_host(b.c, b.tokens, b.seq_offsets, b.tables, None, b.W, b.g, hb, capacity=cap)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    U = int(n_unique.item())
    assert torch.equal(rows[:U].cpu(), b.tables.view(-1, 272)[unique[:U].cpu()])
    assert torch.equal(mem_staged, mem_hbm)
    assert torch.equal(ha.view(torch.int16), hb.view(torch.int16))
    q = sample_queries(b.cfg, b.offs, 200)
    _, _, _, ref_h, _ = b.ref_for(q)
    check_h(hb[torch.from_numpy(q).cuda()], ref_h)


@pytest.mark.parametrize("chunk", [128, 384, 1000, 4096])
def test_host_pipelined_bit_identical_to_hbm(eg, chunk):
    """The chunked, pipelined host path gives the HBM forward's h bits, and
    each chunk stages exactly its own distinct rows."""
    w = Workload(SMALL_HOST, host_tables=True)
    cfg = w.cfg
    h_pipe = w.fresh_h()
    n_unique = eg.engram_forward_host_pipelined(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h_pipe,
                                                chunk=chunk)
    dev_tables, dev_scales = w.tables.cuda(), w.scales.cuda()
    h_hbm = w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, dev_tables, dev_scales, w.W, w.g, h_hbm)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_pipe.view(torch.int16), h_hbm.view(torch.int16))
    ref_idx = w.ref_idx_all()
    c = min(chunk, cfg.tq)
    want = [len(_unique_ref(ref_idx[q0:q0 + c], cfg.R)) for q0 in range(0, cfg.tq, c)]
    assert n_unique.cpu().tolist() == want


def test_host_pipelined_many_tiles_and_mx(eg):
    """83 tiles in chunks of 16 tiles: every chunk's projection splits d as for
    the whole batch (the many-tile kernel), so h keeps the HBM path's bits; and
    MXFP8-style rows through the same pipeline."""
    cfg = CONFIGS["host"].with_(seq_lens=(6000, 4500), R=1 << 16, seed=12)
    w = Workload(cfg, host_tables=True)
    h_pipe, h_hbm = w.fresh_h(), w.fresh_h()
    eg.engram_forward_host_pipelined(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h_pipe, chunk=2048)
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables.cuda(), w.scales.cuda(), w.W, w.g, h_hbm)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_pipe.view(torch.int16), h_hbm.view(torch.int16))
    del w
    m = Workload(SMALL_HOST, host_tables=True, layout="mx")
    h_pipe, h_hbm = m.fresh_h(), m.fresh_h()
    eg.engram_forward_host_pipelined(m.c, m.tokens, m.seq_offsets, m.tables, None, m.W, m.g, h_pipe, chunk=384)
    eg.engram_forward(m.c, m.tokens, m.seq_offsets, m.tables.cuda(), None, m.W, m.g, h_hbm)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_pipe.view(torch.int16), h_hbm.view(torch.int16))


def test_host_tables_on_huge_pages(eg):
    """Tables in engram_host_alloc memory (pinned, transparent huge pages):
    staged bytes equal the table rows, and the host-table forward gives the
    HBM forward's bits."""
    w = Workload(SMALL_HOST, host_tables=True)
    t = eg.host_tables_empty(tuple(w.tables.shape), torch.uint8)
    s = eg.host_tables_empty(tuple(w.scales.shape), torch.float32)
    assert t.is_pinned() and s.is_pinned() and t.data_ptr() % 4096 == 0
    t.copy_(w.tables)
    s.copy_(w.scales)
    cap = w.cfg.tq * 48
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    unique, idx_staged, n_unique = eg.engram_dedup(w.c, idx, cap)
    rows, scales = eg.engram_stage(w.c, t, s, unique, n_unique, cap)
    h1, h2 = w.fresh_h(), w.fresh_h()
    eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, t, s, w.W, w.g, h1, capacity=cap)
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables.cuda(), w.scales.cuda(), w.W, w.g, h2)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    U = int(n_unique.item())
    u = unique[:U].cpu()
    assert torch.equal(rows[:U].cpu(), w.tables.view(-1, 256)[u])
    assert torch.equal(scales[:U].cpu(), w.scales.view(-1)[u])
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    del t, s


def test_host_path_full_size(eg):
    """The host-table workload at full size (51.5 GB of pinned tables)."""
    cfg = CONFIGS["host"]
    try:
        w = Workload(cfg, host_tables=True)
    except RuntimeError as e:  # pinning 53 GB can fail on a small host
        pytest.skip(f"cannot pin {cfg.table_bytes / 1e9:.1f} GB of host memory: {e}")
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    cap = cfg.tq * 48
    h = w.fresh_h()
    n_unique = eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, capacity=cap)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    ref_idx = w.ref_idx_all()
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert int(n_unique.item()) == len(_unique_ref(ref_idx, cfg.R))
    q = sample_queries(cfg, w.offs, 200)
    _, _, _, ref_h, _ = w.ref_for(q)
    check_h(h[torch.from_numpy(q).cuda()], ref_h)
    del w, h, idx
    torch.cuda.empty_cache()


@pytest.mark.parametrize("form", ["one_batch", "pipelined"])
def test_host_path_in_cuda_graph(eg, form):
    """The host-table path captured in a CUDA graph: the dedup on the main
    stream, the staging on a side stream forked and joined by events, then
    the staged gather and projection.  Each replay gives the bits of the same
    call run eagerly (and a second replay applies the update again)."""
    w = Workload(SMALL_HOST, host_tables=True)
    cfg = w.cfg
    nq, cap, chunk = cfg.tq, cfg.tq * 48, 512
    dev = torch.device("cuda")
    side, s = torch.cuda.Stream(), torch.cuda.Stream()
    if form == "one_batch":
        ws = torch.empty(eg.engram_forward_host_workspace_bytes(w.c, nq, cap), dtype=torch.uint8, device=dev)
        nu = torch.zeros(1, dtype=torch.int64, device=dev)
        evs = [torch.cuda.Event(), torch.cuda.Event()]

        def call(h):
            return eg.engram_forward_host(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h,
                                          capacity=cap, workspace=ws, n_unique=nu, stream=s, side_stream=side,
                                          ev_dedup=evs[0], ev_staged=evs[1])
    else:
        ws = torch.empty(eg.engram_forward_host_pipelined_workspace_bytes(w.c, nq, chunk, chunk * 48),
                         dtype=torch.uint8, device=dev)
        nu = torch.zeros(-(-nq // chunk), dtype=torch.int64, device=dev)
        evs = [torch.cuda.Event() for _ in range(6)]

        def call(h):
            return eg.engram_forward_host_pipelined(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h,
                                                    chunk=chunk, workspace=ws, n_unique=nu, stream=s,
                                                    side_stream=side, events=evs)

    h_eager = w.fresh_h()
    torch.cuda.synchronize()  # h is filled on the current stream
    with torch.cuda.stream(s):
        call(h_eager)
        call(h_eager)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    nu_eager = nu.clone()

    h_graph = w.fresh_h()
    nu.zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call(h_graph)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_graph.view(torch.int16), h_eager.view(torch.int16))
    assert torch.equal(nu, nu_eager)
