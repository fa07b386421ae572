"""CUDA path vs the CPU oracle, through the C ABI (needs a GB300)."""

import numpy as np
import pytest
import torch

import oracle
from synth import device as sd
from synth import host
from synth.configs import CONFIGS
from workload import Workload, bf16_to_f64, check_h, check_mem, sample_queries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()  # fail loudly when the CUDA library is missing
    return eg


SMALL = {
    "tiny": CONFIGS["tiny"],
    # ragged sequences (lengths 1 and 2 exercise the pad), prime R
    "ragged_prime": CONFIGS["tiny"].with_(seq_lens=(300, 1, 2, 140, 77), R=4093, seed=5),
    # d = 4096, several 128-token tiles plus a ragged tail, repeated spans
    "prefill_small": CONFIGS["prefill"].with_(seq_lens=(640, 421), R=1 << 16, seed=6),
    # decode: 64 sequences of 4 tokens, only the last one queried
    "decode_small": CONFIGS["decode"].with_(R=1 << 16),
    # 37 queries (the d-split projection's load boxes round up to 40 rows),
    # sequences of 1 to 4 tokens, so the n-gram windows reach the pad
    "decode_ragged": CONFIGS["decode"].with_(R=1 << 16, seq_lens=tuple(1 + (i % 4) for i in range(37)), seed=11),
    # d = 512 (two 256-column chunks)
    "d512": CONFIGS["tiny"].with_(d=512, seq_lens=(333,), seed=7),
    # d = 1280: five chunks, so clusters of 5 CTAs of one chunk each; 9 tiles
    # with a ragged tail (the forward pass takes the cluster kernel)
    "d1280": CONFIGS["tiny"].with_(d=1280, seq_lens=(1000, 77), seed=12),
    # d = 7168: 28 chunks, clusters of 7 CTAs of four chunks; 3 tiles
    "d7168": CONFIGS["tiny"].with_(d=7168, seq_lens=(300, 29), seed=13),
    # d = 7168 in one tile: the d-split projection on 112 CTAs, gates summed
    # in the 7 x 4 chunk order
    "d7168_one_tile": CONFIGS["tiny"].with_(d=7168, seq_lens=(90,), seed=14),
    # the widest d the projection takes: clusters of 8 CTAs of 16 chunks
    "d32768": CONFIGS["tiny"].with_(d=32768, seq_lens=(150,), seed=15),
}


def _clear(eg):
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0


@pytest.mark.parametrize("name", list(SMALL))
def test_hash_bit_exact_small(eg, name):
    w = Workload(SMALL[name], tables=False)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=w.cfg.last_n)
    _clear(eg)
    assert np.array_equal(idx.cpu().numpy(), w.ref_idx_all())


@pytest.mark.parametrize("name", list(SMALL))
def test_gather_reduce_small(eg, name):
    w = Workload(SMALL[name])
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=w.cfg.last_n)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    _clear(eg)
    q = np.arange(w.cfg.tq)
    ridx, rmem, bound, _, _ = w.ref_for(q)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    check_mem(mem.cpu().numpy(), rmem, bound)


@pytest.mark.parametrize("name", list(SMALL))
def test_fuse_small(eg, name):
    """engram_fuse alone: the oracle's mem (as fp32) in, h compared with the
    oracle's fuse of the same fp32 mem."""
    w = Workload(SMALL[name], tables=False)
    cfg = w.cfg
    rng = np.random.default_rng(cfg.seed)
    mem32 = (rng.standard_normal((cfg.tq, 512)) * 6.0).astype(np.float32)
    h = w.fresh_h()
    eg.engram_fuse(w.c, torch.from_numpy(mem32).cuda(), w.W, w.g, h)
    _clear(eg)
    h0 = host.h_rows(cfg.seed, cfg.d, np.arange(cfg.tq))
    ref, _ = oracle.fuse(mem32.astype(np.float64), host.w_out(cfg.seed, cfg.d), host.g_vec(cfg.seed, cfg.d), h0,
                         cfg.rms_eps)
    check_h(h, ref)


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small(eg, name):
    """The one-call path against the oracle on every query token, and against
    the three separate calls (same kernels' arithmetic: bit-identical)."""
    w = Workload(SMALL[name])
    h = w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, last_n=w.cfg.last_n)
    h2 = w.fresh_h()
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=w.cfg.last_n)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    eg.engram_fuse(w.c, mem, w.W, w.g, h2)
    _clear(eg)
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    _, _, _, ref_h, _ = w.ref_for(np.arange(w.cfg.tq))
    check_h(h, ref_h)


@pytest.mark.parametrize("name", ["tiny", "prefill_small", "decode_small", "decode_ragged"])
def test_split_halves_equal_forward(eg, name):
    """engram_gather_x then engram_fuse_x gives engram_forward's bits, and X
    is bf16 of the fp32 module sums of engram_gather_reduce."""
    w = Workload(SMALL[name])
    X = eg.engram_gather_x(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, last_n=w.cfg.last_n)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=w.cfg.last_n)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    h1, h2 = w.fresh_h(), w.fresh_h()
    eg.engram_fuse_x(w.c, X, w.W, w.g, h1)
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h2, last_n=w.cfg.last_n)
    _clear(eg)
    assert torch.equal(X.view(torch.int16), mem.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "ragged_prime", "prefill_small", "decode_small"])
def test_record_layout_same_bits(eg, name):
    """Rows that carry their scale (272-byte records) give the same mem, X and
    h bits as the separate-scales layout, and match the oracle."""
    a = Workload(SMALL[name])
    b = Workload(SMALL[name], layout="record")
    assert torch.equal(b.tables[:, :, :256], a.tables)
    assert torch.equal(b.tables[:, :, 256:260].contiguous().view(torch.float32).squeeze(-1), a.scales)
    ia = eg.engram_hash(a.c, a.tokens, a.seq_offsets, last_n=a.cfg.last_n)
    ma = eg.engram_gather_reduce(a.c, a.tables, a.scales, ia)
    mb = eg.engram_gather_reduce(b.c, b.tables, None, ia)
    ha, hb = a.fresh_h(), b.fresh_h()
    eg.engram_forward(a.c, a.tokens, a.seq_offsets, a.tables, a.scales, a.W, a.g, ha, last_n=a.cfg.last_n)
    eg.engram_forward(b.c, b.tokens, b.seq_offsets, b.tables, None, b.W, b.g, hb, last_n=b.cfg.last_n)
    _clear(eg)
    assert torch.equal(ma, mb)
    assert torch.equal(ha.view(torch.int16), hb.view(torch.int16))
    q = np.arange(a.cfg.tq)
    _, rmem, bound, rh, _ = a.ref_for(q)
    check_mem(mb.cpu().numpy(), rmem, bound)
    check_h(hb, rh)


@pytest.mark.parametrize("name", ["tiny", "ragged_prime", "prefill_small", "decode_small", "d512"])
def test_mx_layout_small(eg, name):
    """MXFP8-style rows (256 e4m3 codes + eight E8M0 block scales): mem and h
    against the oracle on every query token; the split halves and the
    separate calls give engram_forward's bits."""
    w = Workload(SMALL[name], layout="mx")
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=w.cfg.last_n)
    mem = eg.engram_gather_reduce(w.c, w.tables, None, idx)
    X = eg.engram_gather_x(w.c, w.tokens, w.seq_offsets, w.tables, None, last_n=w.cfg.last_n)
    h, h1, h2 = w.fresh_h(), w.fresh_h(), w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, None, w.W, w.g, h, last_n=w.cfg.last_n)
    eg.engram_fuse_x(w.c, X, w.W, w.g, h1)
    eg.engram_fuse(w.c, mem, w.W, w.g, h2)
    _clear(eg)
    assert torch.equal(X.view(torch.int16), mem.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(h.view(torch.int16), h1.view(torch.int16))
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    ridx, rmem, bound, rh, _ = w.ref_for(np.arange(w.cfg.tq))
    assert np.array_equal(idx.cpu().numpy(), ridx)
    check_mem(mem.cpu().numpy(), rmem, bound)
    check_h(h, rh)


def test_mx_block_scales_special_values(eg):
    """Every code e4m3 1.0 and, per 32-column block, the E8M0 bytes 124..129,
    0 (the subnormal 2^-127) and 255 (NaN): each mem entry is exactly
    24 * 2^(E - 127), NaN in the last block."""
    w = Workload(SMALL["tiny"], layout="mx")
    w.tables[:, :, :256] = 0x38
    e = np.array([124, 125, 126, 127, 128, 129, 0, 255], dtype=np.uint8)
    w.tables[:, :, 256:264] = torch.from_numpy(e).cuda()
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    mem = eg.engram_gather_reduce(w.c, w.tables, None, idx)
    _clear(eg)
    want = np.repeat([24.0 * oracle.e8m0_value(int(x)) for x in e], 32)
    want = np.concatenate([want, want])
    got = mem.cpu().numpy().astype(np.float64)
    assert np.array_equal(got[:, :224], np.broadcast_to(want[:224], (len(got), 224)))
    assert np.array_equal(got[:, 256:480], np.broadcast_to(want[256:480], (len(got), 224)))
    assert np.all(np.isnan(got[:, 224:256])) and np.all(np.isnan(got[:, 480:]))
    assert want[192] == 24.0 * 2.0 ** -127 and got[0, 192] > 0  # not flushed to zero
    # the oracle's own MX reduction gives the same values on one token's rows
    rows = np.full((1, 48, 256), 0x38, np.uint8)
    ref = oracle.gather_reduce_mx_rows(rows, np.broadcast_to(e, (1, 48, 8)))
    assert np.array_equal(ref[0, :224], want[:224])


def test_mx_generator_twin_matches_host(eg):
    """The device-filled E8M0 block-scale bytes equal the host draws."""
    cfg = SMALL["ragged_prime"]
    w = Workload(cfg, layout="mx")
    rng = np.random.default_rng(2)
    j = rng.integers(0, 48, 300)
    r = rng.integers(0, cfg.R, 300)
    got = w.tables[torch.from_numpy(j).cuda(), torch.from_numpy(r).cuda()].cpu().numpy()
    assert np.array_equal(got[:, :256], host.table_rows(cfg.seed, j, r))
    assert np.array_equal(got[:, 256:264], host.mx_scales(cfg.seed, j, r))
    assert np.all(got[:, 264:] == 0)


def test_many_tiles_forward(eg):
    """83 tiles of 128 tokens at d = 4096 (the many-tile projection kernel):
    engram_forward and engram_gather_x + engram_fuse_x give the bits of
    hash + gather + fuse from fp32 mem, and h matches the oracle on a seeded
    sample plus every sequence start and the last token."""
    cfg = CONFIGS["prefill"].with_(seq_lens=(6000, 4500), R=1 << 16, seed=8)
    w = Workload(cfg)
    h1, h2, h3 = w.fresh_h(), w.fresh_h(), w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h1)
    X = eg.engram_gather_x(w.c, w.tokens, w.seq_offsets, w.tables, w.scales)
    eg.engram_fuse_x(w.c, X, w.W, w.g, h2)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    eg.engram_fuse(w.c, mem, w.W, w.g, h3)
    _clear(eg)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(h1.view(torch.int16), h3.view(torch.int16))
    q = sample_queries(cfg, w.offs, 256)
    _, _, _, rh, _ = w.ref_for(q)
    check_h(h1[torch.from_numpy(q).cuda()], rh)


@pytest.mark.parametrize("name", ["decode_small", "decode_ragged", "tiny"])
def test_forward_in_cuda_graph(eg, name):
    """engram_forward captured once in a CUDA graph and replayed gives the bits
    of the same call launched eagerly (no host sync or allocation inside)."""
    w = Workload(SMALL[name])
    nq = w.cfg.tq
    ws = torch.empty(max(eg.engram_forward_workspace_bytes(w.c, nq), 1), dtype=torch.uint8, device="cuda")
    h1, h2 = w.fresh_h(), w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h1, last_n=w.cfg.last_n,
                      n_query=nq, workspace=ws)
    h_warm = w.fresh_h()  # first-call set-up (function attributes, occupancy) before capture
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h_warm, last_n=w.cfg.last_n,
                      n_query=nq, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h2, last_n=w.cfg.last_n,
                          n_query=nq, workspace=ws)
    graph.replay()
    _clear(eg)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    graph.replay()  # a second replay applies the update again
    torch.cuda.synchronize()
    assert not torch.equal(h1.view(torch.int16), h2.view(torch.int16))


@pytest.mark.parametrize("name", ["decode_small", "prefill_small", "d7168"])
def test_dependent_forward_steps_in_one_graph(eg, name):
    """Three engram_forward calls on the same h captured in one CUDA graph (each
    step reads the h the previous one wrote, with no host launch gap between
    them) give the bits of the same three calls made eagerly."""
    w = Workload(SMALL[name])
    nq = w.cfg.tq
    ws = torch.empty(max(eg.engram_forward_workspace_bytes(w.c, nq), 1), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def steps(h):
        for _ in range(3):
            eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, last_n=w.cfg.last_n,
                              n_query=nq, workspace=ws, stream=s)

    h_eager, h_graph = w.fresh_h(), w.fresh_h()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        steps(h_eager)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        steps(h_graph)
    graph.replay()
    _clear(eg)
    assert torch.equal(h_eager.view(torch.int16), h_graph.view(torch.int16))


@pytest.mark.parametrize("n", [1, 127, 128, 129, 255, 256, 257, 1153])
def test_forward_at_tile_boundaries(eg, n):
    """Batches of 1 token, one tile less / exactly / one more, two tiles and
    three (d = 4096: the d-split kernel up to two tiles, the cluster kernel
    from three) and a tail of one token after nine tiles: engram_forward
    against the oracle on every token, and equal to the split form's bits."""
    w = Workload(CONFIGS["prefill"].with_(seq_lens=(n,), R=1 << 16, seed=20 + n))
    h1, h2 = w.fresh_h(), w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h1)
    X = eg.engram_gather_x(w.c, w.tokens, w.seq_offsets, w.tables, w.scales)
    eg.engram_fuse_x(w.c, X, w.W, w.g, h2)
    _clear(eg)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    _, _, _, ref_h, _ = w.ref_for(np.arange(n))
    check_h(h1, ref_h)


def test_generator_twin_rows_match_host(eg):
    """The device-filled tables/scales/h equal the host draws bit for bit."""
    cfg = SMALL["ragged_prime"]
    w = Workload(cfg)
    rng = np.random.default_rng(1)
    j = rng.integers(0, 48, 200)
    r = rng.integers(0, cfg.R, 200)
    got = w.tables[torch.from_numpy(j).cuda(), torch.from_numpy(r).cuda()].cpu().numpy()
    assert np.array_equal(got, host.table_rows(cfg.seed, j, r))
    gs = w.scales[torch.from_numpy(j).cuda(), torch.from_numpy(r).cuda()].cpu().numpy()
    assert np.array_equal(gs, host.scales(cfg.seed, j, r))
    h = w.fresh_h()
    assert np.array_equal(h.view(torch.int16).cpu().numpy().view(np.uint16), host.h_rows(cfg.seed, cfg.d, np.arange(cfg.tq)))
    assert np.array_equal(w.W.view(torch.int16).cpu().numpy().view(np.uint16), host.w_out(cfg.seed, cfg.d))


def test_idx_independent_of_tables(eg):
    """Row addresses depend on token ids only: the hash takes no table, and
    overwriting every table leaves the gathered rows' addresses unchanged."""
    w = Workload(SMALL["tiny"])
    idx1 = eg.engram_hash(w.c, w.tokens, w.seq_offsets).clone()
    w.tables.random_(0, 127)
    idx2 = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    _clear(eg)
    assert torch.equal(idx1, idx2)


def test_special_cases_on_gpu(eg):
    """All rows = e4m3 1.0 with unit scales: every mem entry is exactly 24;
    g = 0 gives gate 1/2; W_out = 0 leaves h bit-unchanged."""
    w = Workload(SMALL["tiny"])
    w.tables.fill_(0x38)
    w.scales.fill_(1.0)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    h = w.fresh_h()
    h0 = h.clone()
    eg.engram_fuse(w.c, mem, torch.zeros_like(w.W), w.g, h)
    _clear(eg)
    assert torch.all(mem == 24.0)
    assert torch.equal(h.view(torch.int16), h0.view(torch.int16))
    # g = 0: gate = 1/2 exactly, so h = bf16(h + y/2) with y = 24 * colsum(W)
    h = w.fresh_h()
    eg.engram_fuse(w.c, mem, w.W, torch.zeros_like(w.g), h)
    _clear(eg)
    cfg = w.cfg
    ref, gate = oracle.fuse(np.full((cfg.tq, 512), 24.0), host.w_out(cfg.seed, cfg.d), np.zeros(cfg.d, np.uint16),
                            host.h_rows(cfg.seed, cfg.d, np.arange(cfg.tq)))
    assert np.all(gate == 0.5)
    check_h(h, ref)


def test_empty_and_invalid_arguments(eg):
    w = Workload(SMALL["tiny"])
    e = torch.empty((0, 48), dtype=torch.int64, device="cuda")
    out = eg.engram_gather_reduce(w.c, w.tables, w.scales, e)
    assert out.shape == (0, 512)
    h = torch.empty((0, w.cfg.d), dtype=torch.bfloat16, device="cuda")
    eg.engram_fuse(w.c, torch.empty((0, 512), device="cuda"), w.W, w.g, h)
    bad = eg.make_config(w.cfg.V, w.cfg.R, 200, w.seeds)  # d not a multiple of 256
    hb = torch.zeros((4, 200), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(eg.EngramError) as ex:
        eg.engram_fuse(bad, torch.zeros((4, 512), device="cuda"), torch.zeros((512, 200), dtype=torch.bfloat16,
                       device="cuda"), torch.zeros(200, dtype=torch.bfloat16, device="cuda"), hb)
    assert ex.value.status == 1
    with pytest.raises(eg.EngramError) as ex:  # misaligned tables
        eg.engram_gather_reduce(w.c, w.tables.view(-1)[1:1 + 48 * 10 * 256].view(48, 10, 256), w.scales,
                                torch.zeros((1, 48), dtype=torch.int64, device="cuda"))
    assert ex.value.status == 1
    with pytest.raises(eg.EngramError) as ex:  # workspace too small
        eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, w.fresh_h(),
                          workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert ex.value.status == 6
    with pytest.raises(eg.EngramError):  # last_n > 0 with the wrong query count
        eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=2, n_query=5)
    _clear(eg)


def test_device_range_errors_are_reported(eg):
    """Conditions only the device sees set the sticky error word (no trap)."""
    w = Workload(SMALL["tiny"])
    tok = w.tokens.clone()
    tok[5] = w.cfg.V  # the pad id is not a valid token
    eg.engram_hash(w.c, tok, w.seq_offsets)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 3
    assert eg.engram_last_error() == 0  # cleared
    idx = torch.full((3, 48), w.cfg.R, dtype=torch.int64, device="cuda")  # row index == R
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 3
    assert torch.all(mem == 0)  # out-of-range rows read nothing
    offs = torch.tensor([0, 1, 512], dtype=torch.int64, device="cuda")  # a 1-token sequence with last_n = 2
    eg.engram_hash(w.c, w.tokens, offs, last_n=2)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 3


# ------------------------------------------------------------- full sizes ---

FULL = ["tiny", "decode", "prefill", "large"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_forward(eg, name):
    """The workloads at their full sizes, in the launch configuration the
    benchmark times (engram_forward on one stream): idx on every query token,
    mem and h on a seeded sample plus every sequence start and the last token."""
    cfg = CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    need = cfg.table_bytes * 1.02 + cfg.tq * (cfg.d * 2 * 2 + 512 * 8 + 48 * 8) + (1 << 30)
    if free < need:
        pytest.skip(f"needs {need / 1e9:.1f} GB of device memory, {free / 1e9:.1f} GB free")
    w = Workload(cfg)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=cfg.last_n)
    _clear(eg)
    assert np.array_equal(idx.cpu().numpy(), w.ref_idx_all())
    q = sample_queries(cfg, w.offs, 256 if cfg.d > 256 else cfg.tq)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    h = w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, last_n=cfg.last_n)
    _clear(eg)
    qt = torch.from_numpy(q).cuda()
    _, rmem, bound, rh, _ = w.ref_for(q)
    check_mem(mem[qt].cpu().numpy(), rmem, bound)
    check_h(h[qt], rh)
    del w, idx, mem, h
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["large", "prefill"])
def test_every_token_parallel_oracle(eg, name):
    """The large workload (131,072 query tokens, uniform ids, R = 8,388,608) and
    the prefill workload (8 x 32,768 tokens, Zipf ids with repeated spans,
    R = 2,097,152), d = 4096, at full size through engram_forward, the call the
    benchmark times: mem and h on EVERY query token against the oracle, which
    runs over all host cores in spawned worker processes from the generators'
    host twins."""
    import oracle_pool

    cfg = CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    need = cfg.table_bytes * 1.02 + cfg.tq * (cfg.d * 2 * 2 + 512 * 8 + 48 * 8) + (1 << 30)
    if free < need:
        pytest.skip(f"needs {need / 1e9:.1f} GB of device memory, {free / 1e9:.1f} GB free")
    w = Workload(cfg)
    idx = eg.engram_hash(w.c, w.tokens, w.seq_offsets, last_n=cfg.last_n)
    mem = eg.engram_gather_reduce(w.c, w.tables, w.scales, idx)
    h = w.fresh_h()
    eg.engram_forward(w.c, w.tokens, w.seq_offsets, w.tables, w.scales, w.W, w.g, h, last_n=cfg.last_n)
    _clear(eg)
    gm = mem.cpu().numpy()
    gh = h.view(torch.int16).cpu().numpy().view(np.uint16)
    args = (cfg, w.seeds, w.tok, w.offs, w.qpos)
    del w, idx, mem, h
    torch.cuda.empty_cache()
    s = oracle_pool.check_all_tokens(*args, gm, gh)
    print(f"\nevery-token oracle check: {s['tokens']} tokens in {s['seconds']:.1f} s on {s['procs']} processes "
          f"({s['tokens'] / s['seconds']:.0f} tokens/s); worst mem {s['mem_worst']:.2e} x sum|term|, "
          f"worst h {s['h_worst']:.2e}")
    assert s["tokens"] == cfg.tq
    assert s["mem_bad"] == 0 and s["h_bad"] == 0, s
