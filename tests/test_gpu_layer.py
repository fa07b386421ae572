"""The per-layer Engram read with per-row gates: CUDA path vs the CPU oracle
(needs a GB300)."""

import numpy as np
import pytest
import torch

import oracle
from synth import device as sd
from synth import host
from synth.configs import CONFIGS
from workload import Workload, bf16_to_f64, check_h, sample_queries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eg():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import engram_gram_hash_gb300 as eg

    eg.lib()
    return eg


CASES = {
    "tiny": CONFIGS["tiny"],  # d = 256, one tile of 512 tokens... four tiles
    "d512_ragged": CONFIGS["tiny"].with_(d=512, seq_lens=(333, 2, 100), seed=7),
    "prefill_small": CONFIGS["prefill"].with_(seq_lens=(640, 421), R=1 << 16, seed=6),
    "decode_small": CONFIGS["decode"].with_(R=1 << 16),
    # 37 queries: the d-split projection's load boxes round up to 40 rows
    "decode_ragged": CONFIGS["decode"].with_(R=1 << 16, seq_lens=tuple(1 + (i % 4) for i in range(37)), seed=11),
    # d = 7168: 28 chunks (projection clusters of 7), query K = 7168
    "d7168": CONFIGS["tiny"].with_(d=7168, seq_lens=(300, 29), seed=13),
    "d7168_one_tile": CONFIGS["tiny"].with_(d=7168, seq_lens=(90,), seed=14),
}


def _weights(eg, cfg, m, dev="cuda"):
    wq = torch.empty((cfg.d, 256), dtype=torch.bfloat16, device=dev)
    wk = torch.empty((256, 256), dtype=torch.bfloat16, device=dev)
    wm = torch.empty((256, cfg.d), dtype=torch.bfloat16, device=dev)
    sd.fill_layer_weights(wq, wk, wm, cfg.seed, m)
    return wq, wk, wm


def _oracle_layers(w, q_sel, modules=(0, 1), h_in=None):
    """Oracle h after layers `modules` (and each layer's e and sum_j |r_j|) for
    query tokens q_sel, starting from h_in (bf16 bits [len(q_sel), d]) or the
    workload's h."""
    cfg = w.cfg
    idx = oracle.hash_positions(w.tok, w.offs, cfg.V, cfg.R, w.seeds, w.qpos[q_sel])
    h = host.h_rows(cfg.seed, cfg.d, q_sel) if h_in is None else h_in
    es, bounds = [], []
    for m in modules:
        jj = np.tile(np.arange(24 * m, 24 * m + 24), len(q_sel))
        r = idx[:, 24 * m:24 * m + 24].reshape(-1)
        codes = host.table_rows(cfg.seed, jj, r).reshape(len(q_sel), 24, 256)
        wq, wk, wm = host.layer_weights(cfg.seed, cfg.d, m)
        absv = np.abs(torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy())
        if w.layout == "mx":  # eight E8M0 block scales per row
            sc = host.mx_scales(cfg.seed, jj, r).reshape(len(q_sel), 24, 8)
            absv *= np.ldexp(1.0, np.repeat(sc.astype(np.int32) - 127, 32, axis=2))
        else:
            sc = host.scales(cfg.seed, jj, r).reshape(len(q_sel), 24)
            absv *= sc[:, :, None].astype(np.float64)
        h, _, e = oracle.layer_gated(codes, sc, wq, wk, wm, h, cfg.rms_eps)
        es.append(e)
        bounds.append(absv.sum(axis=1))
    return h, es, bounds


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_layer_keys(eg):
    """W_kk = [W_k^T ; W_k^T], bit for bit."""
    cfg = CONFIGS["tiny"]
    c = eg.make_config(cfg.V, cfg.R, cfg.d, list(range(48)))
    _, wk, _ = _weights(eg, cfg, 1)
    wkk = eg.engram_layer_keys(c, wk)
    torch.cuda.synchronize()
    t = wk.t().contiguous()
    assert torch.equal(wkk.view(torch.int16), torch.cat([t, t]).view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "d512_ragged", "prefill_small"])
def test_layer_stages(eg, name):
    """One layer, each kernel against float64 numpy fed the previous GPU
    stage's output: the query q = rinv(h) h W_qk (GPU W_qk); the gated sum X
    from the GPU's q and the rows (fp32 sums, one bf16 rounding); h + X W_m
    from the GPU's X (one bf16 rounding); then h against the oracle."""
    cfg = CASES[name]
    w = Workload(cfg)
    nq = cfg.tq
    h = w.fresh_h()
    h0 = h.double().cpu().numpy()
    ws = torch.empty(eg.engram_layer_workspace_bytes(w.c, nq), dtype=torch.uint8, device="cuda")
    wq, wk, wm = _weights(eg, cfg, 0)
    wkk = eg.engram_layer_keys(w.c, wk)
    eg.engram_layer_forward(w.c, 0, w.tokens, w.seq_offsets, w.tables, w.scales, wq, wkk, wm, h, n_query=nq,
                            workspace=ws)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    qpair, ug, Xg = eg.layer_workspace_views(ws, nq)
    q = sample_queries(cfg, w.offs, 64)
    qt = torch.from_numpy(q).cuda()
    H = h0[q]
    Wq = wq.double().cpu().numpy()
    Wk = wk.double().cpu().numpy()
    rinv = 1.0 / np.sqrt((H**2).mean(axis=1) + cfg.rms_eps)
    qp = qpair[qt].double().cpu().numpy()
    q_got = qp[:, :256] + qp[:, 256:]
    q_err = np.abs(q_got - rinv[:, None] * (H @ Wq)) / (rinv[:, None] * (np.abs(H) @ np.abs(Wq)))
    assert q_err.max() <= 5e-4, f"query error {q_err.max():.2e}"
    u_got = ug[qt].double().cpu().numpy()
    u_err = np.abs(u_got - q_got @ Wk.T) / (np.abs(q_got) @ np.abs(Wk.T))
    assert u_err.max() <= 1e-4, f"key-side query error {u_err.max():.2e}"
    q_got = u_got  # the gather scores rows against u
    # gated sum from the GPU's query
    idx = oracle.hash_positions(w.tok, w.offs, cfg.V, cfg.R, w.seeds, w.qpos[q])
    jj = np.tile(np.arange(24), len(q))
    codes = host.table_rows(cfg.seed, jj, idx[:, :24].reshape(-1)).reshape(len(q), 24, 256)
    sc = host.scales(cfg.seed, jj, idx[:, :24].reshape(-1)).reshape(len(q), 24)
    rows = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * sc[:, :, None]
    rr = 1.0 / np.sqrt((rows**2).mean(axis=2) + cfg.rms_eps)
    g = 1.0 / (1.0 + np.exp(-(rr * np.einsum("tc,tjc->tj", u_got, rows) / 16.0)))
    e = (g[:, :, None] * rows).sum(axis=1)
    X_got = Xg[qt].double().cpu().numpy()
    absr = np.abs(rows).sum(axis=1)
    x_err = np.abs(X_got - e) - 2.0**-8 * np.abs(e)
    assert np.all(x_err <= 1e-4 * absr), f"gated sum error {float((x_err / absr).max()):.2e} of sum|r|"
    # projection from the GPU's X
    y = X_got @ wm.double().cpu().numpy()
    h_got = h[qt].double().cpu().numpy()
    ref = H + y
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) * 65536.0
    assert np.all(np.abs(h_got - ref) <= ulp + 1e-3 * (np.abs(X_got) @ np.abs(wm.double().cpu().numpy())) + 1e-6), \
        f"projection error {float(np.abs(h_got - ref).max()):.3e}"
    ref_h, _, _ = _oracle_layers(w, q, modules=(0,))
    check_h(h[qt], ref_h)


@pytest.mark.parametrize("name", list(CASES) + ["mx:tiny", "mx:prefill_small", "mx:decode_ragged"])
def test_layers_match_oracle(eg, name):
    """Layer 0 then layer 1 on h, each layer against the oracle applied to the
    same input (the GPU's h before that layer): h within the fused form's
    tolerance, and the layer's X = bf16(sum_j g_j r_j) within 1e-3 of
    sum_j |r_j| plus a bf16 rounding of the oracle's e.  "mx:" cases use
    MXFP8-style rows (eight E8M0 block scales per row)."""
    layout, _, name = name.rpartition(":")
    cfg = CASES[name]
    w = Workload(cfg, layout=layout or "separate")
    nq = cfg.tq
    q = sample_queries(cfg, w.offs, 64 if cfg.d > 512 else nq)
    qt = torch.from_numpy(q).cuda()
    h = w.fresh_h()
    ws = torch.empty(eg.engram_layer_workspace_bytes(w.c, nq), dtype=torch.uint8, device="cuda")
    for m in (0, 1):
        h_before = _bits(h[qt])
        wq, wk, wm = _weights(eg, cfg, m)
        wkk = eg.engram_layer_keys(w.c, wk)
        eg.engram_layer_forward(w.c, m, w.tokens, w.seq_offsets, w.tables, w.scales, wq, wkk, wm, h,
                                last_n=cfg.last_n, n_query=nq, workspace=ws)
        X = eg.layer_workspace_views(ws, nq)[2][qt]
        torch.cuda.synchronize()
        assert eg.engram_last_error() == 0
        ref_h, es, bounds = _oracle_layers(w, q, modules=(m,), h_in=h_before)
        check_h(h[qt], ref_h)
        err = np.abs(bf16_to_f64(X) - es[0])
        assert np.all(err <= 1e-3 * bounds[0] + 2.0**-8 * np.abs(es[0]) + 1e-30), (m, float(err.max()))


@pytest.mark.parametrize("n", [1, 129, 257])
def test_layers_at_tile_boundaries(eg, n):
    """The per-layer form on 1 token, two tiles with a one-token tail, and
    three tiles with a one-token tail (d = 4096: the split-K query products
    and the d-split or cluster projection), both layers against the oracle on
    every token."""
    cfg = CONFIGS["prefill"].with_(seq_lens=(n,), R=1 << 16, seed=40 + n)
    w = Workload(cfg)
    q = np.arange(n)
    qt = torch.from_numpy(q).cuda()
    h = w.fresh_h()
    for m in (0, 1):
        h_before = _bits(h)
        wq, wk, wm = _weights(eg, cfg, m)
        eg.engram_layer_forward(w.c, m, w.tokens, w.seq_offsets, w.tables, w.scales, wq,
                                eg.engram_layer_keys(w.c, wk), wm, h)
        torch.cuda.synchronize()
        assert eg.engram_last_error() == 0
        ref_h, _, _ = _oracle_layers(w, q, modules=(m,), h_in=h_before)
        check_h(h[qt], ref_h)


def test_layers_many_tiles_persistent_loop(eg):
    """41,000 tokens at d = 4096 (321 tiles of 128, more than twice the SM
    count): the query kernels (grid = min(tiles, SMs)) and the ungated
    projection (persistent clusters) each take several tiles per CTA, so
    their ring and accumulator phases wrap across tiles.  Each layer is
    checked against the oracle on the same input h, on a seeded sample plus
    the tokens on both sides of every tile boundary a CTA crosses first (the
    first tile of each CTA's second and third pass) and the last token."""
    cfg = CONFIGS["prefill"].with_(seq_lens=(24000, 17000), R=1 << 16, seed=12)
    w = Workload(cfg)
    nq = cfg.tq
    tiles = -(-nq // 128)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert tiles > 2 * sms
    edges = set()
    for first in (sms // 4, sms // 4 * 2, sms, 2 * sms, tiles - 1):  # cluster and CTA strides, last tile
        for t in (first * 128 - 1, first * 128, first * 128 + 127):
            if 0 <= t < nq:
                edges.add(t)
    q = np.array(sorted(set(sample_queries(cfg, w.offs, 96).tolist()) | edges), dtype=np.int64)
    qt = torch.from_numpy(q).cuda()
    h = w.fresh_h()
    ws = torch.empty(eg.engram_layer_workspace_bytes(w.c, nq), dtype=torch.uint8, device="cuda")
    for m in (0, 1):
        h_before = _bits(h[qt])
        wq, wk, wm = _weights(eg, cfg, m)
        wkk = eg.engram_layer_keys(w.c, wk)
        eg.engram_layer_forward(w.c, m, w.tokens, w.seq_offsets, w.tables, w.scales, wq, wkk, wm, h, n_query=nq,
                                workspace=ws)
        X = eg.layer_workspace_views(ws, nq)[2][qt]
        torch.cuda.synchronize()
        assert eg.engram_last_error() == 0
        ref_h, es, bounds = _oracle_layers(w, q, modules=(m,), h_in=h_before)
        check_h(h[qt], ref_h)
        err = np.abs(bf16_to_f64(X) - es[0])
        assert np.all(err <= 1e-3 * bounds[0] + 2.0**-8 * np.abs(es[0]) + 1e-30), (m, float(err.max()))


def test_layers_every_token_large(eg):
    """The per-layer form on the full large workload (131,072 tokens, 103 GB
    of tables, the benchmark's --variant layers call): each layer on EVERY
    query token against the oracle applied to the GPU's h before that layer
    (every host core, spawned processes)."""
    from oracle_pool import check_layer_all_tokens

    cfg = CONFIGS["large"]
    w = Workload(cfg)
    nq = cfg.tq
    h = w.fresh_h()
    ws = torch.empty(eg.engram_layer_workspace_bytes(w.c, nq), dtype=torch.uint8, device="cuda")
    for m in (0, 1):
        h_in = _bits(h)
        wq, wk, wm = _weights(eg, cfg, m)
        wkk = eg.engram_layer_keys(w.c, wk)
        eg.engram_layer_forward(w.c, m, w.tokens, w.seq_offsets, w.tables, w.scales, wq, wkk, wm, h, n_query=nq,
                                workspace=ws)
        torch.cuda.synchronize()
        assert eg.engram_last_error() == 0
        X = _bits(eg.layer_workspace_views(ws, nq)[2])
        r = check_layer_all_tokens(cfg, w.seeds, w.tok, w.offs, w.qpos, m, h_in, _bits(h), X)
        print(f"layer {m}: {r}")
        assert r["tokens"] == nq and r["h_bad"] == 0 and r["x_bad"] == 0, r


def test_layer_record_layout_same_bits(eg):
    """Rows that carry their scale give the same h bits."""
    cfg = CASES["prefill_small"]
    a, b = Workload(cfg), Workload(cfg, layout="record")
    ha, hb = a.fresh_h(), b.fresh_h()
    wq, wk, wm = _weights(eg, cfg, 0)
    wkk = eg.engram_layer_keys(a.c, wk)
    eg.engram_layer_forward(a.c, 0, a.tokens, a.seq_offsets, a.tables, a.scales, wq, wkk, wm, ha)
    eg.engram_layer_forward(b.c, 0, b.tokens, b.seq_offsets, b.tables, None, wq, wkk, wm, hb)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(ha.view(torch.int16), hb.view(torch.int16))


def test_layer_argument_errors(eg):
    cfg = CASES["tiny"]
    w = Workload(cfg)
    wq, wk, wm = _weights(eg, cfg, 0)
    wkk = eg.engram_layer_keys(w.c, wk)
    with pytest.raises(eg.EngramError) as ex:
        eg.engram_layer_forward(w.c, 2, w.tokens, w.seq_offsets, w.tables, w.scales, wq, wkk, wm, w.fresh_h())
    assert ex.value.status == 1
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0


@pytest.mark.parametrize("name", ["decode_ragged", "prefill_small"])
def test_layers_in_cuda_graph(eg, name):
    """Both layers captured in one CUDA graph (their split-K query kernels,
    reductions and dependent launches included) give the eager bits."""
    cfg = CASES[name]
    w = Workload(cfg)
    nq = cfg.tq
    ws = torch.empty(eg.engram_layer_workspace_bytes(w.c, nq), dtype=torch.uint8, device="cuda")
    mats = []
    for m in (0, 1):
        wq, wk, wm = _weights(eg, cfg, m)
        mats.append((wq, eg.engram_layer_keys(w.c, wk), wm))
    s = torch.cuda.Stream()

    def step(h):
        for m in (0, 1):
            wq, wkk, wm = mats[m]
            eg.engram_layer_forward(w.c, m, w.tokens, w.seq_offsets, w.tables, w.scales, wq, wkk, wm, h,
                                    last_n=cfg.last_n, n_query=nq, workspace=ws, stream=s)

    h_eager = w.fresh_h()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step(h_eager)
        step(h_eager)
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    h_graph = w.fresh_h()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(h_graph)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert eg.engram_last_error() == 0
    assert torch.equal(h_graph.view(torch.int16), h_eager.view(torch.int16))
