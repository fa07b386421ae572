"""The seeded input generators: Philox against numpy's, samplers, recipes."""

import math

import numpy as np
import torch

from synth import host
from synth.configs import CONFIGS, make_tokens, query_positions, span_info
from synth.philox import philox4x64, philox_u32
from synth.sampler import e4m3_normal_table, sample_codes, scale_from_u32


def test_philox_matches_numpy_philox():
    """numpy's Philox bit generator is Philox4x64-10; it bumps the counter
    before each block, so its n-th block is our counter n+1."""
    for key in [(0, 0), (3, 0x300), (0xFFFFFFFFFFFFFFFF, 12345)]:
        bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.zeros(4, dtype=np.uint64))
        ref = bg.random_raw(4 * 64).reshape(64, 4)
        got = philox4x64(np.arange(1, 65, dtype=np.uint64), 0, 0, 0, key[0], key[1])
        assert np.array_equal(got, ref)


def test_philox_u32_word_layout():
    out = philox4x64(np.uint64(5), 0, 0, 0, 7, 9)
    words = philox_u32(7, 9, np.arange(40, 48, dtype=np.uint64))
    assert np.array_equal(words, out.view(np.uint32))


def test_e4m3_sampler_distribution():
    tab = e4m3_normal_table(1.0)
    u = np.random.default_rng(0).integers(0, 1 << 32, 400000, dtype=np.uint64).astype(np.uint32)
    codes = sample_codes(tab, u).astype(np.uint8)
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    assert not np.any((codes & 0x7F) == 0x7F)  # never NaN
    # a code's frequency matches its quantisation interval: 1.0 (0x38) sits
    # between 0.9375 and 1.125, so it owns [0.96875, 1.0625)
    p = 0.5 * (math.erf(1.0625 / math.sqrt(2)) - math.erf(0.96875 / math.sqrt(2)))
    assert abs(np.mean(codes == 0x38) - p) < 5 * math.sqrt(p / len(u))


def test_scales_range_and_exactness():
    u = np.array([0, 0xFFFFFFFF, 1 << 31], dtype=np.uint32)
    s = scale_from_u32(u)
    assert s[0] == 0.5 and s[1] < 2.0 and s.dtype == np.float32
    big = host.scales(4, np.arange(48).repeat(1000), np.arange(48000))
    assert big.min() >= 0.5 and big.max() < 2.0 and abs(big.mean() - 1.25) < 0.01


def test_mx_scales_word_layout_and_range():
    """Byte b of row r is drawn from word r*8 + b of stream 0x400 + j, mapped
    to 125 + floor(5u / 2^32): exponents 125..129 (scales 2^-2 .. 2^2), each
    about equally likely."""
    j = np.array([0, 3, 47, 47])
    r = np.array([0, 1, 999, 2**23 - 1])
    got = host.mx_scales(7, j, r)
    for i in range(len(j)):
        u = philox_u32(np.uint64(7), np.uint64(0x400 + j[i]), np.uint64(r[i]) * np.uint64(8) + np.arange(8, dtype=np.uint64))
        want = [125 + (int(x) * 5 >> 32) for x in u]
        assert got[i].tolist() == want
    e = host.mx_scales(1, np.zeros(40000, np.int64), np.arange(40000))
    counts = np.bincount(e.ravel(), minlength=130)
    assert counts[:125].sum() == 0 and np.all(np.abs(counts[125:] / e.size - 0.2) < 0.01)


def test_rows_are_counter_addressable():
    """A row drawn alone equals the same row drawn inside a batch."""
    a = host.table_rows(3, [5, 5, 47], [0, 1000, 8388607])
    b = host.table_rows(3, [47], [8388607])
    assert np.array_equal(a[2], b[0])
    h1 = host.h_rows(3, 4096, [7, 131071])
    h2 = host.h_rows(3, 4096, [131071])
    assert np.array_equal(h1[1], h2[0])


def test_token_recipes():
    for name, cfg in CONFIGS.items():
        tok, offs = make_tokens(cfg)
        assert tok.dtype == np.int32 and len(tok) == cfg.t_all and offs[-1] == cfg.t_all
        assert tok.min() >= 0 and tok.max() < cfg.V
        assert len(query_positions(cfg, offs)) == cfg.tq
    cfg = CONFIGS["prefill"]
    tok, offs = make_tokens(cfg)
    starts, L = span_info(cfg)
    assert len(starts) == 8 * 102
    first = tok[starts[0] : starts[0] + L]
    for s in starts[:102]:
        assert np.array_equal(tok[s : s + L], first)
    # uniform ids for the large workload
    tok, _ = make_tokens(CONFIGS["large"])
    assert abs(tok.mean() / CONFIGS["large"].V - 0.5) < 0.01
