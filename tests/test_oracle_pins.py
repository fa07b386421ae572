"""Pins for the CPU oracle: checks against facts other than its own formulas.

Each test names the mistake it would catch.  No expected value here comes
from the CUDA path.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from synth import host
from synth.configs import CONFIGS, default_seeds, make_tokens

GOLDEN = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1
HERE = os.path.dirname(os.path.abspath(__file__))


# --------------------------------------------------------------- the hash ---


def _unmix(h, ids):
    """Walk a chain backwards with the INVERSE maps: undo h ^= h >> 29 by
    re-applying the shifted xor until it is a fixed point, multiply by the
    modular inverse of the odd constant, xor the id back out."""
    cinv = pow(GOLDEN, -1, 1 << 64)
    for tok in reversed(ids):
        x = h
        for _ in range(3):  # 29-bit shifts: three passes recover 64 bits
            x = h ^ (x >> 29)
        h = ((x * cinv) & M64) ^ tok
    return h


@pytest.mark.parametrize("ids", [[1, 2], [5, 7, 11], [1024, 1024, 1024, 5], [0, 0], [129279, 3, 77, 129279]])
def test_mix_chain_inverts_to_seed(ids):
    """The chain is a bijection; undoing it with inverse maps must give the
    seed back.  Catches a wrong shift, arithmetic shift, dropped xor, wrong
    constant or ids taken newest-first."""
    for seed in [0, 1, 0xE220A8397B1DCDAF, M64]:
        h = oracle.mix_chain(seed, ids)
        assert _unmix(h, ids) == seed
        if len(set(ids)) > 1:
            assert _unmix(h, list(reversed(ids))) != seed


def test_mix_chain_single_step_closed_form():
    """seed 0 and id 1: h = C, then C ^ (C >> 29)."""
    assert oracle.mix_chain(0, [1]) == GOLDEN ^ (GOLDEN >> 29)
    assert oracle.mix_chain(5, []) == 5


def test_default_seeds_are_splitmix64():
    # published first outputs of SplitMix64 from state 0
    s = default_seeds()
    assert int(s[0]) == 0xE220A8397B1DCDAF
    assert int(s[1]) == 0x6E789E6AA1B965F4


def test_hash_pow2_is_low_bits_and_prime_is_mod():
    """idx = h mod R: for R = 2^k, idx(2^k) = idx(2^20) mod 2^k; for a prime R
    the residues against the mix-chain value agree."""
    cfg = CONFIGS["tiny"]
    tok, offs = make_tokens(cfg)
    seeds = default_seeds()
    a = oracle.hash_tokens(tok[:64], np.array([0, 64]), 0, cfg.V, 1 << 20, seeds)
    b = oracle.hash_tokens(tok[:64], np.array([0, 64]), 0, cfg.V, 4096, seeds)
    assert np.array_equal(a % 4096, b)
    c = oracle.hash_tokens(tok[:64], np.array([0, 64]), 0, cfg.V, 4093, seeds)
    # position 10, table j=16 (module 0, order 4, head 0): 4-gram tok[7..10]
    h = oracle.mix_chain(int(seeds[16]), [int(x) for x in tok[7:11]])
    assert c[10, 16] == h % 4093 and b[10, 16] == h % 4096


def test_hash_table_layout_order_and_head():
    """Table j = (module*3 + order-2)*8 + head: the n-gram length of table j
    shows in which ids change its output."""
    V, R = 1024, 1 << 30
    seeds = default_seeds()
    base = np.array([3, 4, 5, 6, 7], dtype=np.int32)
    offs = np.array([0, 5])
    i0 = oracle.hash_tokens(base, offs, 0, V, R, seeds)[4]
    for back, order_min in [(1, 2), (2, 3), (3, 4)]:
        alt = base.copy()
        alt[4 - back] = 999  # change the id `back` places before the last
        i1 = oracle.hash_tokens(alt, offs, 0, V, R, seeds)[4]
        changed = i1 != i0
        for j in range(48):
            order = 2 + (j % 24) // 8
            assert changed[j] == (order >= order_min), (j, back)


def test_padding_and_sequence_isolation():
    """Positions before a sequence start read the pad id V: the first token
    of every sequence hashes like the same id at position 0; a sequence's
    idx block does not depend on what is packed before it."""
    V, R = 1024, 4096
    seeds = default_seeds()
    rng = np.random.default_rng(1)
    seq = rng.integers(0, V, 20).astype(np.int32)
    other = rng.integers(0, V, 13).astype(np.int32)
    packed = np.concatenate([other, seq, seq])
    offs = np.array([0, 13, 33, 53])
    idx = oracle.hash_tokens(packed, offs, 0, V, R, seeds)
    alone = oracle.hash_tokens(seq, np.array([0, 20]), 0, V, R, seeds)
    assert np.array_equal(idx[13:33], alone) and np.array_equal(idx[33:53], alone)
    # explicit pad ids give the same n-grams as the implicit sequence start
    # (V is the pad; a stream may not contain V itself, so hash the chain)
    for j in range(48):
        n = 2 + (j % 24) // 8
        h = oracle.mix_chain(int(seeds[j]), [V] * (n - 1) + [int(seq[0])])
        assert alone[0, j] == h % R


def test_hash_last_n_selects_tail():
    V, R = 1024, 4096
    seeds = default_seeds()
    tok = np.arange(40, dtype=np.int32) % V
    offs = np.array([0, 10, 25, 40])
    full = oracle.hash_tokens(tok, offs, 0, V, R, seeds)
    last = oracle.hash_tokens(tok, offs, 2, V, R, seeds)
    assert np.array_equal(last, full[[8, 9, 23, 24, 38, 39]])
    with pytest.raises(oracle.OracleError):
        oracle.hash_tokens(tok, np.array([0, 1, 40]), 2, V, R, seeds)


def test_hash_rejects_out_of_range_ids():
    with pytest.raises(oracle.OracleError):
        oracle.hash_tokens(np.array([1, 1024], np.int32), np.array([0, 2]), 0, 1024, 16, default_seeds())


# ------------------------------------------------------------- e4m3 / bf16 ---


def test_e4m3_decode_matches_torch_float8():
    """All 256 codes against torch's float8_e4m3fn (a library decoder)."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0**-9 and math.copysign(1, oracle.e4m3_value(0x80)) < 0


def _bf16_grid():
    codes = np.arange(65536, dtype=np.int64)
    vals = torch.from_numpy(codes.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(vals) & ~((vals == 0) & np.signbit(vals))
    return vals[fin], codes[fin]


def _nearest_bf16_exact(x, grid_vals, grid_codes):
    """Nearest bf16 by exact rational comparison, ties to the even code."""
    fx = Fraction(x)
    i = int(np.searchsorted(grid_vals, x))
    cands = [k for k in (i - 1, i, i + 1) if 0 <= k < len(grid_vals)]
    best = min(cands, key=lambda k: (abs(Fraction(grid_vals[k]) - fx), int(grid_codes[k]) & 1))
    return int(grid_codes[best])


def test_bf16_rne_against_exact_grid():
    """Single rounding of doubles to bf16, checked by exact nearest-neighbour
    search over the bf16 grid (ties to even).  Catches double rounding through
    float32, truncation and ties-away."""
    vals, codes = _bf16_grid()
    order = np.argsort(vals, kind="stable")
    vals, codes = vals[order], codes[order]
    pos = vals >= 0  # +0 is a candidate (ties at half the smallest subnormal)
    pv, pc = vals[pos], codes[pos]
    rng = np.random.default_rng(7)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-5, 6, 3000))
    # exact midpoints, and midpoints nudged by one double ulp both ways
    for k in rng.integers(0, len(pv) - 1, 400):
        mid = (pv[k] + pv[k + 1]) / 2
        xs += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf)]
    xs += [2.0**-133, 2.0**-134, 3 * 2.0**-135, 2.0**-126, 2.0**-127]
    for x in xs:
        x = float(abs(x))
        if x == 0 or x > 3e38:
            continue
        assert oracle.bf16_rne(x) == _nearest_bf16_exact(x, pv, pc), x
        assert oracle.bf16_rne(-x) == _nearest_bf16_exact(x, pv, pc) | 0x8000
    assert oracle.bf16_rne(1.0) == 0x3F80 and oracle.bf16_rne(-0.0) == 0x8000
    assert oracle.bf16_rne(3.5e38) == 0x7F80  # past the largest finite value


def test_bf16_rne_matches_torch_on_float32_inputs():
    """On float32-representable inputs torch's float->bf16 conversion is one
    round-to-nearest-even step: agree with it on random and tie cases."""
    rng = np.random.default_rng(3)
    f = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ties = (rng.integers(0, 1 << 16, 5000).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(x)) for x in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------ gather-reduce --


def _rand_tables(rng, R):
    t = rng.integers(0, 256, size=(48, R, 256)).astype(np.uint8)
    t[(t & 0x7F) == 0x7F] = 0x38  # no NaN codes in inputs
    s = rng.uniform(0.5, 2.0, size=(48, R)).astype(np.float32)
    return t, s


def test_gather_all_ones_counts_rows():
    """Every row = e4m3 1.0 (0x38), every scale 1: each module entry is the
    number of rows summed, 24 -- so 48 rows of 256 values per token."""
    R = 32
    t = np.full((48, R, 256), 0x38, np.uint8)
    s = np.ones((48, R), np.float32)
    idx = np.random.default_rng(0).integers(0, R, size=(16, 48))
    mem = oracle.gather_reduce(t, s, idx)
    assert np.all(mem == 24.0)


def test_gather_brute_force_row_reads_16_tokens():
    """Enumerate every (table, row): light up that one row and see which
    tokens' sums move.  The read set found this way must be exactly
    {(j, idx[t, j])}: 48 reads of 256 B = 12,288 B per token."""
    V, R = 1024, 16
    seeds = default_seeds()
    tok = np.random.default_rng(5).integers(0, V, 16).astype(np.int32)
    offs = np.array([0, 16])
    idx = oracle.hash_tokens(tok, offs, 0, V, R, seeds)
    reads = np.zeros((16, 48), dtype=np.int64)  # count per (token, table)
    found = [[None] * 48 for _ in range(16)]
    s = np.ones((48, R), np.float32)
    for j in range(48):
        m = j // 24
        for r in range(R):
            t = np.zeros((48, R, 256), np.uint8)
            t[j, r, :] = 0x38
            mem = oracle.gather_reduce(t, s, idx)
            hits = mem[:, 256 * m]  # how many times token t read (j, r)
            assert np.all(mem[:, 256 * m : 256 * m + 256] == hits[:, None])
            assert np.all(mem[:, 256 * (1 - m) : 256 * (1 - m) + 256] == 0)
            for tt in np.nonzero(hits)[0]:
                reads[tt, j] += int(hits[tt])
                found[tt][j] = r
    assert np.all(reads == 1)
    assert all(found[t][j] == idx[t, j] for t in range(16) for j in range(48))
    assert reads.sum(axis=1).tolist() == [48] * 16
    assert reads.sum() * 256 // 16 == 12288


def test_gather_matches_dense_one_hot_matmul():
    """mem as a dense product: one-hot(idx) x (scale * decoded rows) summed
    over the module's tables, with torch's float8 decoder and numpy matmul.
    Catches a wrong module split, a transposed idx or a wrong scale row."""
    rng = np.random.default_rng(11)
    R, T = 8, 20
    t, s = _rand_tables(rng, R)
    idx = rng.integers(0, R, size=(T, 48))
    dec = torch.from_numpy(t.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(48, R, 256)
    ref = np.zeros((T, 512))
    for j in range(48):
        onehot = np.zeros((T, R))
        onehot[np.arange(T), idx[:, j]] = 1.0
        ref[:, 256 * (j // 24) : 256 * (j // 24) + 256] += onehot @ (s[j].astype(np.float64)[:, None] * dec[j])
    got = oracle.gather_reduce(t, s, idx)
    assert np.array_equal(got, ref)


def test_gather_is_exact_rational_sum():
    """The double sums are exact (terms are multiples of 2^-33 below 2^10):
    compare with Fractions."""
    rng = np.random.default_rng(12)
    R, T = 4, 3
    t, s = _rand_tables(rng, R)
    idx = rng.integers(0, R, size=(T, 48))
    got = oracle.gather_reduce(t, s, idx)
    ref = torch.from_numpy(t.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(48, R, 256)
    for tt in range(T):
        for c in range(0, 512, 37):
            m, cc = divmod(c, 256)
            exact = sum(Fraction(float(s[j, idx[tt, j]])) * Fraction(ref[j, idx[tt, j], cc]) for j in range(24 * m, 24 * m + 24))
            assert Fraction(got[tt, c]) == exact


def test_gather_scaling_and_permutation():
    rng = np.random.default_rng(13)
    R, T = 16, 10
    t, s = _rand_tables(rng, R)
    idx = rng.integers(0, R, size=(T, 48))
    base = oracle.gather_reduce(t, s, idx)
    assert np.array_equal(oracle.gather_reduce(t, s * np.float32(2), idx), 2 * base)
    perm = rng.permutation(R)
    inv = np.argsort(perm)
    t2, s2 = t[:, perm], s[:, perm]  # row r of t2 is row perm[r] of t
    idx2 = inv[idx]
    assert np.array_equal(oracle.gather_reduce(t2, s2, idx2), base)


def test_gather_rows_entry_matches_tables_entry():
    rng = np.random.default_rng(14)
    R, T = 16, 7
    t, s = _rand_tables(rng, R)
    idx = rng.integers(0, R, size=(T, 48))
    rows = np.stack([t[np.arange(48), idx[k]] for k in range(T)])
    sc = np.stack([s[np.arange(48), idx[k]] for k in range(T)])
    assert np.array_equal(oracle.gather_reduce_rows(rows, sc), oracle.gather_reduce(t, s, idx))


# ------------------------------------------------------------ MXFP8 rows ---


def test_e8m0_decode_matches_torch():
    """All 256 E8M0 codes against torch's float8_e8m0fnu (a library decoder)."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e8m0_value(c)
        assert (math.isnan(v) and math.isnan(ref[c])) or v == ref[c], c
    assert oracle.e8m0_value(127) == 1.0 and oracle.e8m0_value(0) == 2.0**-127


def test_mx_gather_block_scales():
    """Codes all 1.0 with block b scaled by 2^b: each module entry is
    24 * 2^(c // 32) exactly -- catches a wrong block index or bias."""
    T = 3
    rows = np.full((T, 48, 256), 0x38, np.uint8)
    esc = np.tile((127 + np.arange(8)).astype(np.uint8), (T, 48, 1))
    mem = oracle.gather_reduce_mx_rows(rows, esc)
    want = np.tile(24.0 * 2.0 ** (np.arange(256) // 32), 2)
    assert np.array_equal(mem, np.tile(want, (T, 1)))


def test_mx_gather_dense_matches_torch_decoders():
    """MX rows as a dense product with torch's float8 decoders: exact."""
    rng = np.random.default_rng(31)
    T = 6
    rows = rng.integers(0, 256, (T, 48, 256)).astype(np.uint8)
    rows[(rows & 0x7F) == 0x7F] = 0x38
    esc = rng.integers(120, 135, (T, 48, 8)).astype(np.uint8)
    dec = torch.from_numpy(rows.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(T, 48, 256)
    sc = torch.from_numpy(esc.reshape(-1)).view(torch.float8_e8m0fnu).to(torch.float64).numpy().reshape(T, 48, 8)
    full = dec * np.repeat(sc, 32, axis=2)
    ref = np.concatenate([full[:, :24].sum(axis=1), full[:, 24:].sum(axis=1)], axis=1)
    assert np.array_equal(oracle.gather_reduce_mx_rows(rows, esc), ref)


def test_mx_row_bytes_match_page_figure():
    """256 B of codes + 8 B of E8M0 scales = 264 B per row, 48 rows = 12,672 B."""
    fig = _page_figures()
    assert 48 * (256 + 8) == fig["bytes_per_token_with_scales"][0]
    assert 256 // 32 == fig["row_scale_bytes"][0]  # one scale byte per 32-code block


# --------------------------------------------------------------- the fuse ---


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(b):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_gate_closed_forms():
    """Constant h = a with g = 1: rmsnorm(h) = sign(a), dot = sign(a)*d, so
    gate = sigmoid(sign(a)*sqrt(d)).  One-hot h = a*e_i, g = b*e_i: gate =
    sigmoid(sign(a)*b).  h = 0: gate = 1/2.  Catches sum-for-mean, a missing
    1/sqrt(d), a flipped sigmoid and a wrong rms."""
    d = 256
    W = np.zeros((512, d), np.uint16)
    mem = np.zeros((1, 512))
    for a in [1.5, -3.0, 0.25]:
        h = _bf16_bits(np.full((1, d), a))
        _, gate = oracle.fuse(mem, W, _bf16_bits(np.ones(d)), h, eps=0.0)
        assert abs(gate[0] - 1 / (1 + math.exp(-math.copysign(16.0, a)))) < 1e-15
    for a, b, i in [(2.0, 0.75, 3), (-1.0, 1.5, 200)]:
        hv = np.zeros((1, d)); hv[0, i] = a
        gv = np.zeros(d); gv[i] = b
        _, gate = oracle.fuse(mem, W, _bf16_bits(gv), _bf16_bits(hv), eps=0.0)
        assert abs(gate[0] - 1 / (1 + math.exp(-math.copysign(1, a) * b))) < 1e-14
    _, gate = oracle.fuse(mem, W, _bf16_bits(np.ones(d)), np.zeros((1, d), np.uint16), eps=1e-6)
    assert gate[0] == 0.5


def test_fuse_special_cases_leave_h():
    """W = 0 or mem = 0: h is bit-unchanged; g = 0: gate is exactly 1/2."""
    rng = np.random.default_rng(21)
    d, T = 256, 5
    h = host.h_rows(0, d, np.arange(T))
    W = host.w_out(0, d)
    g = host.g_vec(0, d)
    mem = rng.standard_normal((T, 512)) * 5
    hn, _ = oracle.fuse(mem, np.zeros_like(W), g, h)
    assert np.array_equal(hn, h)
    hn, _ = oracle.fuse(np.zeros_like(mem), W, g, h)
    assert np.array_equal(hn, h)
    _, gate = oracle.fuse(mem, W, np.zeros_like(g), h)
    assert np.all(gate == 0.5)
    # scaling h by 2^k leaves the gate unchanged (eps = 0)
    _, g1 = oracle.fuse(mem, W, g, h, eps=0.0)
    _, g2 = oracle.fuse(mem, W, g, _bf16_bits(_bf16_vals(h) * 4), eps=0.0)
    assert np.allclose(g1, g2, rtol=0, atol=1e-15)


def test_fuse_one_hot_projection_indexing():
    """X one-hot at k with a bf16-exact value: y_c = X_k * W[k, c] exactly.
    Catches a transposed W or a wrong k/c index."""
    d = 256
    rng = np.random.default_rng(22)
    W = host.w_out(1, d)
    Wv = _bf16_vals(W)
    h = np.zeros((1, d), np.uint16)
    g = np.zeros(d, np.uint16)  # gate 1/2
    for k in [0, 255, 256, 511]:
        mem = np.zeros((1, 512))
        mem[0, k] = 2.0
        hn, gate = oracle.fuse(mem, W, g, h)
        assert gate[0] == 0.5
        assert np.array_equal(hn[0], _bf16_bits(Wv[k]))  # 0 + 0.5*2*W[k,:]


def test_fuse_against_library_matmul():
    """General case vs numpy's float64 matmul of the bf16 values, with the
    gate from the closed-form pins above; the final rounding of the exact
    value to bf16 must agree except where a double-precision sum lands within
    1e-9 of a bf16 rounding boundary."""
    rng = np.random.default_rng(23)
    d, T = 256, 9
    h = host.h_rows(2, d, np.arange(T))
    W = host.w_out(2, d)
    g = host.g_vec(2, d)
    mem = rng.standard_normal((T, 512)) * 6
    hn, gate = oracle.fuse(mem, W, g, h)
    X = np.array([[oracle.bf16_value(oracle.bf16_rne(v)) for v in row] for row in mem])
    hv = _bf16_vals(h)
    y = X @ _bf16_vals(W)
    rr = 1 / np.sqrt((hv**2).mean(axis=1) + 1e-6)
    gref = 1 / (1 + np.exp(-(rr * (hv @ _bf16_vals(g))) / np.sqrt(d)))
    assert np.allclose(gate, gref, rtol=1e-13, atol=0)
    ref = hv + gref[:, None] * y
    got = _bf16_vals(hn)
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) * 2.0**16
    assert np.all(np.abs(got - ref) <= 0.5 * ulp * (1 + 1e-9))


# ------------------------------------------------------- the pages' figures --


def _page_figures():
    out = {}
    with open(os.path.join(HERE, "golden", "page_figures.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, val, unit, _src = [x.strip() for x in line.split("|", 3)]
            out[name] = (float(val), unit)
    return out


def test_page_figures_from_oracle_accounting():
    """The read the oracle performs (48 rows x 256 B, counted by the
    all-ones test above) reproduces the figures the pages print."""
    fig = _page_figures()
    R = 8
    t = np.full((48, R, 256), 0x38, np.uint8)
    mem = oracle.gather_reduce(t, np.ones((48, R), np.float32), np.zeros((1, 48), np.int64))
    rows = int(mem[0, 0] + mem[0, 256])  # 24 per module
    assert rows == fig["rows_per_token"][0] and rows // 2 == fig["rows_per_layer"][0]
    bytes_tok = rows * int(fig["row_fp8_bytes"][0])
    assert bytes_tok == 12 * 1024 == fig["bytes_per_token_approx"][0] * 1024  # "about 12 KB"
    assert 10 * bytes_tok == fig["decode_bandwidth_10tps"][0] * 1024  # 120 KB/s
    with_scales = rows * int(fig["row_fp8_bytes"][0] + fig["row_scale_bytes"][0])
    assert with_scales == fig["bytes_per_token_with_scales"][0]
    assert round(2000 * with_scales / 1e6) == fig["host_traffic_2000tps"][0]  # 25.3 MB/s
    assert round(131072 * with_scales / 1e9, 1) == fig["prompt_128k_reads"][0]  # 1.66 GB
    assert fig["modules"][0] * 3 * fig["heads_per_order"][0] == rows


# ----------------------------------------------- per-row gated Engram layer --

def _bf16_bits(x):
    """float64 array -> bf16 bit patterns (torch's round-to-nearest-even)."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _e4m3_vals(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _layer_inputs(T=3, d=256, seed=41):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, (T, 24, 256)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
    scales = rng.uniform(0.5, 2.0, (T, 24)).astype(np.float32)
    Wq = _bf16_bits(rng.standard_normal((d, 256)) / np.sqrt(d))
    Wk = _bf16_bits(rng.standard_normal((256, 256)) / 16.0)
    Wm = _bf16_bits(rng.standard_normal((256, d)) / 16.0)
    h = _bf16_bits(rng.standard_normal((T, d)))
    return codes, scales, Wq, Wk, Wm, h


def test_layer_gate_half_when_query_is_zero():
    """W_q = 0: every score is 0, every gate exactly 1/2, e is half the plain
    module sum (torch's decoder), and with W_m = I (d = 256) h becomes
    bf16(h + bf16(e)) (torch's rounding)."""
    codes, scales, Wq, Wk, Wm, h = _layer_inputs()
    Wq = np.zeros_like(Wq)
    eye = _bf16_bits(np.eye(256))
    hn, gates, e = oracle.layer_gated(codes, scales, Wq, Wk, eye, h)
    assert np.all(gates == 0.5)
    plain = (_e4m3_vals(codes) * scales[:, :, None].astype(np.float64)).sum(axis=1)
    assert np.array_equal(e, plain / 2)
    X = _bf16_vals(_bf16_bits(e))
    assert np.array_equal(hn, _bf16_bits(_bf16_vals(h) + X))


def test_layer_zero_projection_leaves_h():
    codes, scales, Wq, Wk, Wm, h = _layer_inputs(d=512)
    hn, _, _ = oracle.layer_gated(codes, scales, Wq, Wk, np.zeros_like(Wm), h)
    assert np.array_equal(hn, h)


def test_layer_closed_form_scores():
    """Constant h and constant rows with eps = 0: rmsnorm gives +-1 vectors, and
    with W_q (2^-9, d = 512) and W_k (2^-8) one-hot in column 0 every dot is
    sign(h) * sign(row) exactly, so each gate is sigmoid(+-1/16): the score is
    divided by sqrt(256), the width of the dot, not by sqrt(d)."""
    T, d = 2, 512
    rng = np.random.default_rng(5)
    codes = np.zeros((T, 24, 256), np.uint8)
    pick = rng.choice(np.array([0x38, 0x40, 0xB8, 0xC4, 0x2A, 0xAA], np.uint8), (T, 24))
    codes[:] = pick[:, :, None]
    scales = rng.uniform(0.5, 2.0, (T, 24)).astype(np.float32)
    Wq = np.zeros((d, 256), np.uint16)
    Wq[:, 0] = _bf16_bits(np.full(d, 2.0**-9))
    Wk = np.zeros((256, 256), np.uint16)
    Wk[:, 0] = _bf16_bits(np.full(256, 2.0**-8))
    hsign = np.array([1.0, -1.0])
    h = _bf16_bits(np.repeat(hsign[:, None] * 0.75, d, axis=1))
    _, gates, e = oracle.layer_gated(codes, scales, Wq, Wk, np.zeros((256, d), np.uint16), h, eps=0.0)
    vals = _e4m3_vals(pick) * scales.astype(np.float64)
    want = 1.0 / (1.0 + np.exp(-(hsign[:, None] * np.sign(vals)) / 16.0))
    assert np.allclose(gates, want, rtol=0, atol=1e-15)
    assert np.allclose(e, (want * vals).sum(axis=1)[:, None] * np.ones(256), rtol=1e-14, atol=0)


def test_layer_gate_symmetries():
    """Negating W_k turns every gate g into 1 - g; permuting a token's rows
    permutes its gates and leaves e unchanged; doubling one row's scale leaves
    its gate (rmsnorm, eps = 0) and adds exactly g_j * r_j to e."""
    codes, scales, Wq, Wk, Wm, h = _layer_inputs(T=2, d=256)
    _, g1, e1 = oracle.layer_gated(codes, scales, Wq, Wk, Wm, h, eps=0.0)
    _, g2, _ = oracle.layer_gated(codes, scales, Wq, Wk ^ np.uint16(0x8000), Wm, h, eps=0.0)
    assert np.allclose(g1 + g2, 1.0, rtol=0, atol=1e-14)
    perm = np.random.default_rng(3).permutation(24)
    _, g3, e3 = oracle.layer_gated(codes[:, perm], scales[:, perm], Wq, Wk, Wm, h, eps=0.0)
    assert np.allclose(g3, g1[:, perm], rtol=0, atol=1e-15)
    assert np.allclose(e3, e1, rtol=1e-13, atol=1e-13)
    s2 = scales.copy()
    s2[:, 7] *= 2
    _, g4, e4 = oracle.layer_gated(codes, s2, Wq, Wk, Wm, h, eps=0.0)
    assert np.allclose(g4, g1, rtol=0, atol=1e-15)
    r7 = _e4m3_vals(codes[:, 7]) * scales[:, 7:8].astype(np.float64)
    assert np.allclose(e4 - e1, g1[:, 7:8] * r7, rtol=1e-12, atol=1e-12)


def test_layer_mx_equal_block_scales_match_one_row_scale():
    """MXFP8-style rows whose eight E8M0 bytes all equal E give exactly the
    one-scale form with scale 2^(E - 127) (the same doubles: a power of two
    times an e4m3 value), for h, gates and e."""
    codes, _, Wq, Wk, Wm, h = _layer_inputs(T=3, d=512, seed=43)
    E = np.random.default_rng(9).integers(124, 131, (3, 24)).astype(np.uint8)
    esc = np.repeat(E[:, :, None], 8, axis=2)
    want = oracle.layer_gated(codes, np.ldexp(1.0, E.astype(np.int32) - 127).astype(np.float32), Wq, Wk, Wm, h)
    got = oracle.layer_gated(codes, esc, Wq, Wk, Wm, h)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


def test_layer_mx_block_scale_applies_to_its_32_codes():
    """Block b's scale byte 128 (x2) against byte 127 (x1) equals doubling the
    values of codes 32b..32b+31 of that row, written as e4m3 codes (normal
    codes with exponent field below 14: code + 8 is the double).  One block
    per row, different blocks in different rows: a scale applied to the wrong
    32 codes fails."""
    T, d = 2, 256
    codes, _, Wq, Wk, Wm, h = _layer_inputs(T=T, d=d, seed=47)
    rng = np.random.default_rng(13)
    exp = rng.integers(1, 14, codes.shape)
    codes = ((codes & 0x80) | (exp << 3) | (codes & 0x07)).astype(np.uint8)  # normal, exponent field 1..13
    esc = np.full((T, 24, 8), 127, np.uint8)
    doubled = codes.copy()
    for t in range(T):
        for j in range(24):
            blk = (3 * j + t) % 8
            esc[t, j, blk] = 128
            doubled[t, j, 32 * blk:32 * blk + 32] += 8
    assert np.array_equal(_e4m3_vals(doubled[0, 0, :32]), 2 * _e4m3_vals(codes[0, 0, :32]))
    want = oracle.layer_gated(doubled, np.ones((T, 24), np.float32), Wq, Wk, Wm, h)
    got = oracle.layer_gated(codes, esc, Wq, Wk, Wm, h)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


def test_hash_positions_entry_rows():
    """The explicit-position entry (used for sampled references) against
    windows built here: any order, repeats, every sequence start and a
    sequence of one token; each row equals the mix chain of its n-gram with
    the pad id before the sequence start, and the rows equal those of the
    every-query entry.  A wrong sequence lookup or window offset in the
    position entry fails here."""
    V, R = 1024, 4093
    seeds = default_seeds()
    rng = np.random.default_rng(11)
    lens = [7, 1, 3, 12]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = rng.integers(0, V, offs[-1]).astype(np.int32)
    pos = np.concatenate([rng.permutation(offs[-1]), [0, 7, 8, 11, 11]]).astype(np.int64)
    got = oracle.hash_positions(tok, offs, V, R, seeds, pos)
    full = oracle.hash_tokens(tok, offs, 0, V, R, seeds)
    assert np.array_equal(got, full[pos])
    for i, p in enumerate(pos):
        s = int(np.searchsorted(offs, p, side="right") - 1)
        for j in range(48):
            n = 2 + (j % 24) // 8
            ids = [int(tok[q]) if q >= offs[s] else V for q in range(p - n + 1, p + 1)]
            assert got[i, j] == oracle.mix_chain(int(seeds[j]), ids) % R
    with pytest.raises(oracle.OracleError):  # a position past the last sequence
        oracle.hash_positions(tok, offs, V, R, seeds, np.array([offs[-1]]))
