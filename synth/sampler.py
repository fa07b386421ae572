"""Discrete inverse-CDF samplers driven by 32-bit uniforms.

"Values N(0, sigma) quantised to a format" is drawn here as: pick the code
whose round-to-nearest interval contains a normal draw, with exactly that
interval's probability (resolved to 2^-32).  The format's value grid comes
from torch's own float8_e4m3fn / bfloat16 dtypes (library conversions, not
this project's arithmetic); interval edges are midpoints of neighbouring
values and probabilities come from the normal CDF via ``math.erfc``.

A table is ``thresholds`` (uint32, n-1 entries, strictly increasing) and
``codes`` (n entries): a uniform u maps to ``codes[#{k: thresholds[k] <= u}]``.
Host and device evaluate that count with the same integer comparisons, so
they agree bit for bit.
"""

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class CdfTable:
    thresholds: np.ndarray  # uint32 [n-1]
    codes: np.ndarray  # uint16 [n] (e4m3 codes fit in the low byte)

    @property
    def n(self):
        return int(self.codes.shape[0])


def _normal_cdf(x, sigma):
    return 0.5 * math.erfc(-x / (sigma * math.sqrt(2.0)))


def _build(values, codes, sigma):
    """values: float64 grid (with -0 and +0 distinguished by sign of code)."""
    # Order by value; -0 sorts just below +0 (their shared edge is exactly 0).
    neg_zero = np.signbit(values) & (values == 0)
    key = values + np.where(neg_zero, -1e-300, 0.0)
    order = np.argsort(key, kind="stable")
    v = values[order]
    c = codes[order]
    n = len(v)
    upper = np.empty(n)
    upper[:-1] = 0.5 * (v[:-1] + v[1:])
    upper[-1] = math.inf
    cum = np.array(
        [1 << 32 if math.isinf(b) else int(round(_normal_cdf(b, sigma) * 2.0**32)) for b in upper],
        dtype=np.int64,
    )
    cum[-1] = 1 << 32
    # keep a code only if its interval has non-zero width at 2^-32 resolution
    prev = np.concatenate([[0], cum[:-1]])
    keep = cum > prev
    cum, c = cum[keep], c[keep]
    assert cum[-1] == 1 << 32 and np.all(np.diff(cum) > 0)
    return CdfTable(thresholds=cum[:-1].astype(np.uint32), codes=c.astype(np.uint16))


def e4m3_normal_table(sigma=1.0):
    """Codes of OCP E4M3FN drawn as RNE-quantised N(0, sigma)."""
    all_codes = np.arange(256, dtype=np.int64)
    vals = (
        torch.from_numpy(all_codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    )
    finite = np.isfinite(vals)
    return _build(vals[finite], all_codes[finite], sigma)


def bf16_normal_table(sigma=1.0):
    """Codes of bfloat16 drawn as RNE-quantised N(0, sigma)."""
    all_codes = np.arange(65536, dtype=np.int64)
    vals = (
        torch.from_numpy(all_codes.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    )
    finite = np.isfinite(vals)
    return _build(vals[finite], all_codes[finite], sigma)


def sample_codes(table, u):
    """Map uint32 uniforms to codes (host side of the device sampler)."""
    i = np.searchsorted(table.thresholds, np.asarray(u, dtype=np.uint32), side="right")
    return table.codes[i]


def scale_from_u32(u):
    """Per-row fp32 scale in [0.5, 2): float32(2^24 + 3*(u>>8)) * 2^-25.

    One int->float32 conversion (round to nearest even) and an exact
    power-of-two multiply, so host and device agree bit for bit.
    """
    u = np.asarray(u, dtype=np.uint32).astype(np.int64)
    x = ((1 << 24) + 3 * (u >> 8)).astype(np.float32)
    return x * np.float32(2.0**-25)
