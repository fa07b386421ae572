"""Host-side (numpy) draws of the workloads' tensors, by counter.

Any table row, scale or residual element can be drawn on its own, so the
oracle side can regenerate exactly the rows it needs while the device twin
(``synth/device.py``) fills whole tables of tens of GB in HBM.
"""

import functools

import numpy as np

from .configs import (
    N_TABLES,
    ROW_BYTES,
    STREAM_G,
    STREAM_H,
    STREAM_MX,
    STREAM_SCALE,
    STREAM_TABLE,
    STREAM_W,
    STREAM_WK,
    STREAM_WM,
    STREAM_WQ,
)
from .philox import philox4x64, philox_u32
from .sampler import bf16_normal_table, e4m3_normal_table, sample_codes, scale_from_u32

W_SIGMA = 1.0 / np.sqrt(512.0)


@functools.lru_cache(maxsize=None)
def e4m3_table():
    return e4m3_normal_table(1.0)


@functools.lru_cache(maxsize=None)
def bf16_table(sigma):
    return bf16_normal_table(float(sigma))


def table_rows(seed, j, row):
    """e4m3 code bytes uint8 [n, 256] of rows (j[i], row[i])."""
    j = np.asarray(j, dtype=np.uint64).reshape(-1)
    row = np.asarray(row, dtype=np.uint64).reshape(-1)
    blocks = row[:, None] * np.uint64(ROW_BYTES // 8) + np.arange(ROW_BYTES // 8, dtype=np.uint64)[None, :]
    out = philox4x64(blocks, 0, 0, 0, np.uint64(seed), (np.uint64(STREAM_TABLE) + j)[:, None])
    u = out.reshape(len(row), -1).view(np.uint32)  # little-endian: low half first
    return sample_codes(e4m3_table(), u).astype(np.uint8).reshape(len(row), ROW_BYTES)


def scales(seed, j, row):
    """fp32 scales [n] of rows (j[i], row[i])."""
    j = np.asarray(j, dtype=np.uint64).reshape(-1)
    row = np.asarray(row, dtype=np.uint64).reshape(-1)
    u = philox_u32(np.uint64(seed), np.uint64(STREAM_SCALE) + j, row)
    return scale_from_u32(u)


def mx_scales(seed, j, row):
    """E8M0 block-scale bytes uint8 [n, 8] of rows (j[i], row[i]): byte b is
    125 + floor(5 u / 2^32) for word row*8 + b of stream (seed, 0x400 + j),
    i.e. block scales 2^-2 .. 2^2."""
    j = np.asarray(j, dtype=np.uint64).reshape(-1)
    row = np.asarray(row, dtype=np.uint64).reshape(-1)
    out = philox4x64(row, 0, 0, 0, np.uint64(seed), np.uint64(STREAM_MX) + j)
    u = out.reshape(len(row), 4).view(np.uint32).astype(np.uint64)  # little-endian: words row*8 + 0..7
    return (125 + ((u * np.uint64(5)) >> np.uint64(32))).astype(np.uint8)


def full_tables(seed, R):
    """Whole tables uint8 [48, R, 256] and scales fp32 [48, R] (small R only)."""
    jj = np.repeat(np.arange(N_TABLES), R)
    rr = np.tile(np.arange(R), N_TABLES)
    t = table_rows(seed, jj, rr).reshape(N_TABLES, R, ROW_BYTES)
    s = scales(seed, jj, rr).reshape(N_TABLES, R)
    return t, s


def bf16_words(seed, stream, sigma, word0, count):
    """bf16 bit patterns uint16 [count] of words word0.. of a stream."""
    w = np.uint64(word0) + np.arange(count, dtype=np.uint64)
    u = philox_u32(np.uint64(seed), np.uint64(stream), w)
    return sample_codes(bf16_table(sigma), u).astype(np.uint16)


def h_rows(seed, d, t_idx):
    """Residual rows h bf16 bits [n, d] of query tokens t_idx (N(0,1))."""
    t_idx = np.asarray(t_idx, dtype=np.uint64).reshape(-1)
    w = t_idx[:, None] * np.uint64(d) + np.arange(d, dtype=np.uint64)[None, :]
    u = philox_u32(np.uint64(seed), np.uint64(STREAM_H), w)
    return sample_codes(bf16_table(1.0), u).astype(np.uint16).reshape(len(t_idx), d)


def w_out(seed, d):
    """W_out bf16 bits [512, d], N(0, 1/512).  Drawn once per (seed, d) (a
    512 x 32768 matrix takes ~20 s to draw); each call gets its own copy."""
    return _w_out(int(seed), int(d)).copy()


@functools.lru_cache(maxsize=4)
def _w_out(seed, d):
    w = bf16_words(seed, STREAM_W, W_SIGMA, 0, 512 * d).reshape(512, d)
    w.setflags(write=False)
    return w


def layer_weights(seed, d, m):
    """Per-layer gate and projection weights (bf16 bits) of Engram layer m:
    W_q [d,256] ~ N(0,1/d), W_k [256,256] ~ N(0,1/256), W_m [256,d] ~ N(0,1/256)."""
    wq = bf16_words(seed, STREAM_WQ + m, 1.0 / np.sqrt(d), 0, d * 256).reshape(d, 256)
    wk = bf16_words(seed, STREAM_WK + m, 1.0 / 16.0, 0, 256 * 256).reshape(256, 256)
    wm = bf16_words(seed, STREAM_WM + m, 1.0 / 16.0, 0, 256 * d).reshape(256, d)
    return wq, wk, wm


def g_vec(seed, d):
    """Gate vector g bf16 bits [d], N(0, 1)."""
    return bf16_words(seed, STREAM_G, 1.0, 0, d)
