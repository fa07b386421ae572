"""Device twin of synth/host.py: fills large tensors with the same draws.

``synth_dev.cu`` is compiled into ``synth/libsynth_dev.so`` by
``__graft_entry__.build()`` (or ``build()`` here).  Targets may be CUDA
tensors or pinned host tensors (the kernels write through unified
addressing).
"""

import ctypes
import os
import subprocess

import numpy as np
import torch

from .configs import N_TABLES, ROW_BYTES, STREAM_G, STREAM_H, STREAM_W, STREAM_WK, STREAM_WM, STREAM_WQ
from .host import W_SIGMA, bf16_table, e4m3_table

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth_dev.cu")
_LIB = os.path.join(_HERE, "libsynth_dev.so")
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build_cmd():
    return ["nvcc", *NVCC_ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-o", _LIB, _SRC]


def build(force=False):
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(build_cmd())
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise RuntimeError(f"{_LIB} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB)
        P, i64, u64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
        lib.synth_fill_tables.argtypes = [P, u64, i32, i32, i64, i64, P, P, i32, P]
        lib.synth_fill_scales.argtypes = [P, u64, i32, i32, i64, i64, i64, P]
        lib.synth_fill_mx_scales.argtypes = [P, u64, i32, i32, i64, i64, i64, P]
        lib.synth_fill_bf16.argtypes = [P, u64, u64, u64, i64, P, P, i32, P]
        for f in (lib.synth_fill_tables, lib.synth_fill_scales, lib.synth_fill_mx_scales, lib.synth_fill_bf16):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


_tables_cache = {}


def _cdf_on_device(kind, sigma, device):
    key = (kind, sigma, str(device))
    if key not in _tables_cache:
        tab = e4m3_table() if kind == "e4m3" else bf16_table(sigma)
        thr = torch.from_numpy(np.concatenate([tab.thresholds, [0]]).astype(np.uint32).view(np.int32)).to(device)
        codes = torch.from_numpy(tab.codes.astype(np.uint16).view(np.int16)).to(device)
        _tables_cache[key] = (thr, codes, tab.n)
    return _tables_cache[key]


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"synth kernel launch failed: cudaError {rc}")


RECORD_BYTES = 272  # 256 e4m3 codes + fp32 scale at byte 256 + padding


def fill_tables(dst, seed, j0=0):
    """dst uint8 [nj, R, 256] or [nj, R, 272] (rows that carry their scale;
    call fill_record_scales too) -- CUDA or pinned CPU tensor."""
    nj, R, rb = dst.shape
    assert rb in (ROW_BYTES, RECORD_BYTES) and dst.dtype == torch.uint8 and dst.is_contiguous() and j0 + nj <= N_TABLES
    thr, codes, n = _cdf_on_device("e4m3", 1.0, "cuda")
    _check(_load().synth_fill_tables(ctypes.c_void_p(dst.data_ptr()), seed, j0, nj, R, rb,
                                     ctypes.c_void_p(thr.data_ptr()), ctypes.c_void_p(codes.data_ptr()), n, _stream()))


def fill_scales(dst, seed, j0=0):
    """dst float32 [nj, R]."""
    nj, R = dst.shape
    assert dst.dtype == torch.float32 and dst.is_contiguous()
    _check(_load().synth_fill_scales(ctypes.c_void_p(dst.data_ptr()), seed, j0, nj, R, 4, 0, _stream()))


def fill_record_scales(dst, seed, j0=0):
    """The fp32 scales into bytes 256..259 of each 272-byte row of dst."""
    nj, R, rb = dst.shape
    assert rb == RECORD_BYTES and dst.dtype == torch.uint8 and dst.is_contiguous()
    _check(_load().synth_fill_scales(ctypes.c_void_p(dst.data_ptr()), seed, j0, nj, R, RECORD_BYTES, ROW_BYTES,
                                     _stream()))


def fill_mx_scales(dst, seed, j0=0):
    """The eight E8M0 block scales into bytes 256..263 of each 272-byte row of
    dst (MXFP8-style rows: 256 e4m3 codes + one scale byte per 32 codes)."""
    nj, R, rb = dst.shape
    assert rb == RECORD_BYTES and dst.dtype == torch.uint8 and dst.is_contiguous()
    _check(_load().synth_fill_mx_scales(ctypes.c_void_p(dst.data_ptr()), seed, j0, nj, R, RECORD_BYTES, ROW_BYTES,
                                        _stream()))


def fill_bf16(dst, seed, stream, sigma, word0=0):
    """dst bfloat16 (any shape, contiguous): words word0.. of (seed, stream)."""
    assert dst.dtype == torch.bfloat16 and dst.is_contiguous()
    thr, codes, n = _cdf_on_device("bf16", float(sigma), "cuda")
    _check(_load().synth_fill_bf16(ctypes.c_void_p(dst.data_ptr()), seed, stream, word0, dst.numel(),
                                   ctypes.c_void_p(thr.data_ptr()), ctypes.c_void_p(codes.data_ptr()), n, _stream()))


def fill_h(dst, seed):
    """Residual h [T, d] bf16, N(0,1): word t*d + c (matches host.h_rows)."""
    fill_bf16(dst, seed, STREAM_H, 1.0)


def fill_w_out(dst, seed):
    fill_bf16(dst, seed, STREAM_W, W_SIGMA)


def fill_layer_weights(wq, wk, wm, seed, m):
    """Device twin of host.layer_weights for Engram layer m."""
    d = wq.shape[0]
    fill_bf16(wq, seed, STREAM_WQ + m, 1.0 / np.sqrt(d))
    fill_bf16(wk, seed, STREAM_WK + m, 1.0 / 16.0)
    fill_bf16(wm, seed, STREAM_WM + m, 1.0 / 16.0)


def fill_g(dst, seed):
    fill_bf16(dst, seed, STREAM_G, 1.0)
