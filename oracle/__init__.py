"""CPU oracle for the Engram memory read.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product path (the CUDA
library and its binding) never imports it and shares no code with it.

Thin numpy wrappers over ``oracle.c`` (plain C, double precision).  Each
function states the definition it computes; the C file cites the passages.
Functions with no independent pin would say "parity unpinned" here; every
function below is pinned by ``tests/test_oracle_pins.py``.
"""

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

N_TABLES = 48
ROW = 256
MEM = 512


def build(force=False):
    """Compile oracle.c into liboracle.so with gcc (plain C11, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm"]
        )
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int32
        lib.orc_mix_chain.restype = ctypes.c_uint64
        lib.orc_mix_chain.argtypes = [ctypes.c_uint64, P, ctypes.c_int]
        lib.orc_hash.restype = ctypes.c_int
        lib.orc_hash.argtypes = [P, P, i64, i32, i32, i64, P, P]
        lib.orc_hash_positions.restype = ctypes.c_int
        lib.orc_hash_positions.argtypes = [P, P, i64, i32, i64, P, P, i64, P]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.orc_gather_reduce_rows.restype = None
        lib.orc_gather_reduce_rows.argtypes = [P, P, i64, P]
        lib.orc_gather_reduce.restype = ctypes.c_int
        lib.orc_gather_reduce.argtypes = [P, P, i64, P, i64, P]
        lib.orc_e8m0_value.restype = ctypes.c_double
        lib.orc_e8m0_value.argtypes = [ctypes.c_uint8]
        lib.orc_gather_reduce_mx_rows.restype = None
        lib.orc_gather_reduce_mx_rows.argtypes = [P, P, i64, P]
        lib.orc_bf16_value.restype = ctypes.c_double
        lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_rne.restype = ctypes.c_uint16
        lib.orc_bf16_rne.argtypes = [ctypes.c_double]
        lib.orc_fuse.restype = ctypes.c_int
        lib.orc_fuse.argtypes = [P, P, P, P, i64, i32, ctypes.c_double, P]
        lib.orc_layer_gated.restype = ctypes.c_int
        lib.orc_layer_gated.argtypes = [P, P, P, P, P, P, i64, i32, ctypes.c_double, P, P]
        lib.orc_layer_gated_mx.restype = ctypes.c_int
        lib.orc_layer_gated_mx.argtypes = [P, P, P, P, P, P, i64, i32, ctypes.c_double, P, P]
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(st):
    if st != 0:
        raise OracleError(f"oracle status {st}")


def mix_chain(seed, ids):
    """h = seed; for id in ids (oldest first): h = (h ^ id) * 0x9E37..15; h ^= h >> 29."""
    a = np.ascontiguousarray(ids, dtype=np.uint64)
    return int(_load().orc_mix_chain(int(seed), _p(a), len(a)))


def hash_tokens(tokens, offs, last_n, V, R, seeds):
    """idx int64 [Tq, 48] for every query token."""
    lib = _load()
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    offs = np.ascontiguousarray(offs, dtype=np.int64)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    n_seqs = len(offs) - 1
    if last_n == 0:
        tq = int(offs[-1] - offs[0])
    else:
        tq = n_seqs * last_n
    idx = np.zeros((tq, N_TABLES), dtype=np.int64)
    _check(lib.orc_hash(_p(tokens), _p(offs), n_seqs, last_n, V, R, _p(seeds), _p(idx)))
    return idx


def hash_positions(tokens, offs, V, R, seeds, positions):
    """idx int64 [len(positions), 48] for explicit global positions."""
    lib = _load()
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    offs = np.ascontiguousarray(offs, dtype=np.int64)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    idx = np.zeros((len(pos), N_TABLES), dtype=np.int64)
    _check(lib.orc_hash_positions(_p(tokens), _p(offs), len(offs) - 1, V, R, _p(seeds), _p(pos), len(pos), _p(idx)))
    return idx


def e4m3_value(code):
    return _load().orc_e4m3_value(int(code))


def gather_reduce_rows(rows, scales):
    """mem float64 [T,512] from rows uint8 [T,48,256] and scales float32 [T,48]."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    T = rows.shape[0]
    assert rows.shape == (T, N_TABLES, ROW) and scales.shape == (T, N_TABLES)
    mem = np.zeros((T, MEM), dtype=np.float64)
    _load().orc_gather_reduce_rows(_p(rows), _p(scales), T, _p(mem))
    return mem


def e8m0_value(code):
    return _load().orc_e8m0_value(int(code))


def gather_reduce_mx_rows(rows, escales):
    """mem float64 [T,512] from MX rows: codes uint8 [T,48,256], E8M0 block scales uint8 [T,48,8]."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    escales = np.ascontiguousarray(escales, dtype=np.uint8)
    T = rows.shape[0]
    assert rows.shape == (T, N_TABLES, ROW) and escales.shape == (T, N_TABLES, 8)
    mem = np.zeros((T, MEM), dtype=np.float64)
    _load().orc_gather_reduce_mx_rows(_p(rows), _p(escales), T, _p(mem))
    return mem


def gather_reduce(tables, scales, idx):
    """mem float64 [T,512] from tables uint8 [48,R,256], scales float32 [48,R], idx [T,48]."""
    tables = np.ascontiguousarray(tables, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    R = tables.shape[1]
    T = idx.shape[0]
    mem = np.zeros((T, MEM), dtype=np.float64)
    _check(_load().orc_gather_reduce(_p(tables), _p(scales), R, _p(idx), T, _p(mem)))
    return mem


def bf16_value(bits):
    return _load().orc_bf16_value(int(bits))


def bf16_rne(x):
    return int(_load().orc_bf16_rne(float(x)))


def fuse(mem, W, g, h, eps=1e-6):
    """Gated projection: returns (h_new uint16 [T,d], gate float64 [T]).

    W uint16 [512,d], g uint16 [d], h uint16 [T,d] are bf16 bit patterns;
    h is not modified (a copy is updated)."""
    mem = np.ascontiguousarray(mem, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    g = np.ascontiguousarray(g, dtype=np.uint16)
    hn = np.array(h, dtype=np.uint16, copy=True, order="C")
    T, d = hn.shape
    gate = np.zeros(T, dtype=np.float64)
    _check(_load().orc_fuse(_p(mem), _p(W), _p(g), _p(hn), T, d, eps, _p(gate)))
    return hn, gate


def layer_gated(codes, scales, Wq, Wk, Wm, h, eps=1e-6):
    """One Engram layer with per-row content-aware gates (see oracle.c):
    returns (h_new uint16 [T,d], gates float64 [T,24], e float64 [T,256]).

    codes uint8 [T,24,256] and scales float32 [T,24] are the layer's 24 rows
    per token (MXFP8-style rows: scales uint8 [T,24,8], the E8M0 scale of each
    32-code block); Wq [d,256], Wk [256,256], Wm [256,d] and h [T,d] are bf16 bit
    patterns (h is not modified; a copy is updated)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    mx = np.asarray(scales).dtype == np.uint8
    scales = np.ascontiguousarray(scales, dtype=np.uint8 if mx else np.float32)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint16)
    Wk = np.ascontiguousarray(Wk, dtype=np.uint16)
    Wm = np.ascontiguousarray(Wm, dtype=np.uint16)
    hn = np.array(h, dtype=np.uint16, copy=True, order="C")
    T, d = hn.shape
    assert codes.shape == (T, 24, ROW) and scales.shape == ((T, 24, 8) if mx else (T, 24))
    assert Wq.shape == (d, ROW) and Wk.shape == (ROW, ROW) and Wm.shape == (ROW, d)
    gates = np.zeros((T, 24), dtype=np.float64)
    e = np.zeros((T, ROW), dtype=np.float64)
    f = _load().orc_layer_gated_mx if mx else _load().orc_layer_gated
    _check(f(_p(codes), _p(scales), _p(Wq), _p(Wk), _p(Wm), _p(hn), T, d, eps, _p(gates), _p(e)))
    return hn, gates, e
