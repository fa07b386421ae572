"""Python binding of libengram.so, the Engram memory read for one GB300.

Argument marshalling only: every step runs in the CUDA kernels of
``csrc/engram_core.cu``; PyTorch supplies device memory and streams.  The
names and semantics are those of ``include/engram.h``.  If the library has not
been built (``__graft_entry__.build()``), importing works but every call
raises: there is no CPU path.
"""

import ctypes
import os

import torch

from .buildlib import LIB_PATH, build  # noqa: F401

N_TABLES = 48
ROW_BYTES = 256
MEM_DIM = 512

STATUS = {
    0: "ENGRAM_OK",
    1: "ENGRAM_EINVAL",
    2: "ENGRAM_ECUDA",
    3: "ENGRAM_ERANGE",
    4: "ENGRAM_ECAPACITY",
    5: "ENGRAM_ETIMEOUT",
    6: "ENGRAM_ENOMEM",
    7: "ENGRAM_EUNSUPPORTED",
}


class EngramError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({engram_status_string(status)})")


class engram_config(ctypes.Structure):
    _fields_ = [
        ("vocab", ctypes.c_int32),
        ("d_model", ctypes.c_int32),
        ("rows", ctypes.c_int64),
        ("rms_eps", ctypes.c_float),
        ("row_layout", ctypes.c_uint32),
        ("seeds", ctypes.c_uint64 * N_TABLES),
    ]


ROWS_SEPARATE = 0  # tables [48][R][256] + scales [48][R]
ROWS_RECORD = 1  # tables [48][R][272]: 256 codes + fp32 scale at byte 256; no scales array
ROWS_MX = 2  # tables [48][R][272]: 256 codes + 8 E8M0 block scales at bytes 256..263; no scales array
RECORD_BYTES = 272


def make_config(vocab, rows, d_model, seeds, rms_eps=1e-6, row_layout=ROWS_SEPARATE):
    """An engram_config: V (pad id), R rows per table, d_model, 48 hash seeds, row layout."""
    c = engram_config()
    c.vocab = int(vocab)
    c.rows = int(rows)
    c.d_model = int(d_model)
    c.rms_eps = float(rms_eps)
    c.row_layout = int(row_layout)
    seeds = [int(s) for s in seeds]
    if len(seeds) != N_TABLES:
        raise ValueError("need 48 seeds")
    for j, s in enumerate(seeds):
        c.seeds[j] = s
    return c


_lib = None


def lib():
    """The loaded libengram.so (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libengram.so not built at {LIB_PATH}; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        C = ctypes.POINTER(engram_config)
        sig = {
            "engram_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "engram_last_error": ([], ctypes.c_int),
            "engram_wait_selftest": ([ctypes.c_uint64, P], ctypes.c_int),
            "engram_hash": ([C, P, P, i64, i32, i64, P, P], ctypes.c_int),
            "engram_gather_reduce": ([C, P, P, P, i64, P, P], ctypes.c_int),
            "engram_fuse": ([C, P, P, P, P, i64, P], ctypes.c_int),
            "engram_forward_workspace_bytes": ([C, i64], sz),
            "engram_forward": ([C, P, P, i64, i32, i64, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "engram_gather_x": ([C, P, P, i64, i32, i64, P, P, P, P], ctypes.c_int),
            "engram_fuse_x": ([C, P, P, P, P, i64, P], ctypes.c_int),
            "engram_shard_rows": ([C, i32], i64),
            "engram_host_cache_bytes": ([C, i64, i64], sz),
            "engram_host_cache_reset": ([C, P, i64, i64, P], ctypes.c_int),
            "engram_forward_host_cached_workspace_bytes": ([C, i64, i64], sz),
            "engram_forward_host_cached": (
                [C, P, P, i64, i32, i64, P, P, P, P, P, P, i64, i64, ctypes.c_uint32, P, sz, P, P, P, P, P],
                ctypes.c_int,
            ),
            "engram_gather_reduce_shard": ([C, i32, i32, P, P, i64, i32, i64, P, P, P, P], ctypes.c_int),
            "engram_forward_no_workspace": ([C, P, P, i64, i32, i64, P, P, P, P, P, P], ctypes.c_int),
            "engram_dedup_workspace_bytes": ([C], sz),
            "engram_dedup": ([C, P, i64, P, sz, P, i64, P, P, P], ctypes.c_int),
            "engram_stage": ([C, P, P, P, P, i64, P, P, P], ctypes.c_int),
            "engram_gather_reduce_staged": ([C, P, P, P, i64, i64, P, P], ctypes.c_int),
            "engram_forward_host_workspace_bytes": ([C, i64, i64], sz),
            "engram_forward_host": (
                [C, P, P, i64, i32, i64, P, P, P, P, P, i64, P, sz, P, P, P, P, P],
                ctypes.c_int,
            ),
            "engram_layer_keys": ([C, P, P, P], ctypes.c_int),
            "engram_layer_workspace_bytes": ([C, i64], sz),
            "engram_layer_forward": ([C, i32, P, P, i64, i32, i64, P, P, P, P, P, P, P, sz, P], ctypes.c_int),
            "engram_host_alloc": ([sz, ctypes.POINTER(P)], ctypes.c_int),
            "engram_host_free": ([P], ctypes.c_int),
            "engram_forward_host_pipelined_workspace_bytes": ([C, i64, i64, i64], sz),
            "engram_forward_host_pipelined": (
                [C, P, P, i64, i32, i64, P, P, P, P, P, i64, i64, P, sz, P, P, P, ctypes.POINTER(P)],
                ctypes.c_int,
            ),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def engram_status_string(status):
    return lib().engram_status_string(int(status)).decode()


def engram_last_error():
    """Sticky device error word of the current device as a status (clears it)."""
    return int(lib().engram_last_error())


def engram_wait_selftest(limit_ns, stream=None):
    """Enqueue the device-side time-limit check: a bounded wait that nothing
    satisfies runs out after limit_ns and sets ETIMEOUT (read it with
    engram_last_error())."""
    _check(lib().engram_wait_selftest(int(limit_ns), _stream(stream)), "engram_wait_selftest")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_rows(t, dtype, name):
    """Tables or scales for the HBM-path gathers: device memory, or pinned
    host memory read in place over unified addressing."""
    if t is not None and not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    _need(t, dtype, name, cuda=False)


def _need(t, dtype, name, cuda=True):
    if t is None and name in ("scales", "host_scales", "staged_scales"):
        return  # rows that carry their scales (ROWS_RECORD, ROWS_MX)
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _check(st, where):
    if st != 0:
        raise EngramError(st, where)


def _n_query(tokens, seq_offsets, last_n, n_query):
    if n_query is not None:
        return int(n_query)
    return tokens.numel() if last_n == 0 else (seq_offsets.numel() - 1) * last_n


def engram_hash(cfg, tokens, seq_offsets, last_n=0, n_query=None, idx=None, stream=None):
    """idx int64 [n_query, 48] (n_query defaults to all tokens, or n_seqs*last_n)."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    if idx is None:
        idx = torch.empty((nq, N_TABLES), dtype=torch.int64, device=tokens.device)
    _need(idx, torch.int64, "idx")
    _check(
        lib().engram_hash(ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq,
                          _ptr(idx), _stream(stream)),
        "engram_hash",
    )
    return idx


def engram_gather_reduce(cfg, tables, scales, idx, mem=None, stream=None):
    """mem fp32 [n_query, 512] from tables uint8 [48, R, 256], scales fp32 [48, R]."""
    _need_rows(tables, torch.uint8, "tables")
    _need_rows(scales, torch.float32, "scales")
    _need(idx, torch.int64, "idx")
    nq = idx.shape[0]
    if mem is None:
        mem = torch.empty((nq, MEM_DIM), dtype=torch.float32, device=idx.device)
    _need(mem, torch.float32, "mem")
    _check(
        lib().engram_gather_reduce(ctypes.byref(cfg), _ptr(tables), _ptr(scales), _ptr(idx), nq, _ptr(mem),
                                   _stream(stream)),
        "engram_gather_reduce",
    )
    return mem


def engram_fuse(cfg, mem, W_out, g, h, stream=None):
    """h (bf16 [n_query, d]) += gate * (bf16(mem) @ W_out), in place; returns h."""
    _need(mem, torch.float32, "mem")
    _need(W_out, torch.bfloat16, "W_out")
    _need(g, torch.bfloat16, "g")
    _need(h, torch.bfloat16, "h")
    _check(
        lib().engram_fuse(ctypes.byref(cfg), _ptr(mem), _ptr(W_out), _ptr(g), _ptr(h), h.shape[0], _stream(stream)),
        "engram_fuse",
    )
    return h


def engram_forward_workspace_bytes(cfg, n_query):
    return int(lib().engram_forward_workspace_bytes(ctypes.byref(cfg), int(n_query)))


def engram_forward(cfg, tokens, seq_offsets, tables, scales, W_out, g, h, last_n=0, n_query=None, workspace=None,
                   stream=None):
    """Hash + gather + fuse in one call (HBM tables); h updated in place."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need_rows(tables, torch.uint8, "tables")
    _need_rows(scales, torch.float32, "scales")
    _need(W_out, torch.bfloat16, "W_out")
    _need(g, torch.bfloat16, "g")
    _need(h, torch.bfloat16, "h")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    need = engram_forward_workspace_bytes(cfg, nq)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    _need(workspace, torch.uint8, "workspace")
    _check(
        lib().engram_forward(ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq,
                             _ptr(tables), _ptr(scales), _ptr(W_out), _ptr(g), _ptr(h), _ptr(workspace),
                             workspace.numel(), _stream(stream)),
        "engram_forward",
    )
    return h


LAYER_WIDTH = 256


def engram_layer_keys(cfg, W_k, W_kk=None, stream=None):
    """W_kk [512,256] = [W_k^T ; W_k^T] for the per-row gates of one Engram layer."""
    _need(W_k, torch.bfloat16, "W_k")
    if W_kk is None:
        W_kk = torch.empty((2 * LAYER_WIDTH, LAYER_WIDTH), dtype=torch.bfloat16, device=W_k.device)
    _check(lib().engram_layer_keys(ctypes.byref(cfg), _ptr(W_k), _ptr(W_kk), _stream(stream)), "engram_layer_keys")
    return W_kk


def engram_layer_workspace_bytes(cfg, n_query):
    return int(lib().engram_layer_workspace_bytes(ctypes.byref(cfg), int(n_query)))


def engram_layer_forward(cfg, module, tokens, seq_offsets, tables, scales, W_q, W_kk, W_m, h, last_n=0,
                         n_query=None, workspace=None, stream=None):
    """One Engram layer (module 0 or 1) with per-row gates, in place on h."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(tables, torch.uint8, "tables")
    _need(scales, torch.float32, "scales")
    _need(W_q, torch.bfloat16, "W_q")
    _need(W_kk, torch.bfloat16, "W_kk")
    _need(W_m, torch.bfloat16, "W_m")
    _need(h, torch.bfloat16, "h")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    if workspace is None:
        workspace = torch.empty(max(engram_layer_workspace_bytes(cfg, nq), 1), dtype=torch.uint8, device=h.device)
    _need(workspace, torch.uint8, "workspace")
    _check(
        lib().engram_layer_forward(ctypes.byref(cfg), int(module), _ptr(tokens), _ptr(seq_offsets),
                                   seq_offsets.numel() - 1, last_n, nq, _ptr(tables), _ptr(scales), _ptr(W_q),
                                   _ptr(W_kk), _ptr(W_m), _ptr(h), _ptr(workspace), workspace.numel(),
                                   _stream(stream)),
        "engram_layer_forward",
    )
    return h


def layer_workspace_views(workspace, n_query):
    """(q pair bf16 [n,512] = [q_hi | q_lo], u fp32 [n,256], X bf16 [n,256]) views
    of an engram_layer_forward workspace."""
    def up(x):
        return (x + 255) // 256 * 256

    n, w = n_query, LAYER_WIDTH
    ou = up(n * 2 * w * 2)
    ox = ou + up(n * w * 4)
    qp = workspace[: n * 2 * w * 2].view(torch.bfloat16).view(n, 2 * w)
    u = workspace[ou: ou + n * w * 4].view(torch.float32).view(n, w)
    X = workspace[ox: ox + n * w * 2].view(torch.bfloat16).view(n, w)
    return qp, u, X


def host_tables_empty(shape, dtype=torch.uint8):
    """A CPU tensor in pinned host memory on transparent huge pages (zeroed),
    from engram_host_alloc.  The tensor's storage holds the buffer object, so
    the memory is released once the last tensor or view of it is gone."""
    n = 1
    for x in shape:
        n *= int(x)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    ptr = ctypes.c_void_p()
    _check(lib().engram_host_alloc(nbytes, ctypes.byref(ptr)), "engram_host_alloc")

    class _HostBuffer(ctypes.c_uint8 * nbytes):
        def __del__(self):
            lib().engram_host_free(ctypes.c_void_p(ctypes.addressof(self)))

    buf = _HostBuffer.from_address(ptr.value)
    return torch.frombuffer(buf, dtype=torch.uint8).view(dtype).view(*shape)


def engram_forward_host_pipelined_workspace_bytes(cfg, n_query, chunk, capacity):
    return int(lib().engram_forward_host_pipelined_workspace_bytes(ctypes.byref(cfg), int(n_query), int(chunk),
                                                                   int(capacity)))


def engram_forward_host_pipelined(cfg, tokens, seq_offsets, host_tables, host_scales, W_out, g, h, chunk,
                                  capacity=None, last_n=0, n_query=None, workspace=None, n_unique=None, stream=None,
                                  side_stream=None, events=None):
    """The host-table path in chunks of `chunk` query tokens: chunk k+1's dedup
    and staging overlap chunk k's gather; one projection follows.  Returns
    n_unique (int64 per chunk).  `capacity` defaults to chunk * 48 rows per
    staging set."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(host_tables, torch.uint8, "host_tables", cuda=False)
    _need(host_scales, torch.float32, "host_scales", cuda=False)
    _need(h, torch.bfloat16, "h")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    dev = h.device
    chunk = int(min(chunk, max(nq, 1)))
    if capacity is None:
        capacity = chunk * N_TABLES
    if workspace is None:
        workspace = torch.empty(engram_forward_host_pipelined_workspace_bytes(cfg, nq, chunk, capacity),
                                dtype=torch.uint8, device=dev)
    n_chunks = max(1, -(-nq // chunk))
    if n_unique is None:
        n_unique = torch.zeros(n_chunks, dtype=torch.int64, device=dev)
    if side_stream is None:
        side_stream = torch.cuda.Stream(device=dev)
    if events is None:
        events = [torch.cuda.Event() for _ in range(6)]
    for ev in events:  # make sure the events exist as CUDA events before passing their handles
        if ev.cuda_event == 0:
            ev.record(torch.cuda.current_stream() if stream is None else stream)
    handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
    _check(
        lib().engram_forward_host_pipelined(
            ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq,
            _ptr(host_tables), _ptr(host_scales), _ptr(W_out), _ptr(g), _ptr(h), chunk, int(capacity),
            _ptr(workspace), workspace.numel(), _ptr(n_unique), _stream(stream),
            ctypes.c_void_p(side_stream.cuda_stream), handles),
        "engram_forward_host_pipelined",
    )
    return n_unique


NO_WORKSPACE_MAX_QUERY = 16384


def engram_forward_no_workspace(cfg, tokens, seq_offsets, tables, scales, W_out, g, h, last_n=0, n_query=None,
                                stream=None):
    """engram_forward with its scratch in the library's own device array (no
    workspace argument, nothing allocated): for callers that cannot allocate
    device memory.  At most NO_WORKSPACE_MAX_QUERY query tokens per call;
    calls that overlap on the GPU share the array and race."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(tables, torch.uint8, "tables")
    _need(scales, torch.float32, "scales")
    _need(W_out, torch.bfloat16, "W_out")
    _need(g, torch.bfloat16, "g")
    _need(h, torch.bfloat16, "h")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    _check(
        lib().engram_forward_no_workspace(ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1,
                                          last_n, nq, _ptr(tables), _ptr(scales), _ptr(W_out), _ptr(g), _ptr(h),
                                          _stream(stream)),
        "engram_forward_no_workspace",
    )
    return h


def engram_gather_x(cfg, tokens, seq_offsets, tables, scales, last_n=0, n_query=None, X=None, stream=None):
    """Hash in registers + gather + reduce: X bf16 [n_query, 512]."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need_rows(tables, torch.uint8, "tables")
    _need_rows(scales, torch.float32, "scales")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    if X is None:
        X = torch.empty((nq, MEM_DIM), dtype=torch.bfloat16, device=tokens.device)
    _need(X, torch.bfloat16, "X")
    _check(
        lib().engram_gather_x(ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq,
                              _ptr(tables), _ptr(scales), _ptr(X), _stream(stream)),
        "engram_gather_x",
    )
    return X


def engram_fuse_x(cfg, X, W_out, g, h, stream=None):
    """h += gate * (X @ W_out) from bf16 X [n_query, 512], in place; returns h."""
    _need(X, torch.bfloat16, "X")
    _need(W_out, torch.bfloat16, "W_out")
    _need(g, torch.bfloat16, "g")
    _need(h, torch.bfloat16, "h")
    _check(
        lib().engram_fuse_x(ctypes.byref(cfg), _ptr(X), _ptr(W_out), _ptr(g), _ptr(h), h.shape[0], _stream(stream)),
        "engram_fuse_x",
    )
    return h


def engram_shard_rows(cfg, n_shards):
    """Rows per table held by each of n_shards row shards: ceil(R / n_shards)."""
    return int(lib().engram_shard_rows(ctypes.byref(cfg), int(n_shards)))


def engram_gather_reduce_shard(cfg, shard, n_shards, tokens, seq_offsets, tables_shard, scales_shard, last_n=0,
                               n_query=None, mem=None, stream=None):
    """This row shard's partial module sums, fp32 [n_query, 512] (rows owned
    by other shards add nothing); the sum over shards is the whole mem."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(tables_shard, torch.uint8, "tables")
    _need(scales_shard, torch.float32, "scales")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    if mem is None:
        mem = torch.empty((nq, MEM_DIM), dtype=torch.float32, device=tokens.device)
    _need(mem, torch.float32, "mem")
    _check(
        lib().engram_gather_reduce_shard(ctypes.byref(cfg), int(shard), int(n_shards), _ptr(tokens),
                                         _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq, _ptr(tables_shard),
                                         _ptr(scales_shard), _ptr(mem), _stream(stream)),
        "engram_gather_reduce_shard",
    )
    return mem


def engram_host_cache_bytes(cfg, slots, capacity):
    """Bytes of a row cache of `slots` rows (a power of two) plus `capacity` overflow rows."""
    return int(lib().engram_host_cache_bytes(ctypes.byref(cfg), int(slots), int(capacity)))


def engram_host_cache_new(cfg, slots, capacity, device=None, stream=None):
    """A row cache on the device, reset (every slot empty)."""
    n = engram_host_cache_bytes(cfg, slots, capacity)
    if n == 0:
        raise ValueError("slots must be a power of two and capacity >= 1")
    cache = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check(lib().engram_host_cache_reset(ctypes.byref(cfg), _ptr(cache), int(slots), int(capacity), _stream(stream)),
           "engram_host_cache_reset")
    return cache


def engram_forward_host_cached_workspace_bytes(cfg, n_query, capacity):
    return int(lib().engram_forward_host_cached_workspace_bytes(ctypes.byref(cfg), n_query, capacity))


def engram_forward_host_cached(cfg, tokens, seq_offsets, host_tables, host_scales, W_out, g, h, cache, slots,
                               capacity, stamp, last_n=0, n_query=None, workspace=None, stats=None, stream=None,
                               side_stream=None, ev_dedup=None, ev_staged=None):
    """The host-table path with staged rows cached in HBM across calls.
    `stamp` must be larger than every earlier call's on this cache since its
    reset.  Returns stats int64 [4] on the device: distinct rows, cache hits,
    rows staged over the host link, rows staged outside the cache."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(host_tables, torch.uint8, "host_tables", cuda=False)
    _need(host_scales, torch.float32, "host_scales", cuda=False)
    _need(h, torch.bfloat16, "h")
    _need(cache, torch.uint8, "cache")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    dev = h.device
    if workspace is None:
        workspace = torch.empty(engram_forward_host_cached_workspace_bytes(cfg, nq, capacity), dtype=torch.uint8,
                                device=dev)
    if stats is None:
        stats = torch.zeros(4, dtype=torch.int64, device=dev)
    if side_stream is None:
        side_stream = torch.cuda.Stream(device=dev)
    ev_dedup = ev_dedup or torch.cuda.Event()
    ev_staged = ev_staged or torch.cuda.Event()
    for ev in (ev_dedup, ev_staged):
        if ev.cuda_event == 0:
            ev.record(torch.cuda.current_stream() if stream is None else stream)
    _check(
        lib().engram_forward_host_cached(
            ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq,
            _ptr(host_tables), _ptr(host_scales), _ptr(W_out), _ptr(g), _ptr(h), _ptr(cache), int(slots),
            int(capacity), int(stamp), _ptr(workspace), workspace.numel(), _ptr(stats), _stream(stream),
            ctypes.c_void_p(side_stream.cuda_stream), ctypes.c_void_p(ev_dedup.cuda_event),
            ctypes.c_void_p(ev_staged.cuda_event)),
        "engram_forward_host_cached",
    )
    return stats


def engram_dedup_workspace_bytes(cfg):
    return int(lib().engram_dedup_workspace_bytes(ctypes.byref(cfg)))


def engram_dedup(cfg, idx, capacity, workspace=None, unique=None, idx_staged=None, n_unique=None, stream=None):
    """Distinct (table,row) pairs of idx: returns (unique int64 [capacity],
    idx_staged int32 [n_query,48], n_unique int64 [1]) -- all on the device."""
    _need(idx, torch.int64, "idx")
    dev = idx.device
    nq = idx.shape[0]
    if workspace is None:
        workspace = torch.empty(engram_dedup_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    if unique is None:
        unique = torch.empty(capacity, dtype=torch.int64, device=dev)
    if idx_staged is None:
        idx_staged = torch.empty((nq, N_TABLES), dtype=torch.int32, device=dev)
    if n_unique is None:
        n_unique = torch.zeros(1, dtype=torch.int64, device=dev)
    _check(
        lib().engram_dedup(ctypes.byref(cfg), _ptr(idx), nq, _ptr(workspace), workspace.numel(), _ptr(unique),
                           int(capacity), _ptr(idx_staged), _ptr(n_unique), _stream(stream)),
        "engram_dedup",
    )
    return unique, idx_staged, n_unique


def engram_stage(cfg, host_tables, host_scales, unique, n_unique, capacity, staged_rows=None, staged_scales=None,
                 stream=None):
    """Copy the unique rows from pinned host tables into device staging buffers
    (256-byte rows + fp32 scales; whole 272-byte rows for ROWS_MX, scales None)."""
    _need(host_tables, torch.uint8, "host_tables", cuda=False)
    _need(host_scales, torch.float32, "host_scales", cuda=False)
    if not (host_tables.is_pinned() and (host_scales is None or host_scales.is_pinned())):
        raise ValueError("host tables and scales must be in pinned host memory")
    dev = unique.device
    mx = cfg.row_layout == ROWS_MX  # MX rows are staged whole, with no scale array
    if staged_rows is None:
        staged_rows = torch.empty((capacity, RECORD_BYTES if mx else ROW_BYTES), dtype=torch.uint8, device=dev)
    if staged_scales is None and not mx:
        staged_scales = torch.empty(capacity, dtype=torch.float32, device=dev)
    _check(
        lib().engram_stage(ctypes.byref(cfg), _ptr(host_tables), _ptr(host_scales), _ptr(unique), _ptr(n_unique),
                           int(capacity), _ptr(staged_rows), _ptr(staged_scales), _stream(stream)),
        "engram_stage",
    )
    return staged_rows, staged_scales


def engram_gather_reduce_staged(cfg, staged_rows, staged_scales, idx_staged, mem=None, stream=None):
    _need(staged_rows, torch.uint8, "staged_rows")
    _need(staged_scales, torch.float32, "staged_scales")
    _need(idx_staged, torch.int32, "idx_staged")
    nq = idx_staged.shape[0]
    if mem is None:
        mem = torch.empty((nq, MEM_DIM), dtype=torch.float32, device=idx_staged.device)
    _check(
        lib().engram_gather_reduce_staged(ctypes.byref(cfg), _ptr(staged_rows), _ptr(staged_scales),
                                          _ptr(idx_staged), nq, staged_rows.shape[0], _ptr(mem), _stream(stream)),
        "engram_gather_reduce_staged",
    )
    return mem


def engram_forward_host_workspace_bytes(cfg, n_query, capacity):
    return int(lib().engram_forward_host_workspace_bytes(ctypes.byref(cfg), int(n_query), int(capacity)))


def engram_forward_host(cfg, tokens, seq_offsets, host_tables, host_scales, W_out, g, h, capacity, last_n=0,
                        n_query=None, workspace=None, n_unique=None, stream=None, side_stream=None, ev_dedup=None,
                        ev_staged=None):
    """The host-table path: hash + dedup on `stream`, row staging on
    `side_stream`, staged gather + fuse back on `stream`.  Returns n_unique."""
    _need(tokens, torch.int32, "tokens")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(host_tables, torch.uint8, "host_tables", cuda=False)
    _need(host_scales, torch.float32, "host_scales", cuda=False)
    _need(h, torch.bfloat16, "h")
    nq = _n_query(tokens, seq_offsets, last_n, n_query)
    dev = h.device
    if workspace is None:
        workspace = torch.empty(engram_forward_host_workspace_bytes(cfg, nq, capacity), dtype=torch.uint8, device=dev)
    if n_unique is None:
        n_unique = torch.zeros(1, dtype=torch.int64, device=dev)
    if side_stream is None:
        side_stream = torch.cuda.Stream(device=dev)
    ev_dedup = ev_dedup or torch.cuda.Event()
    ev_staged = ev_staged or torch.cuda.Event()
    # make sure the events exist as CUDA events before passing their handles
    for ev in (ev_dedup, ev_staged):
        if ev.cuda_event == 0:
            ev.record(torch.cuda.current_stream() if stream is None else stream)
    _check(
        lib().engram_forward_host(
            ctypes.byref(cfg), _ptr(tokens), _ptr(seq_offsets), seq_offsets.numel() - 1, last_n, nq,
            _ptr(host_tables), _ptr(host_scales), _ptr(W_out), _ptr(g), _ptr(h), int(capacity), _ptr(workspace),
            workspace.numel(), _ptr(n_unique), _stream(stream), ctypes.c_void_p(side_stream.cuda_stream),
            ctypes.c_void_p(ev_dedup.cuda_event), ctypes.c_void_p(ev_staged.cuda_event)),
        "engram_forward_host",
    )
    return n_unique
