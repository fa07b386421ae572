"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and validates arguments before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "engram.h")


@pytest.fixture(scope="module")
def eg():
    import engram_gram_hash_gb300 as eg
    eg.build()
    eg.lib()
    return eg


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(engram_[a-z_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ["engram_hash", "engram_gather_reduce", "engram_fuse", "engram_forward", "engram_dedup",
              "engram_stage", "engram_gather_reduce_staged", "engram_forward_host", "engram_last_error",
              "engram_status_string"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(eg):
    lib = ctypes.CDLL(eg.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in engram.h but not exported"


def test_status_strings(eg):
    for k in range(8):
        assert eg.engram_status_string(k)
    assert eg.engram_status_string(0) == "ok"


def test_workspace_sizes(eg):
    from synth.configs import CONFIGS, default_seeds

    cfg = CONFIGS["large"]
    c = eg.make_config(cfg.V, cfg.R, cfg.d, default_seeds())
    ws = eg.engram_forward_workspace_bytes(c, cfg.tq)
    assert ws >= cfg.tq * 512 * 2  # the bf16 X between the two kernels
    d = eg.engram_dedup_workspace_bytes(c)
    assert d >= 2 * 48 * cfg.R // 32 * 4
    assert eg.engram_forward_host_workspace_bytes(c, 100, 4800) >= 4800 * 256
    # the pipelined host path: two staging sets, each sized by the chunk
    p1 = eg.engram_forward_host_pipelined_workspace_bytes(c, 65536, 8192, 8192 * 48)
    p2 = eg.engram_forward_host_pipelined_workspace_bytes(c, 65536, 16384, 16384 * 48)
    assert p2 - p1 >= 2 * 8192 * 48 * 256 and eg.engram_forward_host_pipelined_workspace_bytes(c, 100, 0, 10) == 0
    # MX rows are staged whole: 272 bytes a staged row
    cm = eg.make_config(cfg.V, cfg.R, cfg.d, default_seeds(), row_layout=eg.ROWS_MX)
    assert eg.engram_forward_host_workspace_bytes(cm, 100, 4800) >= 4800 * 272


def test_invalid_arguments_rejected_before_any_device_work(eg):
    lib = eg.lib()
    from synth.configs import default_seeds

    c = eg.make_config(1024, 4096, 256, default_seeds())
    null = ctypes.c_void_p(0)
    # null config
    assert lib.engram_hash(None, null, null, 1, 0, 10, null, null) == 1
    # null buffers with work to do
    assert lib.engram_hash(ctypes.byref(c), null, null, 1, 0, 10, null, null) == 1
    assert lib.engram_gather_reduce(ctypes.byref(c), null, null, null, 10, null, null) == 1
    # d not a multiple of 256
    c2 = eg.make_config(1024, 4096, 200, default_seeds())
    assert lib.engram_fuse(ctypes.byref(c2), ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
                           ctypes.c_void_p(256), 4, null) == 1
    # d above the widest split (8 CTAs of 16 chunks of 256 columns), and d = 0
    for d_bad in (32768 + 256, 0):
        cw = eg.make_config(1024, 4096, d_bad, default_seeds())
        assert lib.engram_fuse(ctypes.byref(cw), ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
                               ctypes.c_void_p(256), 4, null) == 1, d_bad
    # R < 1
    c3 = eg.make_config(1024, 0, 256, default_seeds())
    assert lib.engram_gather_reduce(ctypes.byref(c3), ctypes.c_void_p(256), ctypes.c_void_p(256),
                                    ctypes.c_void_p(256), 4, ctypes.c_void_p(256), null) == 1
    # pipelined host path: chunk < 1, null events
    ev6 = (ctypes.c_void_p * 6)(*([256] * 6))
    assert lib.engram_forward_host_pipelined(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), 1, 0, 4,
                                             ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
                                             ctypes.c_void_p(256), ctypes.c_void_p(256), 0, 64,
                                             ctypes.c_void_p(256), 1 << 30, ctypes.c_void_p(256), null, null,
                                             ev6) == 1
    assert lib.engram_forward_host_pipelined(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), 1, 0, 4,
                                             ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
                                             ctypes.c_void_p(256), ctypes.c_void_p(256), 4, 64,
                                             ctypes.c_void_p(256), 1 << 30, ctypes.c_void_p(256), null, null,
                                             None) == 1
    # host table allocator: zero bytes or a null out-pointer; freeing a foreign pointer
    out = ctypes.c_void_p()
    assert lib.engram_host_alloc(0, ctypes.byref(out)) == 1 and lib.engram_host_alloc(64, None) == 1
    assert lib.engram_host_free(ctypes.c_void_p(4096)) == 1 and lib.engram_host_free(None) == 0
    # unknown row layout
    c4 = eg.make_config(1024, 4096, 256, default_seeds(), row_layout=3)
    assert lib.engram_gather_reduce(ctypes.byref(c4), ctypes.c_void_p(256), ctypes.c_void_p(256),
                                    ctypes.c_void_p(256), 4, ctypes.c_void_p(256), null) == 1
    # MX rows: a null scales array is accepted, a null staging buffer is not
    c5 = eg.make_config(1024, 4096, 256, default_seeds(), row_layout=eg.ROWS_MX)
    assert lib.engram_gather_reduce_staged(ctypes.byref(c5), null, null, ctypes.c_void_p(256), 4, 16,
                                           ctypes.c_void_p(256), null) == 1
    # zero queries is a no-op that succeeds
    assert lib.engram_hash(ctypes.byref(c), null, null, 1, 0, 0, null, null) == 0
    assert lib.engram_gather_reduce(ctypes.byref(c), null, null, null, 0, null, null) == 0
    # workspace too small
    assert lib.engram_dedup(ctypes.byref(c), ctypes.c_void_p(256), 4, ctypes.c_void_p(256), 16,
                            ctypes.c_void_p(256), 100, ctypes.c_void_p(256), ctypes.c_void_p(256), null) == 6
    # row cache: slots must be a power of two; a call needs a stamp >= 1
    assert lib.engram_host_cache_bytes(ctypes.byref(c), 1000, 10) == 0
    assert lib.engram_host_cache_bytes(ctypes.byref(c), 1024, 10) >= 1034 * 260
    assert lib.engram_host_cache_reset(ctypes.byref(c), ctypes.c_void_p(256), 1000, 10, null) == 1
    p256 = ctypes.c_void_p(256)
    assert lib.engram_forward_host_cached(ctypes.byref(c), p256, p256, 1, 0, 4, p256, p256, p256, p256, p256, p256,
                                          1024, 10, 0, p256, 1 << 30, p256, null, null, p256, p256) == 1
    # no-workspace entry: a malformed call is EINVAL even when it is also too large;
    # a well-formed call past the scratch limit is ENOMEM (both before any device work)
    big = 16384 + 1
    p = ctypes.c_void_p(256)
    assert lib.engram_forward_no_workspace(ctypes.byref(c), null, p, 1, 0, big, p, p, p, p, p, null) == 1
    assert lib.engram_forward_no_workspace(ctypes.byref(c), p, p, 1, 0, big, p, p, p, p, p, null) == 6


def test_layer_entry_points_check_arguments_before_device_work(eg):
    """engram_layer_keys / engram_layer_forward reject bad arguments with a
    status before any CUDA call (the fake pointers below are never touched)."""
    lib = eg.lib()
    from synth.configs import default_seeds

    P = ctypes.c_void_p
    a = P(256)  # aligned stand-in, never dereferenced
    c = eg.make_config(1024, 4096, 256, default_seeds())
    assert lib.engram_layer_keys(ctypes.byref(c), None, a, None) == 1
    assert lib.engram_layer_keys(ctypes.byref(c), P(258), a, None) == 1  # misaligned W_k
    n = 1000
    assert eg.engram_layer_workspace_bytes(c, n) >= n * (512 * 2 + 256 * 4 + 256 * 2)

    def fwd(cfg, module=0, n_seqs=1, last_n=0, n_query=4, tables=a, ws_bytes=1 << 30):
        return lib.engram_layer_forward(ctypes.byref(cfg), module, a, a, n_seqs, last_n, n_query, tables, a, a, a, a,
                                        a, a, ws_bytes, None)

    assert fwd(c, module=2) == 1                        # module 0 or 1
    assert fwd(c, n_query=0) == 0                       # nothing to do
    assert fwd(c, tables=None) == 1                     # null tables
    assert fwd(c, n_seqs=2, last_n=1, n_query=4) == 1   # n_query != n_seqs * last_n
    assert fwd(c, ws_bytes=16) == 6                     # workspace too small
    c_mx = eg.make_config(1024, 4096, 256, default_seeds(), row_layout=eg.ROWS_MX)
    assert fwd(c_mx, ws_bytes=16) == 6                  # MX rows: checked the same way (no device work)
    assert fwd(c_mx, module=2) == 1
    c_d = eg.make_config(1024, 4096, 320, default_seeds())
    assert fwd(c_d) == 1                                # d not a multiple of 256


def test_product_path_does_not_import_the_oracle():
    """The binding and the CUDA sources never reference oracle/."""
    pkg = os.path.join(ROOT, "engram_gram_hash_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt and "oracle.c" not in txt, f


def test_wait_selftest_checks_its_limit_before_device_work(eg):
    """engram_wait_selftest rejects a zero or over-long limit with EINVAL and
    enqueues nothing (no GPU is touched here)."""
    lib = eg.lib()
    assert lib.engram_wait_selftest(0, None) == 1
    assert lib.engram_wait_selftest(10**10 + 1, None) == 1


def test_empty_batches_are_no_ops_before_device_work(eg):
    """n_query = 0 returns ENGRAM_OK from every batch entry point, with null
    buffers and without touching the device (this machine may have none)."""
    lib = eg.lib()
    from synth.configs import default_seeds

    c = ctypes.byref(eg.make_config(1024, 4096, 4096, default_seeds()))
    P, I64, I32, SZ, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_uint32
    n, z = P(0), I64(0)
    calls = {
        "engram_hash": (c, n, n, I64(1), I32(0), z, n, n),
        "engram_gather_reduce": (c, n, n, n, z, n, n),
        "engram_fuse": (c, n, n, n, n, z, n),
        "engram_fuse_x": (c, n, n, n, n, z, n),
        "engram_forward": (c, n, n, I64(1), I32(0), z, n, n, n, n, n, n, SZ(0), n),
        "engram_forward_no_workspace": (c, n, n, I64(1), I32(0), z, n, n, n, n, n, n),
        "engram_gather_x": (c, n, n, I64(1), I32(0), z, n, n, n, n),
        "engram_gather_reduce_shard": (c, I32(0), I32(2), n, n, I64(1), I32(0), z, n, n, n, n),
        "engram_gather_reduce_staged": (c, n, n, n, z, I64(1), n, n),
        "engram_layer_forward": (c, I32(1), n, n, I64(1), I32(0), z, n, n, n, n, n, n, n, SZ(0), n),
        "engram_forward_host": (c, n, n, I64(1), I32(0), z, n, n, n, n, n, I64(1), n, SZ(0), n, n, n, n, n),
        "engram_forward_host_pipelined": (c, n, n, I64(1), I32(0), z, n, n, n, n, n, I64(64), I64(1), n, SZ(0), n,
                                          n, n, n),
        "engram_forward_host_cached": (c, n, n, I64(1), I32(0), z, n, n, n, n, n, n, I64(1 << 10), I64(1 << 10),
                                       U32(1), n, SZ(0), n, n, n, n, n),
    }
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for name, args in calls.items():
        decl = re.search(r"\b" + name + r"\s*\(([^;]*)\);", src)
        assert decl and len(decl.group(1).split(",")) == len(args), name  # one value per declared parameter
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        assert f(*args) == 0, name
