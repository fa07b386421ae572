"""Checks of GPU results against the oracle on every query token, spread over
the host's cores by a pool of spawned worker processes (no fork after CUDA
initialisation).  Workers rebuild each token's inputs from the host twins of
the seeded generators and run the oracle; nothing in here touches the GPU or
the CUDA library.  Used by the tests only.
"""

import multiprocessing as mp
import os
import time

import numpy as np

import oracle
from synth import host

H_TOL = 2e-2   # max |gpu - ref| / max(1, |ref|) on the fused residual
MEM_TOL = 1e-5  # |gpu - ref| <= MEM_TOL * sum_j |term_j| on the module sums

_W = {}


def _init(seed, d, eps, V, R, seeds, tok, offs, qpos):
    _W.update(seed=seed, d=d, eps=eps, V=V, R=R, seeds=seeds, tok=tok, offs=offs, qpos=qpos,
              W=host.w_out(seed, d), g=host.g_vec(seed, d))


def _bf16_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def reference(q):
    """Oracle (mem, sum_j |term_j|, h bits) for query tokens q, from host-twin inputs."""
    w = _W
    q = np.asarray(q, np.int64)
    idx = oracle.hash_positions(w["tok"], w["offs"], w["V"], w["R"], w["seeds"], w["qpos"][q])
    jj = np.tile(np.arange(48), len(q))
    rows = host.table_rows(w["seed"], jj, idx.reshape(-1)).reshape(len(q), 48, 256)
    sc = host.scales(w["seed"], jj, idx.reshape(-1)).reshape(len(q), 48)
    mem = oracle.gather_reduce_rows(rows, sc)
    bound = oracle.gather_reduce_rows(rows & 0x7F, sc)
    hn, _ = oracle.fuse(mem, w["W"], w["g"], host.h_rows(w["seed"], w["d"], q), w["eps"])
    return mem, bound, hn


def _check_chunk(job):
    q, gpu_mem, gpu_h = job
    mem, bound, hn = reference(q)
    mem_ratio = np.abs(np.asarray(gpu_mem, np.float64) - mem) / np.maximum(bound, 1e-30)
    g, r = _bf16_f64(gpu_h), _bf16_f64(hn)
    h_rel = np.abs(g - r) / np.maximum(1.0, np.abs(r))
    return len(q), float(mem_ratio.max()), float(h_rel.max()), int((mem_ratio > MEM_TOL).sum()), int((h_rel > H_TOL).sum())


def check_all_tokens(cfg, seeds, tok, offs, qpos, gpu_mem, gpu_h, chunk=512, procs=None):
    """Compare gpu_mem float32 [Tq,512] and gpu_h bf16 bits uint16 [Tq,d] with
    the oracle on every query token.  Returns a summary dict; the caller asserts."""
    tq = gpu_h.shape[0]
    procs = procs or os.cpu_count() or 1
    oracle.build()
    jobs = ((np.arange(a, min(a + chunk, tq)), gpu_mem[a:a + chunk], gpu_h[a:a + chunk]) for a in range(0, tq, chunk))
    t0 = time.time()
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_init,
                  initargs=(cfg.seed, cfg.d, cfg.rms_eps, cfg.V, cfg.R, seeds, tok, offs, qpos)) as pool:
        res = list(pool.imap_unordered(_check_chunk, jobs))
    secs = time.time() - t0
    return {
        "tokens": sum(r[0] for r in res),
        "mem_worst": max(r[1] for r in res),
        "h_worst": max(r[2] for r in res),
        "mem_bad": sum(r[3] for r in res),
        "h_bad": sum(r[4] for r in res),
        "seconds": secs,
        "procs": procs,
    }


# ------------------------------------------------- the per-layer form -------

def _init_layer(seed, d, eps, V, R, seeds, tok, offs, qpos, module):
    wq, wk, wm = host.layer_weights(seed, d, module)
    lut = np.array([abs(oracle.e4m3_value(c)) if c not in (0x7F, 0xFF) else 0.0 for c in range(256)])
    _W.update(seed=seed, d=d, eps=eps, V=V, R=R, seeds=seeds, tok=tok, offs=offs, qpos=qpos, module=module,
              wq=wq, wk=wk, wm=wm, abs_lut=lut)


def _check_layer_chunk(job):
    q, h_in, h_gpu, x_gpu = job
    w = _W
    m = w["module"]
    q = np.asarray(q, np.int64)
    idx = oracle.hash_positions(w["tok"], w["offs"], w["V"], w["R"], w["seeds"], w["qpos"][q])
    jj = np.tile(np.arange(24 * m, 24 * m + 24), len(q))
    r = idx[:, 24 * m:24 * m + 24].reshape(-1)
    codes = host.table_rows(w["seed"], jj, r).reshape(len(q), 24, 256)
    sc = host.scales(w["seed"], jj, r).reshape(len(q), 24)
    hn, _, e = oracle.layer_gated(codes, sc, w["wq"], w["wk"], w["wm"], h_in, w["eps"])
    bound = (w["abs_lut"][codes] * sc[:, :, None].astype(np.float64)).sum(axis=1)  # sum_j |r_j|
    g, ref = _bf16_f64(h_gpu), _bf16_f64(hn)
    h_rel = np.abs(g - ref) / np.maximum(1.0, np.abs(ref))
    x_err = np.abs(_bf16_f64(x_gpu) - e)
    x_bad = x_err > 1e-3 * bound + 2.0**-8 * np.abs(e) + 1e-30
    return len(q), float(h_rel.max()), int((h_rel > H_TOL).sum()), int(x_bad.sum())


def check_layer_all_tokens(cfg, seeds, tok, offs, qpos, module, h_in, h_gpu, x_gpu, chunk=256, procs=None):
    """One Engram layer on every query token: h_gpu (bf16 bits [Tq,d]) against
    the oracle applied to h_in (the GPU's h before the layer), and the
    layer's X (bf16 bits [Tq,256]) against the oracle's gated sum.  Returns a
    summary dict; the caller asserts."""
    tq = h_gpu.shape[0]
    procs = procs or os.cpu_count() or 1
    oracle.build()
    jobs = ((np.arange(a, min(a + chunk, tq)), h_in[a:a + chunk], h_gpu[a:a + chunk], x_gpu[a:a + chunk])
            for a in range(0, tq, chunk))
    t0 = time.time()
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_init_layer,
                  initargs=(cfg.seed, cfg.d, cfg.rms_eps, cfg.V, cfg.R, seeds, tok, offs, qpos, module)) as pool:
        res = list(pool.imap_unordered(_check_layer_chunk, jobs))
    return {"tokens": sum(r[0] for r in res), "h_worst": max(r[1] for r in res), "h_bad": sum(r[2] for r in res),
            "x_bad": sum(r[3] for r in res), "seconds": time.time() - t0, "procs": procs}
