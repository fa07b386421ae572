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
