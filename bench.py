"""Benchmark of the Engram memory read (hash + gather + fuse) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole path over one batch of the workload:
engram_gather_x (n-gram hash in registers + row gather + dequant + module
sums -> bf16 X) then engram_fuse_x (tcgen05 projection + gated residual
update, h in place) through the C ABI -- the two kernels engram_forward
launches, called separately so each is timed with CUDA events.  The
host-table workload runs engram_forward_host (hash, dedup, staging from
pinned host memory on a side stream, staged gather, projection).  Inputs are
resident in HBM when the timed region starts and are larger than L2 (tables
of 13-103 GB, h of 0.5-2 GB), so no L2 flush is needed between steps.

Prints ONE JSON line (rank 0).  For N > 1 (torchrun, one rank per GPU) every
rank runs its own batch of the workload on replicated tables: the path
shards over tokens with no collective ("weak" scaling).

--impl reference times the CPU oracle (the plain C definition) on the host
cores over a bounded sample of the same workload and prints the same line.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Engram tokens/sec (hash+gather+fuse) and achieved GB/s vs HBM/host-link roofline"
UNIT = "tokens/s"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# Algorithmic bytes per query token (what the method must move, as the
# measurement plan counts them): 48 rows of 256 code bytes plus their scales
# for the gather, the residual read and write (4 d bytes) for the projection.
# The bf16 X handed between the two kernels (1 KB each way), the token id and
# the scale bytes fetched beyond the 4 used are reported apart.
def kernel_bytes_per_token(d, layout="separate"):
    """Algorithmic bytes per query token of each kernel: the gather reads 48
    rows of 256 code bytes plus their scales (one fp32, or eight E8M0 bytes
    for MX rows); the projection reads and writes the bf16 residual h."""
    scale = 8 if layout == "mx" else 4
    return {"gather": 48 * (256 + scale), "fuse": 4 * d}


def handoff_bytes_per_token():
    """Bytes per query token outside the method's count: the bf16 X written by
    the gather and read by the projection, and the token id."""
    return {"X_write": 512 * 2, "X_read": 512 * 2, "token": 4}


def nominal_bytes_per_token(d):
    """The path's nominal bytes: 48 rows of 256 B plus the residual read and write."""
    return 48 * 256 + 4 * d


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal, for context beside the measured copy peak


def _code_only(src):
    """C/C++/CUDA source without comments and blank-line or spacing changes,
    so that the hash below moves only when the code does (string literals
    containing comment markers are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(" ".join(line.split()) for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash():
    """sha256 prefix of the kernel sources' code (comments and spacing aside):
    the DRAM-traffic figures under profiles/ are used only while it matches."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "engram_gram_hash_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload, units, layout="separate"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    if there is none for this workload, row layout and the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")  # JSON text
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {})
    if e.get("source_hash") != kernel_source_hash() or "bytes_per_token" not in e:
        return None
    if e.get("workload") != workload or e.get("layout", "separate") != layout:
        return None
    return e["bytes_per_token"] * units


def smi_index(local_rank):
    """nvidia-smi's name for this rank's GPU (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        items = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(items):
            return items[local_rank]
    return str(local_rank)


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver): SM clock, its maximum, and the active clock-event reasons."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(int(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML device")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct = self.ct
        mhz, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz))  # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.reasons_fn(self.h, ct.byref(rs))
        return time.time(), float(mhz.value), float(mx.value), [n for b, n in self.REASONS.items() if rs.value & b]


class ClockSampler:
    """SM clocks and throttle reasons sampled during the timed region: every
    2 ms through NVML in a thread (read-only queries), or every 100 ms from
    nvidia-smi where NVML cannot be loaded."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_s=0.002):
        self.gpu = gpu_index
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.rows = []
        self.path = os.path.join("/tmp", f"engram_clocks_{os.getpid()}.csv")
        self.t_start = self.t_end = None

    def _loop(self):
        while not self._stop.is_set():
            try:
                self.rows.append(self.nvml.sample())
            except OSError:
                break
            self._stop.wait(self.period)

    def __enter__(self):
        import threading

        try:
            self.nvml = _Nvml(self.gpu)
            self._stop = threading.Event()
            self._thr = threading.Thread(target=self._loop, daemon=True)
            self._thr.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while os.path.getsize(self.path) == 0 and time.time() - t0 < 5:  # sampler is up before timing
                time.sleep(0.05)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *a):
        if self.nvml is not None:
            self._stop.set()
            self._thr.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def _smi_rows(self):
        from datetime import datetime

        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]),
                                 [nm for nm, v in zip(names, parts[5:9]) if v.lower() == "active"]))
                except ValueError:
                    continue
        os.unlink(self.path)
        return rows

    def summary(self):
        if self.nvml is not None:
            rows, src = self.rows, "nvml every 2 ms"
        elif self.proc is not None and os.path.exists(self.path):
            rows, src = self._smi_rows(), "nvidia-smi every 100 ms"
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": src}
        window = "timed region"
        sel = [r for r in rows if self.t_start is not None and self.t_start - 0.002 <= r[0] <= self.t_end + 0.002]
        if len(sel) < 2:  # a timed region shorter than the sampling period: use the nearest samples
            window = "timed region shorter than the sampling period; samples nearest to it"
            mid = 0.5 * (self.t_start + self.t_end) if self.t_start else rows[-1][0]
            sel = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
        reasons = sorted({x for r in sel for x in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "sm_mhz_min": min(r[1] for r in sel), "reasons": reasons, "samples": len(sel), "window": window,
                "source": src}


# ------------------------------------------------------ multi-rank pieces ----


def rank_config(base, rank):
    """Rank r's workload under weak scaling: the same tables (the model's
    weights, replicated), its own token batch and residual (seed + 1000 r)."""
    return base if rank == 0 else base.with_(seed=base.seed + 1000 * rank)


def job_rate(local_ms, steps, units_per_rank, world, device):
    """Whole-job throughput: every rank's units over the slowest rank's time.
    Returns (units per second, max ms over ranks)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return units_per_rank * world / (ms_max * 1e-3 / steps), ms_max


# --------------------------------------------------------------- our arm ----


def time_forward_graph(eg, c, cfg, nq, tokens, seq_offsets, tables, scales, W, g, h, dev, reps):
    """engram_forward per step, launched eagerly and replayed from a CUDA graph
    (the same calls captured once); microseconds per step."""
    import torch

    ws = torch.empty(max(eg.engram_forward_workspace_bytes(c, nq), 1), dtype=torch.uint8, device=dev)

    def fwd():
        eg.engram_forward(c, tokens, seq_offsets, tables, scales, W, g, h, last_n=cfg.last_n, n_query=nq,
                          workspace=ws)

    for _ in range(3):
        fwd()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fwd()
    b.record()
    torch.cuda.synchronize()
    eager_us = a.elapsed_time(b) / reps * 1e3
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    graph_us = a.elapsed_time(b) / reps * 1e3
    # As one segment of a larger forward graph: SEQ dependent steps captured
    # in one graph (each reads the h the previous step wrote), so the graph
    # launch itself is paid once per SEQ steps rather than once per step.
    SEQ = 10
    graph_seq = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_seq):
        for _ in range(SEQ):
            fwd()
    for _ in range(3):
        graph_seq.replay()
    torch.cuda.synchronize()
    seq_reps = max(1, reps // SEQ)
    a.record()
    for _ in range(seq_reps):
        graph_seq.replay()
    b.record()
    torch.cuda.synchronize()
    seq_us = a.elapsed_time(b) / (seq_reps * SEQ) * 1e3
    if eg.engram_last_error() != 0:
        raise RuntimeError("device error in the CUDA-graph timing")
    return {"api": "engram_forward (hash + gather + fuse, 2 kernels)", "eager_us_per_step": round(eager_us, 2),
            "graph_us_per_step": round(graph_us, 2), "steps": reps,
            f"graph_{SEQ}_dependent_steps_us_per_step": round(seq_us, 2),
            "graph_note": f"graph_us_per_step: one step per graph replay; graph_{SEQ}_dependent_steps: {SEQ} steps "
                          "captured in one graph, each reading the h the previous one wrote (the graph launch "
                          f"paid once per {SEQ} steps, as for a segment of a model's forward graph)"}


def time_host_pipelined(eg, c, cfg, nq, tokens, seq_offsets, tables, scales, W, g, h, dev, chunk, steps):
    """The chunked, pipelined host-table forward: ms per step and rows staged."""
    import torch

    cap = chunk * 48
    ws = torch.empty(eg.engram_forward_host_pipelined_workspace_bytes(c, nq, chunk, cap), dtype=torch.uint8,
                     device=dev)
    n_unique = torch.zeros(-(-nq // chunk), dtype=torch.int64, device=dev)
    side = torch.cuda.Stream(device=dev)
    events = [torch.cuda.Event() for _ in range(6)]

    def fwd():
        eg.engram_forward_host_pipelined(c, tokens, seq_offsets, tables, scales, W, g, h, chunk, capacity=cap,
                                         last_n=cfg.last_n, n_query=nq, workspace=ws, n_unique=n_unique,
                                         side_stream=side, events=events)

    for _ in range(3):
        fwd()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fwd()
    b.record()
    torch.cuda.synchronize()
    if eg.engram_last_error() != 0:
        raise RuntimeError("device error in the pipelined host path")
    ms = a.elapsed_time(b) / steps
    return {"chunk": chunk, "ms_per_step": round(ms, 4), "tokens_per_s": round(nq / (ms * 1e-3), 1),
            "rows_staged_per_step": int(n_unique.sum().item()), "steps": steps}


def time_host_cached(eg, c, cfg, tables, scales, W, g, h, dev, slots, steps):
    """The host-table path on a stream of distinct token batches (one per
    call), with and without the HBM cache of staged rows: ms per step, the
    cache's hit rate and the rows that crossed the host link."""
    import torch

    from synth.configs import make_tokens

    nq = cfg.tq
    n_b = steps + 3
    batches = []
    for k in range(n_b):
        tok, offs = make_tokens(cfg.with_(seed=cfg.seed * 1000 + 17 + k))
        batches.append((torch.from_numpy(tok).to(dev), torch.from_numpy(offs).to(dev)))
    cap = nq * 48
    cache = eg.engram_host_cache_new(c, slots, cap, device=dev)
    ws = torch.empty(eg.engram_forward_host_cached_workspace_bytes(c, nq, cap), dtype=torch.uint8, device=dev)
    stats = torch.zeros((n_b, 4), dtype=torch.int64, device=dev)
    side = torch.cuda.Stream(device=dev)
    ea, eb = torch.cuda.Event(), torch.cuda.Event()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(3):  # warm-up calls fill the cache
        eg.engram_forward_host_cached(c, batches[k][0], batches[k][1], tables, scales, W, g, h, cache, slots, cap,
                                      stamp=k + 1, n_query=nq, workspace=ws, stats=stats[k], side_stream=side,
                                      ev_dedup=ea, ev_staged=eb)
    torch.cuda.synchronize()
    a.record()
    for k in range(3, n_b):
        eg.engram_forward_host_cached(c, batches[k][0], batches[k][1], tables, scales, W, g, h, cache, slots, cap,
                                      stamp=k + 1, n_query=nq, workspace=ws, stats=stats[k], side_stream=side,
                                      ev_dedup=ea, ev_staged=eb)
    b.record()
    torch.cuda.synchronize()
    if eg.engram_last_error() != 0:
        raise RuntimeError("device error in the cached host path")
    ms_cached = a.elapsed_time(b) / steps
    st = stats[3:].double().cpu().numpy()
    fws = torch.empty(eg.engram_forward_host_workspace_bytes(c, nq, cap), dtype=torch.uint8, device=dev)
    nu = torch.zeros(1, dtype=torch.int64, device=dev)
    a.record()
    for k in range(3, n_b):
        eg.engram_forward_host(c, batches[k][0], batches[k][1], tables, scales, W, g, h, cap, n_query=nq,
                               workspace=fws, n_unique=nu, side_stream=side, ev_dedup=ea, ev_staged=eb)
    b.record()
    torch.cuda.synchronize()
    ms_plain = a.elapsed_time(b) / steps
    return {"slots": slots, "steps": steps, "batches": "a new token batch every call",
            "ms_per_step": round(ms_cached, 4), "tokens_per_s": round(nq / (ms_cached * 1e-3), 1),
            "uncached_ms_per_step": round(ms_plain, 4),
            "distinct_rows_per_step": round(float(st[:, 0].mean()), 1),
            "hit_rate": round(float(st[:, 1].sum() / st[:, 0].sum()), 4),
            "rows_over_link_per_step": round(float(st[:, 2].mean()), 1),
            "overflow_rows_per_step": round(float(st[:, 3].mean()), 1),
            "link_bytes_per_step": round(float(st[:, 2].mean()) * 260)}


def time_workload(eg, name, dev, steps, warmup):
    """engram_forward on another workload of the measurement plan, timed the
    same way (CUDA events around `steps` calls after `warmup`): ms per step,
    tokens/s and the fraction of the nominal-bytes roofline; decode-sized
    batches also eager against CUDA-graph replay."""
    import torch

    from synth import device as sd
    from synth.configs import CONFIGS, default_seeds, make_tokens

    cfg = CONFIGS[name]
    c = eg.make_config(cfg.V, cfg.R, cfg.d, default_seeds(), cfg.rms_eps)
    tok, offs = make_tokens(cfg)
    tokens, seq_offsets = torch.from_numpy(tok).to(dev), torch.from_numpy(offs).to(dev)
    host = cfg.host_tables
    if host:  # pinned host memory on huge pages, as the host-table line of run_ours
        tables = eg.host_tables_empty((48, cfg.R, 256), torch.uint8)
        scales = eg.host_tables_empty((48, cfg.R), torch.float32)
    else:
        tables = torch.zeros((48, cfg.R, 256), dtype=torch.uint8, device=dev)
        scales = torch.empty((48, cfg.R), dtype=torch.float32, device=dev)
    sd.fill_tables(tables, cfg.seed)
    sd.fill_scales(scales, cfg.seed)
    W = torch.empty((512, cfg.d), dtype=torch.bfloat16, device=dev)
    g = torch.empty(cfg.d, dtype=torch.bfloat16, device=dev)
    h = torch.empty((cfg.tq, cfg.d), dtype=torch.bfloat16, device=dev)
    sd.fill_w_out(W, cfg.seed)
    sd.fill_g(g, cfg.seed)
    sd.fill_h(h, cfg.seed)
    nq = cfg.tq
    if host:
        cap = nq * 48
        ws = torch.empty(eg.engram_forward_host_workspace_bytes(c, nq, cap), dtype=torch.uint8, device=dev)
        n_unique = torch.zeros(1, dtype=torch.int64, device=dev)
        side = torch.cuda.Stream(device=dev)
        ev_a, ev_b = torch.cuda.Event(), torch.cuda.Event()

        def fwd():
            eg.engram_forward_host(c, tokens, seq_offsets, tables, scales, W, g, h, cap, last_n=cfg.last_n,
                                   n_query=nq, workspace=ws, n_unique=n_unique, side_stream=side, ev_dedup=ev_a,
                                   ev_staged=ev_b)
    else:
        ws = torch.empty(eg.engram_forward_workspace_bytes(c, nq), dtype=torch.uint8, device=dev)

        def fwd():
            eg.engram_forward(c, tokens, seq_offsets, tables, scales, W, g, h, last_n=cfg.last_n, n_query=nq,
                              workspace=ws)

    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fwd()
    b.record()
    torch.cuda.synchronize()
    if eg.engram_last_error() != 0:
        raise RuntimeError(f"device error in the {name} workload")
    ms = a.elapsed_time(b) / steps
    gbs = nominal_bytes_per_token(cfg.d) * nq / (ms * 1e-3) / 1e9
    res = {"workload": name, "query_tokens": nq, "R": cfg.R, "steps": steps, "ms_per_step": round(ms, 4),
           "tokens_per_s": round(nq / (ms * 1e-3), 1)}
    if host:  # bound by the host link: the staging kernel against a pinned host-to-device copy
        res["tables_in"] = "pinned host memory (huge pages)"
        res["api"] = "engram_forward_host"
        res["host_link_roofline"] = host_link_roofline(eg, c, cfg, tokens, seq_offsets, tables, scales, nq, dev)
    else:
        res["step_roofline_frac"] = round(gbs / measured_peaks()["hbm_gbs"], 4)
    if nq <= 4096 and not host:
        res["cuda_graph"] = time_forward_graph(eg, c, cfg, nq, tokens, seq_offsets, tables, scales, W, g, h, dev,
                                               max(steps, 200))
        w_out = 512 * cfg.d * 2
        res["step_frac_with_W_out"] = round(
            (nominal_bytes_per_token(cfg.d) * nq + w_out) / (res["cuda_graph"]["graph_us_per_step"] * 1e-6) / 1e9
            / measured_peaks()["hbm_gbs"], 4)
    del tables, scales, h, ws
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import engram_gram_hash_gb300 as eg
    from synth import device as sd
    from synth.configs import CONFIGS, default_seeds, make_tokens

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    eg.lib()
    base = CONFIGS[args.workload]
    if args.rows:
        base = base.with_(R=args.rows)
    if args.tokens:
        base = base.with_(seq_lens=tuple(min(L, args.tokens) for L in base.seq_lens))
    # weak scaling: rank r draws its own token batch (tables are replicated weights)
    sharded = args.shard == "rows"
    # weak scaling: every rank its own batch; row-sharded tables: one batch on
    # every rank (each rank holds 1/world of every table's rows)
    cfg = base if sharded else rank_config(base, rank)
    seeds = default_seeds()
    record = args.layout != "separate"  # rows carry their scales (fp32, or MX block scales)
    c = eg.make_config(cfg.V, cfg.R, cfg.d, seeds, cfg.rms_eps,
                       row_layout={"separate": eg.ROWS_SEPARATE, "record": eg.ROWS_RECORD,
                                   "mx": eg.ROWS_MX}[args.layout])
    tok, offs = make_tokens(cfg)
    tokens = torch.from_numpy(tok).to(dev)
    seq_offsets = torch.from_numpy(offs).to(dev)
    rb = eg.RECORD_BYTES if record else 256
    kw = {"pin_memory": True} if cfg.host_tables else {"device": dev}
    huge = cfg.host_tables and args.host_alloc == "huge"
    if sharded and (cfg.host_tables or args.layout != "separate" or args.variant != "concat"):
        raise SystemExit("--shard rows runs the concatenated form on HBM tables with fp32 row scales")
    if sharded:  # this rank's rows r = rank + k * world of every table, generated one table at a time
        rows_per = eg.engram_shard_rows(c, world)
        tables = torch.zeros((48, rows_per, 256), dtype=torch.uint8, device=dev)
        scales = torch.zeros((48, rows_per), dtype=torch.float32, device=dev)
        tmp_t = torch.empty((1, cfg.R, 256), dtype=torch.uint8, device=dev)
        tmp_s = torch.empty((1, cfg.R), dtype=torch.float32, device=dev)
        for j in range(48):
            sd.fill_tables(tmp_t, base.seed, j0=j)
            sd.fill_scales(tmp_s, base.seed, j0=j)
            mine_t, mine_s = tmp_t[0, rank::world], tmp_s[0, rank::world]
            tables[j, :mine_t.shape[0]] = mine_t
            scales[j, :mine_s.shape[0]] = mine_s
        del tmp_t, tmp_s
    elif huge:  # pinned, on transparent huge pages (engram_host_alloc), zeroed
        tables = eg.host_tables_empty((48, cfg.R, rb), torch.uint8)
    else:
        tables = torch.zeros((48, cfg.R, rb), dtype=torch.uint8, **kw)
    if not sharded:
        sd.fill_tables(tables, base.seed)
        scales = None
        if args.layout == "mx":
            sd.fill_mx_scales(tables, base.seed)
        elif record:
            sd.fill_record_scales(tables, base.seed)
        else:
            scales = (eg.host_tables_empty((48, cfg.R), torch.float32) if huge
                      else torch.empty((48, cfg.R), dtype=torch.float32, **kw))
            sd.fill_scales(scales, base.seed)
    W = torch.empty((512, cfg.d), dtype=torch.bfloat16, device=dev)
    g = torch.empty(cfg.d, dtype=torch.bfloat16, device=dev)
    h = torch.empty((cfg.tq, cfg.d), dtype=torch.bfloat16, device=dev)
    sd.fill_w_out(W, base.seed)
    sd.fill_g(g, base.seed)
    sd.fill_h(h, cfg.seed)
    nq = cfg.tq
    X = torch.empty((nq, 512), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    host = cfg.host_tables
    layers = args.variant == "layers"
    if layers:  # the per-layer form: layer 0 (module 0) then layer 1 (module 1), per-row gates
        if host:
            raise SystemExit("--variant layers runs on HBM tables")
        lw = []
        for m in (0, 1):
            wq = torch.empty((cfg.d, 256), dtype=torch.bfloat16, device=dev)
            wk = torch.empty((256, 256), dtype=torch.bfloat16, device=dev)
            wm = torch.empty((256, cfg.d), dtype=torch.bfloat16, device=dev)
            sd.fill_layer_weights(wq, wk, wm, base.seed, m)
            lw.append((wq, eg.engram_layer_keys(c, wk), wm))
        lws = torch.empty(eg.engram_layer_workspace_bytes(c, nq), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
    if host:
        cap = nq * 48
        fws = torch.empty(eg.engram_forward_host_workspace_bytes(c, nq, cap), dtype=torch.uint8, device=dev)
        n_unique = torch.zeros(1, dtype=torch.int64, device=dev)
        side = torch.cuda.Stream(device=dev)
        ev_a, ev_b = torch.cuda.Event(), torch.cuda.Event()
    elif sharded:
        from engram_gram_hash_gb300 import shard as eshard

        mem = torch.empty((nq, 512), dtype=torch.float32, device=dev)
    elif not layers:
        fws = torch.empty(eg.engram_forward_workspace_bytes(c, nq), dtype=torch.uint8, device=dev)

    def step():
        """One pass of the whole path; returns the kernels it launched."""
        if host:
            eg.engram_forward_host(c, tokens, seq_offsets, tables, scales, W, g, h, cap, last_n=cfg.last_n,
                                   n_query=nq, workspace=fws, n_unique=n_unique, side_stream=side, ev_dedup=ev_a,
                                   ev_staged=ev_b)
            return 9  # hash, 5 dedup kernels, stage, staged gather, fuse
        if layers:
            for m in (0, 1):
                eg.engram_layer_forward(c, m, tokens, seq_offsets, tables, scales, lw[m][0], lw[m][1], lw[m][2], h,
                                        last_n=cfg.last_n, n_query=nq, workspace=lws)
            return 8  # per layer: query, key-side query, gated gather, projection
        if sharded:  # partial gather of this rank's rows, all-reduce of mem, projection
            eshard.forward_row_sharded(c, rank, world, tokens, seq_offsets, tables, scales, W, g, h,
                                       last_n=cfg.last_n, n_query=nq, mem=mem)
            return 2
        # engram_forward: the gather kernel, then the projection launched as its
        # programmatic dependent (its gate pass starts while the gather drains)
        eg.engram_forward(c, tokens, seq_offsets, tables, scales, W, g, h, last_n=cfg.last_n, n_query=nq,
                          workspace=fws)
        return 2

    def split_step(ev):
        """The same pass with CUDA events between its kernels (for the
        per-kernel times; the events keep the kernels apart)."""
        if layers:
            for m in (0, 1):
                ev[m].record(stream)
                eg.engram_layer_forward(c, m, tokens, seq_offsets, tables, scales, lw[m][0], lw[m][1], lw[m][2], h,
                                        last_n=cfg.last_n, n_query=nq, workspace=lws)
            ev[2].record(stream)
            return
        ev[0].record(stream)
        if sharded:
            eg.engram_gather_reduce_shard(c, rank, world, tokens, seq_offsets, tables, scales, last_n=cfg.last_n,
                                          n_query=nq, mem=mem)
            eshard.reduce_partials(mem)
        else:
            eg.engram_gather_x(c, tokens, seq_offsets, tables, scales, last_n=cfg.last_n, n_query=nq, X=X)
        ev[1].record(stream)
        if sharded:
            eg.engram_fuse(c, mem, W, g, h)
        else:
            eg.engram_fuse_x(c, X, W, g, h)
        ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if eg.engram_last_error() != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with ClockSampler(smi_index(local_rank)) as cs:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        cs.mark_start()
        t0.record(stream)
        for k in range(K):
            launches += step()
        t1.record(stream)
        torch.cuda.synchronize()
        cs.mark_end()
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    status = eg.engram_last_error()
    if status != 0:
        raise RuntimeError(f"device error {status} in the timed region")
    # whole-job tokens per step: every rank's batch, or the one shared batch when sharded
    value, ms_max = job_rate(ms, K, cfg.tq / world if sharded else cfg.tq, world, dev)
    clocks = cs.summary()
    if clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        clocks["time_x_median_mhz"] = round(ms / K * clocks["sm_mhz"], 2)  # ms x MHz, for comparing runs

    # per-kernel times: a separate pass with events between the kernels
    per_kernel_ms = {}
    if not host:
        KS = max(3, min(K, 20))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KS)]
        for k in range(KS):
            split_step(evs[k])
        torch.cuda.synchronize()
        if eg.engram_last_error() != 0:
            raise RuntimeError("device error in the per-kernel pass")
        names = ("layer0", "layer1") if layers else ("gather", "fuse")
        per_kernel_ms = {names[0]: sum(e[0].elapsed_time(e[1]) for e in evs) / KS,
                         names[1]: sum(e[1].elapsed_time(e[2]) for e in evs) / KS}

    # What stays in L2 between timed steps (129 MB): tables are always far larger;
    # a small batch's h and W_out are not.
    resident = nq * cfg.d * 2 + 512 * cfg.d * 2 + nq * 512 * 2
    l2_note = ("inputs larger than L2 (no flush)" if resident > 129e6 else
               f"no flush: table rows random over {48 * cfg.R * rb / 1e9:.1f} GB, but h, X and W_out "
               f"({resident / 1e6:.1f} MB) stay in L2 between steps")
    cuda_graph = None
    if not host and not layers and nq <= 4096:  # decode-sized batches: launch latency matters
        cuda_graph = time_forward_graph(eg, c, cfg, nq, tokens, seq_offsets, tables, scales, W, g, h, dev,
                                        max(K, 200))
    elif layers and nq <= 4096:  # the per-layer form's launches, replayed from a CUDA graph
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            step()
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        reps = max(K, 200)
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record()
        for _ in range(reps):
            gr.replay()
        gb.record()
        torch.cuda.synchronize()
        if eg.engram_last_error() != 0:
            raise RuntimeError("device error in the CUDA-graph timing")
        cuda_graph = {"api": "engram_layer_forward x 2 (module 0, then module 1)",
                      "graph_us_per_step": round(ga.elapsed_time(gb) / reps * 1e3, 2), "steps": reps}

    peaks = measured_peaks()
    # algorithmic bytes per token; a layer moves its 24 rows + scales and h once each way
    row_bytes = 264 if args.layout == "mx" else 260
    kb = ({"layer0": 24 * row_bytes + 4 * cfg.d, "layer1": 24 * row_bytes + 4 * cfg.d} if layers
          else kernel_bytes_per_token(cfg.d, args.layout))
    if sharded:  # this rank's share of the rows; the fp32 mem is written, exchanged and read
        kb = {"gather": -(-48 * 260 // world), "fuse": 4 * cfg.d}
    kernels = {}
    for name, kms in per_kernel_ms.items():
        gbs = kb[name] * nq / (kms * 1e-3) / 1e9
        kernels[name] = {"ms": round(kms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 3),
                         "algorithmic_bytes_per_token": kb[name]}
    if not layers and not host and not sharded:
        hb = handoff_bytes_per_token()
        kernels["gather"]["also_moved_per_token"] = {"X_write": hb["X_write"], "token": hb["token"],
                                                     "scale_sector_bytes_beyond_used": 48 * (32 - 4)}
        kernels["fuse"]["also_moved_per_token"] = {"X_read": hb["X_read"]}
        kernels["pdl_overlap_ms"] = round(sum(per_kernel_ms.values()) - ms / K, 4)
    roofline = None
    if per_kernel_ms:
        dom = max(per_kernel_ms, key=per_kernel_ms.get)
        ach = kb[dom] * nq / (per_kernel_ms[dom] * 1e-3) / 1e9
        tr = None if (args.rows or args.tokens or layers) else ncu_traffic(dom, args.workload, nq, args.layout)
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": tr,
                    "algorithmic_bytes_per_launch": kb[dom] * nq,
                    "peak_src": f"{peaks['src']} hbm_gbs (burst copy)",
                    "frac_vs_nominal_7900": round(ach / NOMINAL_HBM_GBS, 4)}

    if host:
        roofline = host_link_roofline(eg, c, cfg, tokens, seq_offsets, tables, scales, nq, dev)

    nominal = 2 * (24 * 256 + 4 * cfg.d) if layers else nominal_bytes_per_token(cfg.d)
    step_gbs = nominal * nq / (ms_max * 1e-3 / K) / 1e9
    step_roofline = {"nominal_bytes_per_token": nominal, "achieved_GBps": round(step_gbs, 1),
                     "peak_GBps": peaks["hbm_gbs"], "frac": round(step_gbs / peaks["hbm_gbs"], 4),
                     "frac_vs_nominal_7900": round(step_gbs / NOMINAL_HBM_GBS, 4)}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_max / K, 4), "higher_is_better": True, "scaling": "strong" if sharded else "weak",
        "vs_baseline": None,
        "dtype": "e4m3->f32 gather, bf16 x bf16 -> f32 projection, bf16 residual",
        "data": ("synthetic (seeded; tables e4m3 ~ quantised N(0,1), "
                 + ("E8M0 block scales 2^-2..2^2 per 32 codes)" if args.layout == "mx"
                    else "per-row fp32 scales U[0.5,2])")),
        "config": {"workload": args.workload + (" (reduced)" if args.rows or args.tokens else ""), "V": cfg.V, "R": cfg.R, "n_seqs": cfg.n_seqs,
                   "tokens_per_step_per_gpu": cfg.t_all, "query_tokens_per_step_per_gpu": nq, "d_model": cfg.d,
                   "table_bytes": 48 * cfg.R * rb, "tables_in": "pinned host" if host else "HBM",
                   "row_layout": {"record": "272-byte records: 256 e4m3 codes + the row's fp32 scale",
                                  "mx": "272-byte MX records: 256 e4m3 codes + 8 E8M0 block scales",
                                  "separate": "256-byte rows + separate fp32 scale array"}[args.layout],
                   "token_ids": ("uniform" if cfg.zipf_s == 0 else f"Zipf({cfg.zipf_s})"),
                   "l2": l2_note,
                   "parallelism": (f"row-sharded tables over {world} rank(s), all-reduce of mem" if sharded
                                   else f"dp{world} (replicated tables)")},
        "step_roofline": step_roofline,
        "roofline": roofline, "kernels": kernels, "gpu_launches": launches, "clocks": clocks,
    }
    if layers:
        out["config"]["variant"] = ("per-layer: layer 0 (module 0) then layer 1 (module 1), 24 rows each, "
                                    "per-row gates sigmoid(<rmsnorm(h) W_q, rmsnorm(r) W_k> / 16), W_m 256 x d")
        out["dtype"] = ("e4m3->f32 gather, bf16 x bf16 -> f32 query / key / projection (q as two bf16 halves), "
                        "bf16 residual")
    if cuda_graph is not None:
        out["cuda_graph"] = cuda_graph
    if host:
        out["config"]["n_unique_rows"] = int(n_unique.item())
        out["config"]["host_memory"] = ("pinned, transparent huge pages (engram_host_alloc)" if huge
                                        else "pinned (cudaHostAlloc via torch)")
        out["pipelined"] = [time_host_pipelined(eg, c, cfg, nq, tokens, seq_offsets, tables, scales, W, g, h, dev,
                                                ch, max(3, min(K, 20)))
                            for ch in args.host_chunks if 0 < ch < nq]
        if args.host_cache_slots > 0 and args.layout != "mx":
            out["cached"] = time_host_cached(eg, c, cfg, tables, scales, W, g, h, dev, args.host_cache_slots,
                                             max(3, min(K, 20)))
        if scales is not None:  # the same call with the fp32 scale array held in HBM instead (rows only cross the link)
            scales_dev = scales.to(dev)

            def fwd_dev_scales():
                eg.engram_forward_host(c, tokens, seq_offsets, tables, scales_dev, W, g, h, cap, last_n=cfg.last_n,
                                       n_query=nq, workspace=fws, n_unique=n_unique, side_stream=side, ev_dedup=ev_a,
                                       ev_staged=ev_b)

            for _ in range(3):
                fwd_dev_scales()
            torch.cuda.synchronize()
            da, db = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(3, min(K, 20))
            da.record()
            for _ in range(reps):
                fwd_dev_scales()
            db.record()
            torch.cuda.synchronize()
            if eg.engram_last_error() != 0:
                raise RuntimeError("device error in the device-scales host-table timing")
            dms = da.elapsed_time(db) / reps
            out["scales_in_hbm"] = {"ms_per_step": round(dms, 4), "tokens_per_s": round(nq / (dms * 1e-3), 1),
                                    "steps": reps, "note": "tables in pinned host memory, the fp32 scale array "
                                    "(48 x R x 4 B) in HBM: the link carries rows only"}
            del scales_dev
    if not args.no_e2e and not layers and not sharded:
        out["e2e"] = e2e_ours(args, eg, c, cfg, tokens, seq_offsets, tables, scales, W, g, h, nq, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not layers and not sharded:
        out["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    if world == 1 and args.also and not (args.rows or args.tokens or layers or sharded or host):
        del tables, scales
        torch.cuda.empty_cache()
        out["also"] = []
        for nm in args.also.split(","):
            if not nm or nm == args.workload:
                continue
            try:
                out["also"].append(time_workload(eg, nm, dev, 20, 5))
            except Exception as e:  # an extra line never costs the main one
                out["also"].append({"workload": nm, "error": f"{type(e).__name__}: {e}"[:300]})
                torch.cuda.empty_cache()
    return out


def host_link_roofline(eg, c, cfg, tokens, seq_offsets, tables, scales, nq, dev):
    """The staging kernel of the host-table path against the measured host
    link: unique rows x (256 B row + 4 B scale) moved over the link, divided
    by the stage kernel's CUDA-event time, against a pinned host-to-device
    copy of 2 GB measured here (cudaMemcpyAsync)."""
    import torch

    idx = eg.engram_hash(c, tokens, seq_offsets, last_n=cfg.last_n, n_query=nq)
    cap = nq * 48
    unique, idx_staged, n_unique = eg.engram_dedup(c, idx, cap)
    rows = torch.empty((cap, 256), dtype=torch.uint8, device=dev)
    scs = torch.empty(cap, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    for _ in range(2):
        eg.engram_stage(c, tables, scales, unique, n_unique, cap, rows, scs)
    reps = 10
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        eg.engram_stage(c, tables, scales, unique, n_unique, cap, rows, scs)
    b.record(st)
    torch.cuda.synchronize()
    stage_ms = a.elapsed_time(b) / reps
    U = int(n_unique.item())
    link_bytes = U * (256 + 4)
    # measured host link: pinned H2D copy
    src = torch.empty(1 << 31, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 31, dtype=torch.uint8, device=dev)
    dst.copy_(src, non_blocking=True)
    a.record(st)
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    b.record(st)
    torch.cuda.synchronize()
    h2d_gbs = 3 * (1 << 31) / (a.elapsed_time(b) * 1e-3) / 1e9
    ach = link_bytes / (stage_ms * 1e-3) / 1e9
    return {"kernel": "stage", "bound": "host-link", "achieved": round(ach, 1), "peak": round(h2d_gbs, 1),
            "unit": "GB/s", "frac": round(ach / h2d_gbs, 4), "traffic": None,
            "algorithmic_bytes_per_launch": link_bytes, "unique_rows": U, "stage_ms": round(stage_ms, 4),
            "peak_src": "measured here: pinned host-to-device cudaMemcpyAsync of 2 GiB"}


def e2e_ours(args, eg, c, cfg, tokens, seq_offsets, tables, scales, W, g, h_dev, nq, dev, world):
    """Same metric through the public API with host buffers: every step copies
    the step's tokens, offsets and residual h from pinned host memory to the
    device, runs engram_forward (or engram_forward_host), and reads h back to
    pinned host memory.  Two ways of driving the steps are timed and the
    faster is the value: serial (copy in, forward, copy out on one stream) and
    pipelined the way a server would run them (copies in, the forward pass and
    copies out on three streams over two sets of device buffers, so step k's
    forward pass overlaps step k+1's copy in and step k-1's copy out; the host
    link is full duplex).  With host tables the forward pass itself streams
    rows over the host link, so there the overlapping copies compete with it.
    The timed region runs from the first copy in to the last copy out."""
    import torch
    import torch.distributed as dist

    tok_h = tokens.cpu().pin_memory()
    off_h = seq_offsets.cpu().pin_memory()
    h_in = h_dev.cpu().pin_memory()
    h_out = [torch.empty_like(h_in).pin_memory() for _ in range(2)]
    bufs = [(torch.empty_like(tokens), torch.empty_like(seq_offsets), torch.empty_like(h_dev)) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    if cfg.host_tables:
        cap = nq * 48
        ws = torch.empty(eg.engram_forward_host_workspace_bytes(c, nq, cap), dtype=torch.uint8, device=dev)
        nu = torch.zeros(1, dtype=torch.int64, device=dev)
        side = torch.cuda.Stream(device=dev)
        ea, eb = torch.cuda.Event(), torch.cuda.Event()
    else:
        ws = torch.empty(eg.engram_forward_workspace_bytes(c, nq), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def run(tok_d, off_d, h_d):
        if cfg.host_tables:
            eg.engram_forward_host(c, tok_d, off_d, tables, scales, W, g, h_d, cap, last_n=cfg.last_n, n_query=nq,
                                   workspace=ws, n_unique=nu, stream=s_comp, side_stream=side, ev_dedup=ea,
                                   ev_staged=eb)
        else:
            eg.engram_forward(c, tok_d, off_d, tables, scales, W, g, h_d, last_n=cfg.last_n, n_query=nq, workspace=ws,
                              stream=s_comp)

    def one(k, pipelined):
        b = k % 2 if pipelined else 0
        tok_d, off_d, h_d = bufs[b]
        if not pipelined:  # everything in order on one stream
            with torch.cuda.stream(s_comp):
                tok_d.copy_(tok_h, non_blocking=True)
                off_d.copy_(off_h, non_blocking=True)
                h_d.copy_(h_in, non_blocking=True)
            run(tok_d, off_d, h_d)
            with torch.cuda.stream(s_comp):
                h_out[0].copy_(h_d, non_blocking=True)
            return
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_free[b])  # step k-2's copy out has read these buffers
            tok_d.copy_(tok_h, non_blocking=True)
            off_d.copy_(off_h, non_blocking=True)
            h_d.copy_(h_in, non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        run(tok_d, off_d, h_d)
        ev_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            h_out[b].copy_(h_d, non_blocking=True)
            ev_free[b].record(s_out)

    K = args.e2e_steps
    timed = {}
    for pipelined in (False, True):
        for k in range(max(2, args.warmup)):
            one(k, pipelined)
        torch.cuda.synchronize()
        a, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        first, last = (s_in, s_out) if pipelined else (s_comp, s_comp)
        a.record(first)
        for k in range(K):
            one(k, pipelined)
        b_ev.record(last)
        torch.cuda.synchronize()
        if eg.engram_last_error() != 0:
            raise RuntimeError("device error in the end-to-end steps")
        timed[pipelined] = job_rate(a.elapsed_time(b_ev), K, nq, world, dev)
    best = max(timed, key=lambda m: timed[m][0])
    rate, ms = timed[best]
    h2d = tok_h.numel() * 4 + off_h.numel() * 8 + h_in.numel() * 2
    d2h = h_out[0].numel() * 2
    api = "engram_forward_host" if cfg.host_tables else "engram_forward"
    out = {"value": round(rate, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms / K, 4), "api": api,
           "driving": "pipelined: copy in / forward / copy out on three streams, two buffer sets" if best
           else "serial: copy in, forward, copy out on one stream",
           "serial_ms_per_step": round(timed[False][1] / K, 4),
           "pipelined_ms_per_step": round(timed[True][1] / K, 4)}
    out["link"] = link_rates(h_in, bufs[0][2], bufs[1][2], h_out[1], s_in, s_out)
    if not cfg.host_tables and K >= 10:
        # Pipelined steady state: each step's h crosses the link once each
        # way while the other direction runs, so the duplex rate bounds it
        # (a run of a few steps is mostly pipeline fill and drain).
        bound = max(h2d, d2h) / (out["link"]["duplex_GBps_per_direction"] * 1e9) * 1e3
        out["link"]["pipelined_bound_ms_per_step"] = round(bound, 3)
        out["link"]["pipelined_frac"] = round(bound / (timed[True][1] / K), 3)
    return out


def link_rates(h_in, d_a, d_b, h_back, s_in, s_out, reps=3):
    """Pinned-host <-> device copy rates of the step's h, measured beside the
    end-to-end steps with the same buffers and streams: host to device alone,
    device to host alone, and both at once (the pipelined steps' case)."""
    import torch

    nbytes = h_in.numel() * h_in.element_size()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(to_dev, to_host, n):
        torch.cuda.synchronize()
        t0.record(s_in)
        s_out.wait_event(t0)
        for _ in range(n):
            if to_dev:
                with torch.cuda.stream(s_in):
                    d_a.copy_(h_in, non_blocking=True)
            if to_host:
                with torch.cuda.stream(s_out):
                    h_back.copy_(d_b, non_blocking=True)
        joined = torch.cuda.Event()
        joined.record(s_out)
        s_in.wait_event(joined)
        t1.record(s_in)
        torch.cuda.synchronize()
        return round(n * nbytes / (t0.elapsed_time(t1) * 1e-3) / 1e9, 1)

    timed(True, True, 1)
    return {"bytes_each_way": int(nbytes), "h2d_GBps": timed(True, False, reps),
            "d2h_GBps": timed(False, True, reps), "duplex_GBps_per_direction": timed(True, True, reps)}


# --------------------------------------------------------- the CPU oracle ---


def oracle_sample_tokens_per_s(cfg, seconds, seed=0):
    """Run the CPU oracle (hash + gather + fuse) on a sample of query tokens
    of the workload, growing the sample until it takes ~`seconds` of CPU.
    Rows, scales and h for the sample are drawn on the host beforehand and
    are not timed.  Returns (tokens/s, n_tokens, seconds)."""
    import oracle
    from synth import host
    from synth.configs import default_seeds, make_tokens, query_positions

    tok, offs = make_tokens(cfg)
    qpos = query_positions(cfg, offs)
    seeds = default_seeds()
    W = host.w_out(cfg.seed, cfg.d)
    g = host.g_vec(cfg.seed, cfg.d)
    rng = np.random.default_rng(seed)
    n = 16
    done_t, done_s = 0, 0.0
    while True:
        q = np.sort(rng.choice(cfg.tq, size=min(n, cfg.tq), replace=False))
        pos = qpos[q]
        # draw the inputs the oracle needs (untimed): rows for the oracle's own idx
        idx0 = oracle.hash_positions(tok, offs, cfg.V, cfg.R, seeds, pos)
        jj = np.tile(np.arange(48), len(q))
        rows = host.table_rows(cfg.seed, jj, idx0.reshape(-1)).reshape(len(q), 48, 256)
        sc = host.scales(cfg.seed, jj, idx0.reshape(-1)).reshape(len(q), 48)
        h0 = host.h_rows(cfg.seed, cfg.d, q)
        t0 = time.perf_counter()
        idx = oracle.hash_positions(tok, offs, cfg.V, cfg.R, seeds, pos)
        mem = oracle.gather_reduce_rows(rows, sc)
        oracle.fuse(mem, W, g, h0, cfg.rms_eps)
        dt = time.perf_counter() - t0
        assert np.array_equal(idx, idx0)
        done_t += len(q)
        done_s += dt
        if done_s >= seconds or len(q) == cfg.tq:
            break
        n = min(cfg.tq, max(n * 2, int(n * seconds / max(dt, 1e-3) * 0.5)))
    return done_t / done_s, done_t, done_s


def _oracle_job(job):
    """Pool worker (spawned): the oracle's tokens/s on its own random sample."""
    cfg, seconds, seed = job
    _, n, secs = oracle_sample_tokens_per_s(cfg, seconds, seed=seed)
    return n, secs


def oracle_pool(procs):
    """A pool of `procs` spawned processes (never forked: the parent may hold
    a CUDA context)."""
    import multiprocessing as mp

    return mp.get_context("spawn").Pool(procs)


def oracle_all_cores(cfg, seconds, pool, procs, seed0):
    """The same oracle on `procs` worker processes at once (one per host
    core), each on its own random sample for ~`seconds` of CPU.  Returns
    (aggregate tokens/s = sum of the workers' rates, tokens, the slowest
    worker's oracle seconds)."""
    res = pool.map(_oracle_job, [(cfg, seconds, seed0 + i) for i in range(procs)], chunksize=1)
    return sum(n / s for n, s in res), sum(n for n, _ in res), max(s for _, s in res)


def cpu_baseline(cfg, seconds):
    """The oracle on the host: all cores at once (the value) and one core."""
    nproc = os.cpu_count() or 1
    v1, n1, s1 = oracle_sample_tokens_per_s(cfg, seconds)
    with oracle_pool(nproc) as pool:
        va, na, sa = oracle_all_cores(cfg, max(2.0, seconds / 2), pool, nproc, 1000)
    return {"value": round(va, 2), "unit": UNIT, "cores": nproc, "kind": "oracle", "box_cores": nproc,
            "sample": f"{na} query tokens of the {cfg.name} workload drawn at random, {nproc} spawned processes "
                      f"at once (~{sa:.1f} s each; hash + gather + fuse, input draws untimed)",
            "single_core": {"value": round(v1, 2), "cores": 1,
                            "sample": f"{n1} query tokens, {s1:.1f} s single-threaded"}}


def run_reference(args, rank, world):
    from synth.configs import CONFIGS

    cfg = CONFIGS[args.workload]
    nproc = os.cpu_count() or 1
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    total_t, total_s = 0, 0.0
    with oracle_pool(nproc) as pool:
        oracle_all_cores(cfg, 0.2, pool, nproc, 0)  # warm-up: workers start, oracle loads
        for k in range(args.steps):
            v, n, s = oracle_all_cores(cfg, per_step, pool, nproc, 1000 * (k + 1))
            total_t += n
            total_s += n / v  # this step's tokens at its aggregate rate
    value = total_t / total_s
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
        "data": "synthetic (seeded)", "config": {"workload": args.workload, "V": cfg.V, "R": cfg.R, "d_model": cfg.d,
                                                  "query_tokens_per_step_per_gpu": cfg.tq},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": nproc, "kind": "oracle",
                         "box_cores": nproc,
                         "sample": f"{total_t} query tokens over {args.steps} steps, {nproc} spawned processes "
                                   "at once, each step a random sample of the workload per process"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_probe(args):
    """Ceilings for the gather: random 256-byte rows over a large buffer, with
    and without one 4-byte scale per row from a second array; and the host
    link measured two ways: random 256-byte rows read by the kernel from
    pinned host memory over unified addressing (zero-copy), and a pinned
    host-to-device cudaMemcpyAsync."""
    import ctypes

    import torch

    lib = ctypes.CDLL(os.path.join(ROOT, "libbench_probes.so"))
    lib.probe_random_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
    n_rows = 1 << ((args.probe_gb << 30) // 256).bit_length() - 1  # power of two
    rows = torch.empty(n_rows * 256, dtype=torch.uint8, device="cuda")
    rows.fill_(1)
    scales = torch.ones(n_rows, dtype=torch.float32, device="cuda")
    sink = torch.zeros(1, device="cuda")
    n_warps = 262144  # 24 rows per warp: 6.3 M rows = 1.6 GB per launch
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = {"probe": "random 256-byte rows", "buffer_GB": args.probe_gb, "rows_per_launch": n_warps * 24}
    for name, sc in (("rows", None), ("rows+scales", scales)):
        scp = ctypes.c_void_p(sc.data_ptr() if sc is not None else 0)
        for k in range(3):
            lib.probe_random_rows(ctypes.c_void_p(rows.data_ptr()), scp, n_rows, n_warps, k, ctypes.c_void_p(sink.data_ptr()), st)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record()
        for k in range(reps):
            lib.probe_random_rows(ctypes.c_void_p(rows.data_ptr()), scp, n_rows, n_warps, 100 + k,
                                  ctypes.c_void_p(sink.data_ptr()), st)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        useful = n_warps * 24 * (256 + (4 if sc is not None else 0))
        out[name] = {"ms": round(ms, 4), "useful_GBps": round(useful / ms / 1e6, 1),
                     "frac_of_copy_peak": round(useful / ms / 1e6 / measured_peaks()["hbm_gbs"], 3)}
    # the scale read's cache operator (scattered 4-byte reads: the DRAM bytes each costs)
    lib.probe_random_rows_flavor.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    names = ["ld.global.nc", "ld.global.cg", "ld.global.nc.L1::no_allocate", "ld.global.L1::no_allocate"]
    out["scale_load"] = {}
    for fl, nm in enumerate(names):
        for k in range(2):
            lib.probe_random_rows_flavor(ctypes.c_void_p(rows.data_ptr()), ctypes.c_void_p(scales.data_ptr()), n_rows,
                                         n_warps, k, ctypes.c_void_p(sink.data_ptr()), fl, st)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for k in range(10):
            lib.probe_random_rows_flavor(ctypes.c_void_p(rows.data_ptr()), ctypes.c_void_p(scales.data_ptr()), n_rows,
                                         n_warps, 300 + k, ctypes.c_void_p(sink.data_ptr()), fl, st)
        b.record()
        torch.cuda.synchronize()
        out["scale_load"][nm] = {"ms": round(a.elapsed_time(b) / 10, 4)}
    del rows, scales
    if args.probe_host_gb > 0:
        out["host_link"] = probe_host_link(lib, args.probe_host_gb, sink, st)
    return out


def probe_host_link(lib, host_gb, sink, st):
    """The host-link denominator two ways: zero-copy random 256-byte rows
    from pinned host memory (the staging kernel's access pattern), and a
    pinned host-to-device copy of 2 GiB."""
    import ctypes

    import torch

    n_rows = 1 << ((host_gb << 30) // 256).bit_length() - 1
    host = torch.empty(n_rows * 256, dtype=torch.uint8, pin_memory=True)
    host[::4096].fill_(1)  # touch every page
    n_warps = 16384  # 393,216 rows = 100 MB per launch
    res = {"buffer_GB": round(n_rows * 256 / 2**30, 1), "rows_per_launch": n_warps * 24}
    lib.probe_random_host_rows.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                           ctypes.c_void_p, ctypes.c_void_p]
    for k in range(2):
        lib.probe_random_host_rows(ctypes.c_void_p(host.data_ptr()), n_rows, n_warps, k,
                                   ctypes.c_void_p(sink.data_ptr()), st)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    a.record()
    for k in range(reps):
        lib.probe_random_host_rows(ctypes.c_void_p(host.data_ptr()), n_rows, n_warps, 200 + k,
                                   ctypes.c_void_p(sink.data_ptr()), st)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    res["zero_copy_random_rows"] = {"ms": round(ms, 3), "GBps": round(n_warps * 24 * 256 / ms / 1e6, 1)}
    src = host[: 1 << 31]
    dst = torch.empty(1 << 31, dtype=torch.uint8, device="cuda")
    dst.copy_(src, non_blocking=True)
    a.record()
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    res["pinned_h2d_copy"] = {"GBps": round(3 * (1 << 31) / (a.elapsed_time(b) * 1e-3) / 1e9, 1)}
    res["denominator_GBps"] = max(res["zero_copy_random_rows"]["GBps"], res["pinned_h2d_copy"]["GBps"])
    return res


def launch_ranks(n, argv=None):
    """Start this script once per GPU under torch.distributed.run on this node
    (rendezvous on 127.0.0.1); returns the launcher's exit code.  Rank 0
    prints the JSON line."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)]
    return subprocess.call(cmd + list(sys.argv[1:] if argv is None else argv))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large", choices=["tiny", "decode", "prefill", "large", "host"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="concat", choices=["concat", "layers"],
                    help="concat: one [T,512] projection with a token gate (the headline path); layers: two "
                         "Engram layers with per-row gates")
    ap.add_argument("--shard", default="none", choices=["none", "rows"],
                    help="rows: every rank holds 1/N of every table's rows, gathers its share for one shared "
                         "batch, and the partial sums are all-reduced before the projection")
    ap.add_argument("--layout", default="separate", choices=["record", "separate", "mx"],
                    help="table rows that carry their fp32 scale (record), MXFP8-style rows with eight E8M0 "
                         "block scales (mx), or a separate scale array")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--host-alloc", default="huge", choices=["huge", "torch"],
                    help="host tables in engram_host_alloc memory (huge pages) or torch pinned memory")
    ap.add_argument("--host-chunks", type=int, nargs="*", default=[32768],
                    help="chunk sizes for the pipelined host-table path (host workload)")
    ap.add_argument("--also", default="prefill,decode,host",
                    help="other workloads timed after the main line (engram_forward, or engram_forward_host for host "
                         "tables; 20 steps), comma-separated")
    ap.add_argument("--host-cache-slots", type=int, default=1 << 24,
                    help="rows of the HBM cache of staged rows timed beside the host-table path (0: skip)")
    ap.add_argument("--probe", action="store_true", help="print the random-row bandwidth ceilings and exit")
    ap.add_argument("--probe-gb", type=int, default=32)
    ap.add_argument("--probe-host-gb", type=int, default=16, help="pinned host buffer for the host-link probe (0: skip)")
    ap.add_argument("--rows", type=int, default=0, help="override R (reduced case for profiling)")
    ap.add_argument("--tokens", type=int, default=0, help="override tokens per sequence (reduced case)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3  # at least three warm-up steps
    if "WORLD_SIZE" not in os.environ and args.gpus > 1 and not args.probe:
        sys.exit(launch_ranks(args.gpus))  # one process per GPU, then this script in each
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus and not args.probe:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one rank per GPU "
                 f"(torch.distributed.run --nproc-per-node {args.gpus})")
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.probe:
        print(json.dumps(run_probe(args)), flush=True)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
