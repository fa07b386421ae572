"""Test helpers: a workload on the device and oracle references for it.

Device tensors come from the device twin of the generators; every expected
value comes from the oracle run on host-side draws of the same counters
(never from the CUDA path).
"""

import numpy as np
import torch

import oracle
from synth import device as sd
from synth import host
from synth.configs import default_seeds, make_tokens, query_positions

H_TOL = 2e-2  # max |gpu - ref| / max(1, |ref|) on the fused residual
MEM_TOL = 1e-5  # |gpu - ref| <= MEM_TOL * sum_j |term_j| on the module sums


class Workload:
    """layout "separate": tables [48,R,256] + scales [48,R];
    layout "record": tables [48,R,272] with each row's fp32 scale at byte 256 (scales None);
    layout "mx": tables [48,R,272] with eight E8M0 block scales at bytes 256..263 (scales None)."""

    def __init__(self, cfg, device="cuda", tables=True, host_tables=False, layout="separate"):
        import engram_gram_hash_gb300 as eg

        self.cfg = cfg
        self.dev = torch.device(device)
        self.seeds = default_seeds()
        self.layout = layout
        rl = {"separate": eg.ROWS_SEPARATE, "record": eg.ROWS_RECORD, "mx": eg.ROWS_MX}[layout]
        self.c = eg.make_config(cfg.V, cfg.R, cfg.d, self.seeds, cfg.rms_eps, row_layout=rl)
        self.tok, self.offs = make_tokens(cfg)
        self.qpos = query_positions(cfg, self.offs)
        self.tokens = torch.from_numpy(self.tok).to(self.dev)
        self.seq_offsets = torch.from_numpy(self.offs).to(self.dev)
        self.tables = self.scales = None
        if tables:
            rb = 256 if layout == "separate" else 272
            if host_tables:
                self.tables = torch.zeros((48, cfg.R, rb), dtype=torch.uint8, pin_memory=True)
            else:
                self.tables = torch.zeros((48, cfg.R, rb), dtype=torch.uint8, device=self.dev)
            sd.fill_tables(self.tables, cfg.seed)
            if layout == "record":
                sd.fill_record_scales(self.tables, cfg.seed)
            elif layout == "mx":
                sd.fill_mx_scales(self.tables, cfg.seed)
            else:
                kw = {"pin_memory": True} if host_tables else {"device": self.dev}
                self.scales = torch.empty((48, cfg.R), dtype=torch.float32, **kw)
                sd.fill_scales(self.scales, cfg.seed)
        self.W = torch.empty((512, cfg.d), dtype=torch.bfloat16, device=self.dev)
        self.g = torch.empty(cfg.d, dtype=torch.bfloat16, device=self.dev)
        sd.fill_w_out(self.W, cfg.seed)
        sd.fill_g(self.g, cfg.seed)
        torch.cuda.synchronize()

    def fresh_h(self):
        h = torch.empty((self.cfg.tq, self.cfg.d), dtype=torch.bfloat16, device=self.dev)
        sd.fill_h(h, self.cfg.seed)
        return h

    # ---------------------------------------------------------- references --
    def ref_idx_all(self):
        return oracle.hash_tokens(self.tok, self.offs, self.cfg.last_n, self.cfg.V, self.cfg.R, self.seeds)

    def ref_for(self, q_sel):
        """Oracle (idx, mem, mem_abs_bound, h) for query tokens q_sel."""
        cfg = self.cfg
        q_sel = np.asarray(q_sel, dtype=np.int64)
        idx = oracle.hash_positions(self.tok, self.offs, cfg.V, cfg.R, self.seeds, self.qpos[q_sel])
        jj = np.tile(np.arange(48), len(q_sel))
        rows = host.table_rows(cfg.seed, jj, idx.reshape(-1)).reshape(len(q_sel), 48, 256)
        if self.layout == "mx":
            esc = host.mx_scales(cfg.seed, jj, idx.reshape(-1)).reshape(len(q_sel), 48, 8)
            mem = oracle.gather_reduce_mx_rows(rows, esc)
            bound = oracle.gather_reduce_mx_rows(rows & 0x7F, esc)  # sum_j |term_j|
        else:
            sc = host.scales(cfg.seed, jj, idx.reshape(-1)).reshape(len(q_sel), 48)
            mem = oracle.gather_reduce_rows(rows, sc)
            bound = oracle.gather_reduce_rows(rows & 0x7F, sc)  # sum_j |term_j|
        h0 = host.h_rows(cfg.seed, cfg.d, q_sel)
        hn, gate = oracle.fuse(mem, host.w_out(cfg.seed, cfg.d), host.g_vec(cfg.seed, cfg.d), h0, cfg.rms_eps)
        return idx, mem, bound, hn, gate


def bf16_to_f64(t):
    if isinstance(t, np.ndarray):
        return torch.from_numpy(t.view(np.int16)).view(torch.bfloat16).double().numpy()
    return t.double().cpu().numpy()


def check_mem(got, ref, bound):
    err = np.abs(np.asarray(got, np.float64) - ref)
    worst = float(np.max(err / np.maximum(bound, 1e-30)))
    assert np.all(err <= MEM_TOL * bound), f"mem error {worst:.3e} x sum|term| exceeds {MEM_TOL}"
    return worst


def check_h(got_bf16, ref_bits):
    g = bf16_to_f64(got_bf16)
    r = bf16_to_f64(ref_bits)
    rel = np.abs(g - r) / np.maximum(1.0, np.abs(r))
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= H_TOL, f"h scaled error {worst:.3e} exceeds {H_TOL}"
    # also in bf16 ulps of the reference, for the record
    ulp = np.spacing(np.abs(r).astype(np.float32)).astype(np.float64) * 65536.0
    return worst, float(np.max(np.abs(g - r) / np.maximum(ulp, 1e-45)))


def sample_queries(cfg, offs, n, seed=0):
    """A seeded sample of query tokens plus every sequence-start and the last token."""
    tq = cfg.tq
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(tq, size=min(n, tq), replace=False).tolist())
    if cfg.last_n == 0:
        pick.update(int(x) for x in offs[:-1] if x < tq)
    pick.add(tq - 1)
    return np.array(sorted(pick), dtype=np.int64)
