#!/usr/bin/env python3
"""Benchmark of one speculative verification step on GB300.

A step is one pass of the whole hot path over one batch of seeded synthetic
input already resident in HBM: paged verification attention (the gamma+1
queries of every sequence over its paged K/V history), the draft/target
rejection sampler, and the block-table commit/rollback.  Default workload: the
70B-shaped grouped-query configuration, the largest that fits one GPU (batch
64, contexts uniform in [8192, 32768], gamma = 5, 64 query / 8 kv heads,
head_dim 128, bf16 pages; sampler vocabulary 128256).  The same run times the
attention alone on the other workloads (7B-shape MHA, FP8 pages, FP8 pages
with 64-element tile scales, draft tree with shared prefix): the line's
`per_config` object.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 70b|7b|fp8|fp8_t64|tree|tiny]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Prints one JSON line.  value = algorithmic K/V bytes per step / step time
(GB/s); the roofline object covers the attention kernel alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_verify_paged_attn_gb300 import svpa  # noqa: E402
from speculative_verify_paged_attn_gb300 import workloads as W  # noqa: E402

METRIC = "paged verify-attn KV GB/s (% of GB300 HBM peak); spec_accept rows/s"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
L2_BYTES = 129 * 1024 * 1024


def flush_l2(buf: torch.Tensor) -> None:
    """Evict L2 before a timed launch: write a buffer twice the size of L2,
    then read it back.  The read writes back the dirty lines the fill left,
    so the timed launch starts from an L2 that holds only clean, unrelated
    lines (as ncu's cache control does) instead of paying for up to 129 MB of
    the flush's own write-backs inside its timed region."""
    buf.fill_(1)
    buf.sum()
# the sources that decide an attention kernel's DRAM traffic: its own file,
# the shared device helpers and the launch planning
KERNEL_SOURCES = {
    "pva_kernel": ["speculative_verify_paged_attn_gb300/csrc/paged_verify_attn.cu"],
    "pva_tc_kernel": ["speculative_verify_paged_attn_gb300/csrc/paged_verify_attn_tc.cu"],
    "pva_f8_kernel": ["speculative_verify_paged_attn_gb300/csrc/paged_verify_attn_f8.cu"],
}
KERNEL_LABELS = {"pva_kernel": "pva_kernel (warp-level MMA)", "pva_tc_kernel": "pva_tc_kernel (tcgen05/TMEM)",
                 "pva_f8_kernel": "pva_f8_kernel (tcgen05/TMEM, E4M3 scores)"}


def attn_kernel_name(params, wl) -> str:
    """The attention kernel the library runs for these parameters: the warp-level
    MMA kernel, or on the tcgen05 path the FP8 kernel for FP8 pages and the
    bf16 tcgen05 kernel otherwise."""
    if svpa.attn_kernel(params) != 2:
        return "pva_kernel"
    return "pva_f8_kernel" if wl.kv_fp8 else "pva_tc_kernel"
SHARED_SOURCES = ["speculative_verify_paged_attn_gb300/csrc/svpa_device.cuh",
                  "speculative_verify_paged_attn_gb300/csrc/svpa_api.cu"]


def code_only(text: str) -> str:
    """C/C++ source without comments and blank lines (string literals in these
    files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_hash(kernel: str) -> str:
    """Hash of the code (comments excluded) that decides a kernel's traffic."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel] + SHARED_SOURCES:
        h.update(code_only(open(os.path.join(ROOT, f)).read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(config: str, kernel: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current sources of that kernel."""
    p = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(config)
    if not e or e.get("kernel_hash") != kernel_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks sampled every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


class Step:
    """Device buffers and the three library calls of one verification step."""

    def __init__(self, wl: W.Workload, seed: int, dev: torch.device, variant: int = 0):
        self.wl, self.dev = wl, dev
        inp = W.make_attention(wl, seed, device=dev, poison=False)
        smp = W.make_sampler(wl, seed, device=dev)
        self.inp, self.smp = inp, smp
        B, n_q, Hq, D = inp.q.shape
        self.B, self.n_q = B, n_q
        self.params = svpa.attn_params(B, n_q, Hq, wl.num_kv_heads, D, inp.block_table.shape[1],
                                       inp.num_blocks, kv_fp8=wl.kv_fp8, sm_scale=wl.sm_scale,
                                       variant=variant, scale_tile=wl.scale_tile)
        self.ws = torch.zeros(svpa.attn_workspace_size(self.params), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty((B, n_q, Hq, D), dtype=torch.bfloat16, device=dev)
        self.kp = inp.k_pool.view(torch.uint8) if wl.kv_fp8 else inp.k_pool
        self.vp = inp.v_pool.view(torch.uint8) if wl.kv_fp8 else inp.v_pool
        self.mask = None if inp.ancestor_mask is None else [int(x) for x in inp.ancestor_mask.cpu().tolist()]
        self.tree = wl.tree_branching is not None
        V = smp.p.shape[2]
        self.k = torch.empty(B, dtype=torch.int32, device=dev)
        if self.tree:
            self.parent = wl.parent
            width = max(self._depth(i) for i in range(len(self.parent))) + 1
            self.path = torch.empty((B, width), dtype=torch.int32, device=dev)
            self.toks = torch.empty((B, width), dtype=torch.int32, device=dev)
            self.sws = None
        else:
            self.toks = torch.empty((B, wl.gamma + 1), dtype=torch.int32, device=dev)
            self.sws = torch.zeros(svpa.spec_accept_workspace_size(B, V), dtype=torch.uint8, device=dev)
        # commit state, reset before every step so that every step does the same work
        self.bt0, self.cl0 = inp.block_table.clone(), inp.context_lens.clone()
        self.rc0, self.fs0 = inp.refcount.clone(), inp.free_stack.clone()
        self.ft0 = torch.tensor([inp.free_top], dtype=torch.int32, device=dev)
        self.bt, self.cl = inp.block_table, inp.context_lens
        self.rc, self.fs = inp.refcount, inp.free_stack
        self.ft = self.ft0.clone()
        self.kv_bytes = inp.kv_bytes()
        pages = int(((self.cl0.long() + n_q + 15) // 16).sum().item())
        self.attn_bytes = (self.kv_bytes + 2 * inp.q.numel() * 2 + B * n_q * Hq * 4 + pages * 4)
        self.flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def _depth(self, i):
        d = 0
        while i > 0:
            i = self.parent[i]
            d += 1
        return d

    def reset(self):
        self.bt.copy_(self.bt0)
        self.cl.copy_(self.cl0)
        self.rc.copy_(self.rc0)
        self.fs.copy_(self.fs0)
        self.ft.copy_(self.ft0)

    def flush_l2(self):
        flush_l2(self.flush_buf)

    def attention(self):
        inp = self.inp
        svpa.paged_verify_attn(self.params, inp.q, self.kp, self.vp, self.bt, self.cl, self.out,
                               workspace=self.ws, error_flag=self.err, k_scale=inp.k_scale,
                               v_scale=inp.v_scale, ancestor_mask=self.mask)

    def sample(self):
        s = self.smp
        if self.tree:
            svpa.spec_accept_tree(self.parent, s.p, s.q, s.tokens, s.u_accept, s.u_sample, self.k,
                                  self.path, self.toks, error_flag=self.err)
        else:
            svpa.spec_accept(s.p, s.q, s.tokens, s.u_accept, s.u_sample, self.k, self.toks,
                             workspace=self.sws, error_flag=self.err)

    def commit(self):
        wl = self.wl
        svpa.block_table_commit(self.n_q, self.bt, self.cl, self.k, self.rc, self.fs, self.ft,
                                error_flag=self.err,
                                path_nodes=self.path if self.tree else None,
                                k_pool=self.inp.k_pool if self.tree else None,
                                v_pool=self.inp.v_pool if self.tree else None,
                                num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, kv_fp8=wl.kv_fp8)


class Append:
    """The K/V append of the same workload (n_q rows per sequence) on its own
    cache state, restored before every call so that each call does the same
    work: tables, counts and free stack, and for FP8 the partly filled pages
    (and scales) whose history a call may requantise."""

    def __init__(self, wl: W.Workload, seed: int, dev: torch.device):
        inp = W.make_append(wl, seed + 17, device=dev)
        self.inp, self.fp8, self.tile = inp, wl.kv_fp8, wl.scale_tile
        self.kp = inp.k_pool.view(torch.uint8) if self.fp8 else inp.k_pool
        self.vp = inp.v_pool.view(torch.uint8) if self.fp8 else inp.v_pool
        self.bt0, self.rc0, self.fs0 = inp.block_table.clone(), inp.refcount.clone(), inp.free_stack.clone()
        self.ft0 = torch.tensor([inp.free_top], dtype=torch.int32, device=dev)
        self.ft = self.ft0.clone()
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        L = inp.context_lens.long()
        first = inp.block_table.gather(1, (L // 16)[:, None]).squeeze(1)
        self.partial = first[(L % 16 != 0) & (first >= 0)].long()
        if self.fp8:
            self.saved = [t[self.partial].clone() for t in (self.kp, self.vp, inp.k_scale, inp.v_scale)]
        self.bytes = inp.write_bytes()

    def reset(self):
        inp = self.inp
        inp.block_table.copy_(self.bt0)
        inp.refcount.copy_(self.rc0)
        inp.free_stack.copy_(self.fs0)
        self.ft.copy_(self.ft0)
        if self.fp8:
            for t, v in zip((self.kp, self.vp, inp.k_scale, inp.v_scale), self.saved):
                t[self.partial] = v

    def run(self):
        inp = self.inp
        svpa.kv_append(inp.new_k, inp.new_v, inp.block_table, inp.context_lens, inp.refcount,
                       inp.free_stack, self.ft, self.kp, self.vp, error_flag=self.err,
                       k_scale=inp.k_scale, v_scale=inp.v_scale, scale_tile=self.tile)


class WholeStep(Append):
    """A whole verification step in call order on the append's cache state:
    K/V append, attention over the appended cache, sampler (the main step's
    inputs), commit/rollback and the draft-length update.  The cache state
    (tables, lengths, counts, free stack, FP8 partial pages) is restored
    before every step."""

    def __init__(self, wl: W.Workload, seed: int, dev: torch.device, step: "Step"):
        super().__init__(wl, seed, dev)
        inp, self.wl, self.st = self.inp, wl, step
        B = inp.new_k.shape[0]
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 29)
        self.q = torch.randn((B, wl.n_q, wl.num_q_heads, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
        self.cl0 = inp.context_lens.clone()
        self.params = svpa.attn_params(B, wl.n_q, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                       inp.block_table.shape[1], self.kp.shape[0], kv_fp8=wl.kv_fp8,
                                       sm_scale=wl.sm_scale, scale_tile=wl.scale_tile)
        self.ws = torch.zeros(svpa.attn_workspace_size(self.params), dtype=torch.uint8, device=dev)
        self.out = torch.empty((B, wl.n_q, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
        self.gs = torch.zeros((B, 2), dtype=torch.float32, device=dev)
        self.gq = torch.zeros(B, dtype=torch.int32, device=dev)
        self.gb = torch.zeros(2, dtype=torch.float32, device=dev)
        self.gg = torch.zeros(1, dtype=torch.int32, device=dev)
        self.tel = torch.zeros(4, dtype=torch.float32, device=dev)
        self.gamma = step.path.shape[1] - 1 if step.tree else wl.gamma
        T = self.cl0.long() + wl.n_q
        self.kv_bytes = int(T.sum().item()) * wl.num_kv_heads * wl.head_dim * 2 * (1 if wl.kv_fp8 else 2)

    def reset(self):
        super().reset()
        self.inp.context_lens.copy_(self.cl0)

    def run_step(self):
        inp, st, wl = self.inp, self.st, self.wl
        self.run()
        svpa.paged_verify_attn(self.params, self.q, self.kp, self.vp, inp.block_table, inp.context_lens, self.out,
                               workspace=self.ws, error_flag=self.err, k_scale=inp.k_scale, v_scale=inp.v_scale,
                               ancestor_mask=st.mask)
        st.sample()
        svpa.block_table_commit(wl.n_q, inp.block_table, inp.context_lens, st.k, inp.refcount, inp.free_stack,
                                self.ft, error_flag=self.err, path_nodes=st.path if st.tree else None,
                                k_pool=self.kp if st.tree else None, v_pool=self.vp if st.tree else None,
                                num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, kv_fp8=wl.kv_fp8)
        svpa.gamma_update(self.gamma, st.k, self.gb, self.gg, self.tel, error_flag=self.err, seq_state=self.gs,
                          seq_gamma=self.gq, draft_cost_ratio=0.08)


def time_whole_step(ws: WholeStep, steps: int, warmup: int, stream) -> float:
    """Average device time (ms) of a whole step, L2 flushed before each."""
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=ws.ft.device)
    for _ in range(warmup):
        ws.reset()
        ws.run_step()
    ms = []
    for _ in range(steps):
        ws.reset()
        flush_l2(flush)
        gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ws.run_step()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert svpa.check_error(ws.err) == 0 and svpa.check_error(ws.st.err) == 0, "device error in the whole step"
    return sum(ms) / len(ms)


def time_append(ap: Append, steps: int, warmup: int, stream) -> float:
    """Average device time (ms) of one svpa_kv_append, L2 flushed before each."""
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=ap.ft.device)
    for _ in range(warmup):
        ap.reset()
        ap.run()
    ms = []
    for _ in range(steps):
        ap.reset()
        flush_l2(flush)
        gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ap.run()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert svpa.check_error(ap.err) == 0, "device error in the append"
    return sum(ms) / len(ms)


def time_logits(wl: W.Workload, seed: int, steps: int, warmup: int, stream):
    """The sampler's logits front-end (svpa_spec_accept_logits) on the
    workload's sampler shape: B sequences, gamma + 1 target and gamma draft
    logit rows of V fp32 each, read once; L2 flushed before each launch.
    Returns (average ms, per-launch ms list, algorithmic bytes per launch)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    li = W.make_logits(wl, seed + 5, device=dev)
    B, g1, V = li.lp.shape
    k = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, g1), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(svpa.spec_accept_logits_workspace_size(B, g1 - 1, V), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def run():
        svpa.spec_accept_logits(li.lp, li.lq, li.tokens, li.u_accept, li.u_sample, k, toks, workspace=ws,
                                error_flag=err, temperature=li.temperature)

    for _ in range(warmup):
        run()
    ms = []
    for _ in range(steps):
        flush_l2(flush)
        gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert svpa.check_error(err) == 0, "device error in the logits front-end"
    g = g1 - 1
    nbytes = (2 * g + 1) * B * V * 4 + B * g * 8 + B * 4 + B * (g1 + 1) * 4
    return sum(ms) / len(ms), ms, nbytes


def time_tree_logits(wl: W.Workload, seed: int, steps: int, warmup: int, stream, peak: float):
    """The draft-tree sampler fed by logits (svpa_spec_accept_tree_logits) on
    the draft-tree workload's sampler shape: B sequences, a target logit row at
    every node and a draft row at every internal node, V fp32 each; L2 flushed
    before each launch.  The walk reads only the rows of the nodes it visits
    (a target row per node on the accepted path, the draft row of each
    internal node on it), so the algorithmic bytes count those rows from the
    launch's own paths; `dense_bytes` counts every row (what a front-end that
    forms all softmax statistics first would read)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    ti = W.make_tree_logits(wl, seed + 6, device=dev)
    B, n, V = ti.lp.shape
    par = ti.parent.tolist()
    depth = [0] * n
    for i in range(1, n):
        depth[i] = depth[par[i]] + 1
    Wd = max(depth) + 1
    internal = {p for p in par[1:]}
    k = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, Wd), dtype=torch.int32, device=dev)
    toks = torch.empty((B, Wd), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def run():
        svpa.spec_accept_tree_logits(par, ti.lp, ti.lq, ti.tokens, ti.u_accept, ti.u_sample, k, path, toks,
                                     error_flag=err, temperature=ti.temperature)

    for _ in range(warmup):
        run()
    ms = []
    for _ in range(steps):
        flush_l2(flush)
        gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert svpa.check_error(err) == 0, "device error in the tree logits front-end"
    rows = 0
    for b_path, b_k in zip(path.cpu().tolist(), k.cpu().tolist()):
        nodes = b_path[:b_k + 1]
        rows += len(nodes) + sum(1 for x in nodes if x in internal)
    small = B * n * (4 + 4) + B * 4 + B * Wd * 4 * 2 + B * 4
    nbytes = rows * V * 4 + small
    dense = (n + len(internal)) * B * V * 4 + small
    avg = sum(ms) / len(ms)
    gbs = nbytes / (avg * 1e-3) / 1e9
    return {"us": round(avg * 1e3, 2), "gbs": round(gbs, 2), "frac_of_peak": round(gbs / peak, 4),
            "bytes_per_launch": nbytes, "dense_bytes": dense, "rows_read_per_seq": round(rows / B, 3),
            "p10_p50_p90_us": [round(x * 1e3, 2) for x in percentiles(ms)],
            "shape": f"B={B}, {n} nodes ({len(internal)} internal), V={V}, fp32 logits",
            "bytes": "the visited rows' logits (target row per node on the path, draft row per internal node "
                     "on it), plus tokens, uniforms and outputs"}


LEAD_CYCLES = 200_000  # about 0.1 ms of GPU spin at GB300 clocks
LAUNCH_BOUND_US = 10.0  # roofline time below which a call is flagged launch-bound


def gpu_lead():
    """A GPU-side spin enqueued just before a timed region's first event: the
    host enqueues the region's calls while it runs, so the events time the GPU
    work rather than gaps left by the host's launch path (the e2e figure
    includes that path)."""
    torch.cuda._sleep(LEAD_CYCLES)


def time_gamma(st: "Step", steps: int, warmup: int, stream) -> float:
    """Average device time (ms) of one svpa_gamma_update on the step's
    accepted lengths (per-sequence and batch moving averages)."""
    dev, B = st.k.device, st.B
    ss = torch.zeros((B, 2), dtype=torch.float32, device=dev)
    sg = torch.zeros(B, dtype=torch.int32, device=dev)
    bs = torch.zeros(2, dtype=torch.float32, device=dev)
    bg = torch.zeros(1, dtype=torch.int32, device=dev)
    tel = torch.zeros(4, dtype=torch.float32, device=dev)
    g = st.path.shape[1] - 1 if st.tree else st.wl.gamma

    def run():
        svpa.gamma_update(g, st.k, bs, bg, tel, error_flag=st.err, seq_state=ss, seq_gamma=sg,
                          draft_cost_ratio=0.08)

    for _ in range(warmup):
        run()
    ms = []
    for _ in range(steps):
        gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert svpa.check_error(st.err) == 0, "device error in the draft-length update"
    return sum(ms) / len(ms)


PER_CONFIG = ("7b", "70b", "fp8", "fp8_t64", "tree")


def time_attention_only(name: str, steps: int, warmup: int, peak: float):
    """The attention call of workload `name` alone (its own seeded inputs,
    one launch per step, L2 flushed before each): µs, KV GB/s, the roofline
    fraction of its algorithmic bytes (K/V of valid tokens, FP8 scales,
    queries, outputs, LSE, block ids) and the DRAM traffic recorded for it."""
    wl = W.WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    inp = W.make_attention(wl, W.SEEDS[name], device=dev, poison=False)
    B, n_q, Hq, D = inp.q.shape
    params = svpa.attn_params(B, n_q, Hq, wl.num_kv_heads, D, inp.block_table.shape[1], inp.num_blocks,
                              kv_fp8=wl.kv_fp8, sm_scale=wl.sm_scale, scale_tile=wl.scale_tile)
    ws = torch.zeros(svpa.attn_workspace_size(params), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((B, n_q, Hq, D), dtype=torch.bfloat16, device=dev)
    kp = inp.k_pool.view(torch.uint8) if wl.kv_fp8 else inp.k_pool
    vp = inp.v_pool.view(torch.uint8) if wl.kv_fp8 else inp.v_pool
    mask = None if inp.ancestor_mask is None else [int(x) for x in inp.ancestor_mask.cpu().tolist()]
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def run():
        svpa.paged_verify_attn(params, inp.q, kp, vp, inp.block_table, inp.context_lens, out, workspace=ws,
                               error_flag=err, k_scale=inp.k_scale, v_scale=inp.v_scale, ancestor_mask=mask)

    for _ in range(warmup):
        run()
    ms = []
    for _ in range(steps):
        flush_l2(flush)
        gpu_lead()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert svpa.check_error(err) == 0, f"device error in the {name} attention"
    avg = sum(ms) / len(ms)
    kv = inp.kv_bytes()
    pages = int(((inp.context_lens.long() + n_q + 15) // 16).sum().item())
    alg = kv + 2 * inp.q.numel() * 2 + B * n_q * Hq * 4 + pages * 4
    kname = attn_kernel_name(params, wl)
    return {"attn_us": round(avg * 1e3, 2), "kv_gbs": round(kv / (avg * 1e-3) / 1e9, 2),
            "frac": round(alg / (avg * 1e-3) / 1e9 / peak, 4), "frac_kv": round(kv / (avg * 1e-3) / 1e9 / peak, 4),
            "traffic": recorded_traffic(name, kname), "algorithmic_bytes_per_launch": alg, "kernel": kname,
            "p10_p50_p90_us": [round(x * 1e3, 2) for x in percentiles(ms)],
            "workload": config_dict(wl)["workload"]}


def sampler_metrics(st: "Step", draws: int = 64, seed: int = 9090):
    """Acceptance statistics of the workload's sampler rows (P, Q and drafts
    fixed, `draws` fresh sets of uniforms, each one svpa call): the accepted
    length histogram, the mean accepted length with its standard error, and,
    for linear drafts, the expected accepted length of the same rows from
    "LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING" (Verification
    Acceptance Probabilities and Speedup Math): E[K] = sum_i prod_{j<=i}
    alpha_j with alpha_j = min(1, P_j(x_j) / Q_j(x_j)), averaged over rows;
    and how many final draws fell within 1e-6 of a CDF boundary."""
    s, dev, B = st.smp, st.k.device, st.B
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    near = torch.zeros(B, dtype=torch.uint8, device=dev)
    ks, nears = [], 0
    for _ in range(draws):
        ua = torch.rand(s.u_accept.shape, generator=g, device=dev)
        us = torch.rand(s.u_sample.shape, generator=g, device=dev)
        if st.tree:
            svpa.spec_accept_tree(st.parent, s.p, s.q, s.tokens, ua, us, st.k, st.path, st.toks,
                                  error_flag=st.err, near_boundary=near)
        else:
            svpa.spec_accept(s.p, s.q, s.tokens, ua, us, st.k, st.toks, workspace=st.sws, error_flag=st.err,
                             near_boundary=near)
        ks.append(st.k.clone())
        nears += int(near.sum().item())
    assert svpa.check_error(st.err) == 0, "device error in the sampler draws"
    k = torch.stack(ks).double()
    width = (st.path.shape[1] - 1) if st.tree else st.wl.gamma
    hist = torch.bincount(k.long().flatten(), minlength=width + 1).tolist()
    m = {"draws": draws * B, "rows": B, "accepted_len_hist": hist,
         "mean_k": round(float(k.mean()), 5),
         "mean_k_stderr": round(float(k.std() / (k.numel() ** 0.5)), 5),
         "near_boundary": nears, "near_boundary_frac": round(nears / (draws * B), 6)}
    if not st.tree:
        x = s.tokens.long()
        px = s.p[:, :-1, :].gather(2, x[:, :, None]).squeeze(2).double()
        qx = s.q.gather(2, x[:, :, None]).squeeze(2).double()
        alpha = torch.where(qx > 0, torch.clamp(px / qx.clamp(min=1e-300), max=1.0), torch.ones_like(px))
        ek = torch.cumprod(alpha, dim=1).sum(dim=1)
        m["expected_k_formula"] = round(float(ek.mean()), 5)
        m["formula"] = "E[K] = sum_i prod_{j<=i} min(1, P_j(x_j)/Q_j(x_j)), mean over the rows"
    else:
        m["expected_k_formula"] = None
        m["formula"] = "the pages' E[K] is for a chain of drafts; not evaluated for the tree sampler"
    return m


def percentiles(xs):
    """(p10, p50, p90) of a list of timings."""
    a = sorted(xs)
    pick = lambda q: a[min(len(a) - 1, max(0, int(round(q * (len(a) - 1)))))]
    return [round(pick(0.1), 5), round(pick(0.5), 5), round(pick(0.9), 5)]


def graph_launch_us(fn, launches: int = 100) -> float:
    """Device time per call of `fn` replayed from one CUDA graph of `launches`
    calls (no L2 flush between them: the launch-bound view of small calls)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # settle per-device launch facts outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(launches):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) * 1e3 / launches


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def subset_to_cpu(inp: W.AttnInputs, smp: W.SamplerInputs, seqs):
    """The selected sequences on the host: their queries, tables and lengths,
    a compacted pool holding only their pages (block ids renumbered), and their
    sampler rows.  (The oracle then needs no copy of a multi-GB pool.)"""
    seqs = torch.as_tensor(list(seqs), dtype=torch.long, device=inp.q.device)
    bt = inp.block_table[seqs]
    used = torch.unique(bt[bt >= 0]).long()
    remap = torch.full((inp.num_blocks,), -1, dtype=torch.int32, device=bt.device)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=bt.device)
    nbt = torch.where(bt >= 0, remap[bt.clamp(min=0).long()], bt)
    n = int(used.numel())
    d = dict(inp.__dict__)
    d.update(q=inp.q[seqs].cpu(), block_table=nbt.cpu(), context_lens=inp.context_lens[seqs].cpu(),
             k_pool=inp.k_pool[used].cpu(), v_pool=inp.v_pool[used].cpu(),
             k_scale=None if inp.k_scale is None else inp.k_scale[used].cpu(),
             v_scale=None if inp.v_scale is None else inp.v_scale[used].cpu(),
             ancestor_mask=None if inp.ancestor_mask is None else inp.ancestor_mask.cpu(),
             refcount=inp.refcount[used].cpu(), free_stack=torch.full((n,), -1, dtype=torch.int32),
             free_top=0)
    s = W.SamplerInputs(p=smp.p[seqs].cpu(), q=smp.q[seqs].cpu(), tokens=smp.tokens[seqs].cpu(),
                        u_accept=smp.u_accept[seqs].cpu(), u_sample=smp.u_sample[seqs].cpu())
    return W.AttnInputs(**d), s


def cpu_baseline(wl: W.Workload, inp: W.AttnInputs, smp: W.SamplerInputs, seed: int, budget_s: float = 12.0,
                 nthreads: int = 0):
    """The oracle, as it stands, on the host cores: attention, sampler and
    commit over chunks of the workload's sequences, taken in a seeded random
    order (one sequence per thread and chunk, wrapping around the batch), until
    the time budget is used.  Only the oracle calls are timed (not the copies
    of a chunk's pages to the host).  Returns (GB/s, cores, sample, sequences
    per second); the rate is K/V bytes of the sequences done over oracle time,
    i.e. the subset extrapolated to the workload by bytes."""
    import oracle
    oracle.build()
    cores = oracle.max_threads() if nthreads == 0 else nthreads
    B = inp.q.shape[0]
    n_q = wl.n_q
    eb = 1 if wl.kv_fp8 else 2
    order = torch.randperm(B, generator=torch.Generator().manual_seed(seed + 4242)).tolist()
    chunk = max(1, min(B, cores))  # one sequence per thread and pass
    done_bytes, t_total, nseq = 0, 0.0, 0
    start, passes = 0, 0
    while t_total < budget_s:
        sel = order[start:min(B, start + chunk)]
        c, s = subset_to_cpu(inp, smp, sel)
        am = None if c.ancestor_mask is None else c.ancestor_mask.numpy().view(np.uint64)
        t0 = time.perf_counter()
        oracle.paged_verify_attn(c.q, c.k_pool, c.v_pool, c.block_table, c.context_lens,
                                 num_kv_heads=wl.num_kv_heads, sm_scale=wl.sm_scale, kv_fp8=wl.kv_fp8,
                                 k_scale=c.k_scale, scale_tile=wl.scale_tile, v_scale=c.v_scale,
                                 ancestor_mask=am, nthreads=nthreads)
        if wl.tree_branching:
            oracle.spec_accept_tree(np.array(wl.parent, np.int32), s.p, s.q, s.tokens, s.u_accept,
                                    s.u_sample, nthreads=nthreads)
            k = np.zeros(len(sel), np.int32)
        else:
            k, *_ = oracle.spec_accept(s.p, s.q, s.tokens, s.u_accept, s.u_sample, nthreads=nthreads)
        oracle.block_table_commit(c.block_table, c.context_lens, k, c.refcount, c.free_stack, c.free_top,
                                  n_q=n_q)
        t_total += time.perf_counter() - t0
        T = c.context_lens.long() + n_q
        done_bytes += int(T.sum().item()) * wl.num_kv_heads * wl.head_dim * 2 * eb
        nseq += len(sel)
        start += chunk
        if start >= B:
            start, passes = 0, passes + 1
    gbs = done_bytes / t_total / 1e9
    sample = (f"{nseq} sequence-steps of the {wl.name} workload ({B} sequences, taken in a seeded random "
              f"order, {chunk} per chunk; {passes} full passes), attention + sampler + commit, "
              f"{t_total:.1f} s of oracle time; GB/s = K/V bytes of those sequences / oracle time")
    return gbs, cores, sample, nseq / t_total


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = W.WORKLOADS[args.config]
    seed = W.SEEDS[args.config]
    # inputs drawn with the same generators as the GPU arm (on the GPU when
    # there is one: a 5 GB pool is slow to draw on the host)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_attention(wl, seed, device=dev, poison=False)
    smp = W.make_sampler(wl, seed, device=dev)
    budget = max(4.0, min(60.0, 3.0 * (args.steps + args.warmup)))
    gbs, cores, sample, seq_per_s = cpu_baseline(wl, inp, smp, seed, budget_s=budget)
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(wl),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "spec_accept_rows_per_s": round(seq_per_s, 3)}
    print(json.dumps(line), flush=True)


def config_dict(wl: W.Workload):
    d = {"workload": f"{wl.name}: batch {wl.batch}, contexts U[{wl.ctx_lo},{wl.ctx_hi}]"
                     + (f" + {wl.shared_prefix} shared" if wl.shared_prefix else "")
                     + f", n_q {wl.n_q}, {wl.num_q_heads}/{wl.num_kv_heads} heads, head_dim {wl.head_dim}, "
                     + ("fp8-e4m3" if wl.kv_fp8 else "bf16") + f" pages of 16, vocab {wl.vocab}",
         "batch": wl.batch, "n_q": wl.n_q, "num_q_heads": wl.num_q_heads,
         "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "vocab": wl.vocab,
         "kv_dtype": "fp8_e4m3" if wl.kv_fp8 else "bf16",
         "l2": "flushed before every step, outside the step events: 256 MiB written, then read back so "
               "that the step starts from a clean L2 (the inputs are also larger than L2)",
         "timing": "CUDA events on the launching stream; a 0.1 ms GPU spin precedes each step's "
                   "first event so the host's enqueue path is not counted (e2e counts it)",
         "parallelism": "replicas (one independent batch per GPU)"}
    return d


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="70b", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the attention timings of the other workloads")
    ap.add_argument("--impl", default="svpa", choices=["svpa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", type=int, default=0, choices=[0, 1, 2],
                    help="attention kernel: 0 library's choice, 1 warp-level MMA, 2 tcgen05")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        run_reference(args)
        return

    rank, world, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    svpa.load()
    wl = W.WORKLOADS[args.config]
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    seed = W.SEEDS[args.config] + 7 * rank
    st = Step(wl, seed, dev, variant=args.variant)
    stream = torch.cuda.current_stream()

    # warm-up
    for _ in range(args.warmup):
        st.reset()
        st.attention()
        st.sample()
        st.commit()
    torch.cuda.synchronize()
    assert svpa.check_error(st.err) == 0, "device error during warm-up"

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        st.reset()
        st.flush_l2()
        gpu_lead()
        e = ev[i]
        e[0].record(stream)
        st.attention()
        e[1].record(stream)
        st.sample()
        e[2].record(stream)
        st.commit()
        e[3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    assert svpa.check_error(st.err) == 0, "device error in the timed region"
    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    attn_ms = [e[0].elapsed_time(e[1]) for e in ev]
    samp_ms = [e[1].elapsed_time(e[2]) for e in ev]
    comm_ms = [e[2].elapsed_time(e[3]) for e in ev]
    ms_local = sum(step_ms) / K
    ms = max_over_ranks(ms_local, world, dev)
    total_bytes = sum_over_ranks(float(st.kv_bytes), world, dev)
    value = total_bytes / (ms * 1e-3) / 1e9
    attn_avg = sum(attn_ms) / K
    achieved = st.attn_bytes / (attn_avg * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    rows_per_s = st.B / (sum(samp_ms) / K * 1e-3)

    # end to end through the C ABI with host buffers: inputs copied from
    # pinned host memory each step, results read back
    host = {
        "q": st.inp.q.cpu().pin_memory(), "bt": st.bt0.cpu().pin_memory(),
        "cl": st.cl0.cpu().pin_memory(), "p": st.smp.p.cpu().pin_memory(),
        "qq": st.smp.q.cpu().pin_memory(), "tok": st.smp.tokens.cpu().pin_memory(),
        "ua": st.smp.u_accept.cpu().pin_memory(), "us": st.smp.u_sample.cpu().pin_memory(),
    }
    dev_in = {"q": st.inp.q, "bt": st.bt, "cl": st.cl, "p": st.smp.p, "qq": st.smp.q,
              "tok": st.smp.tokens, "ua": st.smp.u_accept, "us": st.smp.u_sample}
    out_h = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    k_h = torch.empty(st.k.shape, dtype=torch.int32).pin_memory()
    t_h = torch.empty(st.toks.shape, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in (out_h, k_h, t_h))
    Ke = max(3, min(K, 10))
    e2e_ms = []
    # the attention's inputs go first on the step's stream; the sampler's rows
    # (the bulk of the bytes) cross on two side streams while the attention
    # runs, and the sampler waits for them
    side = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    side_keys = [("p", "tok", "ua", "us"), ("qq",)]
    torch.cuda.synchronize()
    barrier(world)
    for i in range(Ke):
        st.rc.copy_(st.rc0)
        st.fs.copy_(st.fs0)
        st.ft.copy_(st.ft0)
        st.flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        done = []
        for sd, keys in zip(side, side_keys):
            sd.wait_event(a)
            with torch.cuda.stream(sd):
                for k_ in keys:
                    dev_in[k_].copy_(host[k_], non_blocking=True)
            ev_ = torch.cuda.Event()
            ev_.record(sd)
            done.append(ev_)
        for k_ in ("q", "bt", "cl"):
            dev_in[k_].copy_(host[k_], non_blocking=True)
        st.attention()
        for ev_ in done:
            stream.wait_event(ev_)
        st.sample()
        st.commit()
        out_h.copy_(st.out, non_blocking=True)
        k_h.copy_(st.k, non_blocking=True)
        t_h.copy_(st.toks, non_blocking=True)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    barrier(world)
    e2e_local = sum(e2e_ms) / Ke
    e2e = max_over_ranks(e2e_local, world, dev)
    e2e_value = total_bytes / (e2e * 1e-3) / 1e9

    # the K/V append that precedes a verification step, timed on its own, and
    # the whole step in call order on the same cache state
    ap = WholeStep(wl, seed, dev, st)
    app_ms = time_append(ap, K, args.warmup, stream)
    app_bytes = ap.bytes
    whole_ms = time_whole_step(ap, K, args.warmup, stream)
    whole_bytes = ap.kv_bytes
    del ap
    # the draft-length controller on this step's accepted lengths
    gam_ms = time_gamma(st, K, args.warmup, stream)
    # the sampler fed by logits
    logit = None
    if st.tree:
        logit = time_tree_logits(wl, seed, K, args.warmup, stream, peak)
    else:
        lg_ms, lg_list, lg_bytes = time_logits(wl, seed, K, args.warmup, stream)
        lg_gbs = lg_bytes / (lg_ms * 1e-3) / 1e9
        logit = {"us": round(lg_ms * 1e3, 2), "gbs": round(lg_gbs, 2), "frac_of_peak": round(lg_gbs / peak, 4),
                 "bytes_per_launch": lg_bytes, "p10_p50_p90_us": [round(x * 1e3, 2) for x in percentiles(lg_list)],
                 "shape": f"B={st.B}, gamma={wl.gamma}, V={wl.vocab}, fp32 logits",
                 "bytes": "every target and draft logit read once, plus tokens, uniforms and outputs"}
    # per-launch times from CUDA graphs of 100 launches (launch-bound view)
    st.reset()
    graph_attn_us = graph_launch_us(st.attention)
    graph_samp_us = graph_launch_us(st.sample)
    torch.cuda.synchronize()
    assert svpa.check_error(st.err) == 0, "device error in the graph replays"
    # sampler bytes from each row's outcome: the P row it scanned, and the Q
    # row too when a draft was rejected, plus the gathered test values
    kk = st.k.cpu()
    V = st.smp.p.shape[2]
    if st.tree:
        samp_bytes = st.B * V * 4 * 2  # a rejection scans the residual (P and Q rows); bonus: P row
    else:
        rej = (kk < wl.gamma).to(torch.int64)
        samp_bytes = int((V * 4 * (1 + rej)).sum().item()) + st.B * 2 * wl.gamma * 4
    flops = 4 * wl.head_dim * st.n_q * wl.num_q_heads * int((st.cl0.long() + st.n_q).sum().item())
    # a call whose algorithmic bytes would take under 10 us at the measured peak is
    # launch/latency-bound: its fraction of peak is reported but says little about bandwidth
    roof_us = lambda nbytes: nbytes / (peak * 1e9) * 1e6
    launch_bound = {"attn": roof_us(st.attn_bytes) < LAUNCH_BOUND_US,
                    "spec_accept": roof_us(samp_bytes) < LAUNCH_BOUND_US}
    if logit is not None:
        launch_bound["spec_accept_logits"] = roof_us(logit["bytes_per_launch"]) < LAUNCH_BOUND_US

    smetrics = sampler_metrics(st)
    per_config = None
    if not args.no_per_config and not args.batch:
        per_config = {}
        for name in PER_CONFIG:
            if name == args.config:
                continue
            per_config[name] = time_attention_only(name, K, args.warmup, peak)
            torch.cuda.empty_cache()
            if W.WORKLOADS[name].tree_branching:
                per_config[name]["spec_accept_tree_logits"] = time_tree_logits(
                    W.WORKLOADS[name], W.SEEDS[name], K, args.warmup, stream, peak)
                torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, cores, sample, _ = cpu_baseline(wl, st.inp, st.smp, seed)
        gbs1, _, sample1, _ = cpu_baseline(wl, st.inp, st.smp, seed, budget_s=4.0, nthreads=1)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": sample, "single_thread": {"value": round(gbs1, 4), "sample": sample1}}

    kname = attn_kernel_name(st.params, wl)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if not wl.kv_fp8 else "fp8_e4m3+bf16",
            "data": "synthetic (seeded N(0,1) K/V and queries, shuffled block pool; "
                    "softmax(N(0,s)) target/draft rows)",
            "config": config_dict(wl),
            "attn_us": round(attn_avg * 1e3, 2),
            "attn_kv_gbs": round(st.kv_bytes / (attn_avg * 1e-3) / 1e9, 2),
            "attn_frac_of_peak": round(st.kv_bytes / (attn_avg * 1e-3) / 1e9 / peak, 4),
            "spec_accept_us": round(sum(samp_ms) / K * 1e3, 2),
            "spec_accept_rows_per_s": round(rows_per_s, 1),
            "commit_us": round(sum(comm_ms) / K * 1e3, 2),
            "kv_append_us": round(app_ms * 1e3, 2),
            "kv_append_gbs": round(app_bytes / (app_ms * 1e-3) / 1e9, 2),
            "gamma_update_us": round(gam_ms * 1e3, 2),
            "spec_accept_logits": logit,
            "whole_step": {"us": round(whole_ms * 1e3, 2), "kv_bytes": whole_bytes,
                           "kv_gbs": round(whole_bytes / (whole_ms * 1e-3) / 1e9, 2),
                           "calls": "kv_append, paged_verify_attn, spec_accept, block_table_commit, gamma_update",
                           "state": "the append's cache (its own context lengths), restored before each step"},
            "kv_bytes_per_step": st.kv_bytes,
            "kv_bytes_logical_per_step": int((st.cl0.long() + st.n_q).sum().item()) * wl.num_kv_heads
                                         * wl.head_dim * 2 * (1 if wl.kv_fp8 else 2),
            "attn_frac_of_nominal": round(st.kv_bytes / (attn_avg * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "attn_tflops": round(flops / (attn_avg * 1e-3) / 1e12, 2),
            "spec_accept_gbs": round(samp_bytes / (sum(samp_ms) / K * 1e-3) / 1e9, 2),
            "percentiles_p10_p50_p90": {"attn_us": [round(x * 1e3, 2) for x in percentiles(attn_ms)],
                                        "spec_accept_us": [round(x * 1e3, 2) for x in percentiles(samp_ms)],
                                        "step_ms": percentiles(step_ms)},
            "launch_bound": launch_bound,
            "sampler_metrics": smetrics,
            "per_config": per_config,
            "graph_us_per_launch": {"attn": round(graph_attn_us, 2), "spec_accept": round(graph_samp_us, 2),
                                    "launches": 100, "l2": "not flushed between launches"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic(args.config, kname),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s",
                         "kernel": KERNEL_LABELS[kname],
                         "algorithmic_bytes_per_launch": st.attn_bytes},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e, 4),
                    "copies": "pinned host buffers; the attention's inputs on the step's stream, the "
                              "sampler's rows on two side streams overlapping the attention"},
            # per step: the attention (1, or 2 with the unit ranking or the FP8
            # kernel's block prefix), sampler, commit
            "gpu_launches": (svpa.attn_launches(st.params) + 2) * K,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
