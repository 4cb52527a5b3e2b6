"""Benchmark of one decode step: KV append, self-attention, cross-attention of
every layer, then the fused sampler, on one batch of synthetic input.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

Default workload: 5, the batch-128 stress case (24 layers, paged bf16 KV with
block size 16, self lengths U{512..4096}, cross 256, sampler 128x9x1088 with
planted ties, top-k 250, T=0.7, per-row seeds) -- the batch >= 32 regime in
which the self-attention's HBM bandwidth is the figure of merit.  After it the
default run measures workloads 1-4 and the e4m3 cache at 4 and 5 (--sub), and
reports them in the line's "workloads" object, each with its own clock record;
--workload I --sub none measures one workload alone.

Metric: algorithmic HBM GB/s of the whole decode step (bytes the step must
move: valid K/V, q, outputs, block-table entries, appended rows, logits and
tokens) divided by the step time, summed over ranks (each rank a replica with
its own batch: weak scaling, no collective on the data path).  The line also
carries the step time, the fused layer kernel's roofline, the standalone
self-attention call timed on its own (self_attn_standalone), the sampler time,
an end-to-end figure with host buffers, and the CPU oracle timed on a bounded
sample (cpu_baseline).  --impl reference times that oracle alone.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_attention_self_gb300 import workloads as W  # noqa: E402

METRIC = "decode-step attention µs & HBM GB/s (% of GB300 peak); fused sampler µs/step"
L2_BYTES = 129 * 2 ** 20
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------
# bytes the step must move (algorithmic, not measured)
# ---------------------------------------------------------------------------
HEAD_COPIES = 8   # distinct LM-head weight / embedding-table copies: 8 x 20 MB, more than the 129 MB L2


def step_bytes(w: W.Workload, out_bytes: int = 2, kv_bytes: int = 2):
    """Bytes one decode step must move; kv_bytes is the self cache's element size (2 bf16, 1 e4m3)."""
    BHD = w.B * w.H * w.D
    L = w.seq_len.astype(np.int64)
    self_b = int(2 * kv_bytes * w.H * w.D * L.sum()) + BHD * 2 + BHD * out_bytes
    if w.layout == "paged":
        self_b += int(4 * ((L + 15) // 16).sum())
    cross_b = int(4 * w.H * w.D * w.enc_len.astype(np.int64).sum()) + BHD * 2 + BHD * out_bytes
    append_b = 2 * BHD * 2 + 2 * BHD * kv_bytes          # k_new, v_new read; two rows written
    sampler_b = w.B * w.C * w.V * 4 + w.B * w.C * 4
    per_layer = self_b + cross_b + append_b
    return dict(self=self_b, cross=cross_b, append=append_b, sampler=sampler_b,
                step=w.layers * per_layer + sampler_b)


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group(backend=backend)
        return dist
    return None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while the timed regions run.

    Entering starts the sampler and waits for its first sample, so that it is already running when the first
    timed region starts.  A reader thread stamps each sample with its arrival time.  Timed regions much shorter
    than the sampling interval (batch 1: a few milliseconds) would see no sample at all, so `hold` keeps the GPU
    busy with untimed replays of the same work until the window has lasted MIN_WINDOW_S; the summary covers
    the samples of that window (the timed regions plus those replays) and says how long it was."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 100
    MIN_WINDOW_S = 0.35

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index
        self.stamped = []          # (arrival time, line)
        self.t0 = self.t1 = None

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.stamped.append((time.perf_counter(), line))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        if self.proc is not None:
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            deadline = time.perf_counter() + 5.0
            while not self.stamped and time.perf_counter() < deadline and self.proc.poll() is None:
                time.sleep(0.005)
        self.t0 = time.perf_counter()
        return self

    def hold(self, replay):
        """Run `replay()` (untimed, the same work as the timed regions) until the window is MIN_WINDOW_S long."""
        if self.proc is None:
            return
        while time.perf_counter() - self.t0 < self.MIN_WINDOW_S:
            replay()

    def __exit__(self, *exc):
        self.t1 = time.perf_counter()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.stamped:
            if self.t0 is None or not (self.t0 <= t <= self.t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm),
                "window_s": round(self.t1 - self.t0, 3)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def sources_digest(names) -> str:
    """First 16 hex digits of the SHA-256 of the named csrc files' code, concatenated in order.  Comments are
    removed and whitespace collapsed first, so that only a change to the code itself voids a capture."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "decode_attention_self_gb300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments (no '//' inside strings here)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's sources (its code and the launch
    planning) are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec or sources_digest(rec["sources"]) != rec.get("sources_sha256_16"):
        return None
    return rec


# ---------------------------------------------------------------------------
# the step on the GPU
# ---------------------------------------------------------------------------
class DeviceStep:
    """One decode step on the GPU: per layer one fused dr_decode_layer launch (append + self + cross), or with
    fused=False the three separate calls; then dr_sample_topk_delayed once.

    copies > 1 keeps that many copies of every layer's buffers (caches, description K/V, step inputs) at
    different addresses, and step i uses copy i % copies: a step then finds none of its data in L2 from the
    previous step when one step's bytes are below the L2 size (batch 1)."""

    def __init__(self, w: W.Workload, dev, rank: int, fused: bool = True, fp8: bool = False, copies: int = 1):
        from decode_attention_self_gb300 import api

        self.api, self.w, self.dev, self.fused, self.copies = api, w, dev, fused, copies
        base = []
        for l in range(w.layers):
            c = (W.make_self_cache_fp8 if fp8 else W.make_self_cache)(w, 1000 * rank + l, device=dev)
            kx, vx = W.make_cross_kv(w, 1000 * rank + l, device=dev)
            q, qx, kn, vn = W.make_step_inputs(w, 1000 * rank + l, device=dev)
            base.append(dict(c=c, kx=kx, vx=vx, q=q, qx=qx, kn=kn, vn=vn))
        self.sets = []
        for cp in range(copies):
            layers = []
            for b in base:
                t = {k: (v if cp == 0 else v.clone()) for k, v in b.items() if k != "c"}
                c = b["c"]
                k, v = (c.k, c.v) if cp == 0 else (c.k.clone(), c.v.clone())
                table = c.block_table.to(dev) if c.block_table is not None else None
                t["kv"] = api.KVCache(k, v, table, c.k_scale, c.v_scale)
                layers.append(t)
            self.sets.append(layers)
        self.layers = self.sets[0]
        self.pos = torch.from_numpy(w.seq_len - 1).to(dev)
        self.seq = torch.from_numpy(w.seq_len).to(dev)
        self.enc = torch.from_numpy(w.enc_len).to(dev)
        self.logits = W.make_logits(w, step_key=rank).to(dev)
        self.seeds = torch.from_numpy(w.seeds.view(np.int64)).to(dev)
        self.step = torch.from_numpy(w.steps.copy()).to(dev)
        self.tokens = torch.empty((w.B, w.C), dtype=torch.int32, device=dev)
        self.out_s = torch.empty((w.layers, w.B, w.H, w.D), dtype=torch.bfloat16, device=dev)
        self.out_x = torch.empty_like(self.out_s)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.hint = int(w.seq_len.max())
        self.hidden = self.w_head = self.w_emb = None

    def make_decoder_ends(self, rank: int = 0):
        """The decoder's output and input ends (not part of the timed step): merged LM head and merged
        embedding lookup, synthetic weights [C*V, 1024] bf16.  HEAD_COPIES distinct copies of each (160 MB in
        all, more than L2) are used in turn, so every call reads its weights from HBM."""
        w, dev = self.w, self.dev
        self.hidden = W.randn_bf16((w.B, 1024), dev, w.index, 500 + rank)
        self.w_head = [(W.randn_bf16((w.C * w.V, 1024), dev, w.index, 501 + 2 * i) * 0.1).contiguous()
                       for i in range(HEAD_COPIES)]
        self.w_emb = [W.randn_bf16((w.C * w.V, 1024), dev, w.index, 502 + 2 * i) for i in range(HEAD_COPIES)]
        self.head_logits = torch.empty((w.B, w.C, w.ldv), dtype=torch.float32, device=dev)
        self.emb_out = torch.empty((w.B, 1024), dtype=torch.bfloat16, device=dev)

    def run_lm_head(self, i: int = 0):
        self.api.dr_lm_head(self.hidden, self.w_head[i % HEAD_COPIES], self.w.C, self.head_logits,
                            err_flag=self.err)

    def run_embed(self, i: int = 0):
        self.api.dr_embed_tokens(self.tokens, self.w_emb[i % HEAD_COPIES], self.w.V, self.emb_out,
                                 err_flag=self.err)

    def launches_per_step(self) -> int:
        return (1 if self.fused else 3) * self.w.layers + 1

    def run_layer(self, l, seq=None, pos=None, copy: int = 0):
        """Layer l of the step; seq/pos (device int32 [B]) default to the workload's lengths."""
        api, L = self.api, self.sets[copy % self.copies][l]
        seq = self.seq if seq is None else seq
        pos = self.pos if pos is None else pos
        if self.fused:
            api.dr_decode_layer(L["q"], L["kv"], L["kn"], L["vn"], seq, L["qx"], L["kx"], L["vx"], self.enc,
                                self.out_s[l], self.out_x[l], max_seq_len_hint=self.hint, err_flag=self.err)
        else:
            api.dr_kv_append(L["kv"], L["kn"], L["vn"], pos, err_flag=self.err)
            api.dr_decode_self_attn(L["q"], L["kv"], seq, self.out_s[l], max_seq_len_hint=self.hint,
                                    err_flag=self.err)
            api.dr_decode_cross_attn(L["qx"], L["kx"], L["vx"], self.enc, self.out_x[l], err_flag=self.err)

    def run_dominant(self, i: int = 0):
        """The dominant kernel's launches of step i: the fused layer launches, or the self-attention calls."""
        for l in range(self.w.layers):
            if self.fused:
                self.run_layer(l, copy=i)
            else:
                self.run_self_attn(l, i)

    def run_self_attn(self, l: int, i: int = 0):
        L = self.sets[i % self.copies][l]
        self.api.dr_decode_self_attn(L["q"], L["kv"], self.seq, self.out_s[l], max_seq_len_hint=self.hint,
                                     err_flag=self.err)

    def run_sampler_only(self):
        w = self.w
        self.api.dr_sample_topk_delayed(self.logits, w.temperature, w.top_k, self.seeds, self.step, w.pad_id,
                                        self.tokens, V=w.V)

    def run(self, i: int = 0):
        for l in range(self.w.layers):
            self.run_layer(l, copy=i)
        self.run_sampler_only()


def time_long_output(ds: DeviceStep, kv_bytes: int, start: int = 0, chunk: int = 128) -> dict:
    """The long-output run itself (batch 1): n_steps consecutive steps, step t appending key start + t of every
    layer, attending start + t + 1 keys and sampling with the device step counter advancing.  Captured as
    graphs of `chunk` steps (the lengths come from a device array, one element per step) and replayed back to
    back between two events.  Overwrites the caches' keys start .. start + n_steps - 1.  With ds.copies > 1,
    step t appends into and attends over copy t % copies of the layers' buffers: every step moves the same
    bytes, and none of them stay in L2 from the step before."""
    w, api, dev = ds.w, ds.api, ds.dev
    assert w.B == 1 and w.n_steps > 1 and start + w.n_steps <= w.cap
    T = w.n_steps
    lens = torch.arange(start + 1, start + T + 1, dtype=torch.int32, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)

    pos_all = lens - 1   # the separate append call reads its position from here
    hint, ds.hint = ds.hint, start + T   # the run's own length bound
    graphs = []
    for t0 in range(0, T, chunk):
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cs):
            for t in range(t0, min(T, t0 + chunk)):
                for l in range(w.layers):
                    ds.run_layer(l, seq=lens[t:t + 1], pos=pos_all[t:t + 1], copy=t)
                api.dr_sample_topk_delayed(ds.logits, w.temperature, w.top_k, ds.seeds, step, w.pad_id, ds.tokens,
                                           V=w.V, advance=True)
        torch.cuda.current_stream().wait_stream(cs)
        graphs.append(g)
    ds.hint = hint
    for g in graphs:                                          # untimed pass: first-touch costs
        g.replay()
    torch.cuda.synchronize()
    step.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    total_ms = e0.elapsed_time(e1)
    total_bytes = sum(step_bytes(dataclasses.replace(w, seq_len=np.array([start + t + 1], np.int32)),
                                 kv_bytes=kv_bytes)["step"] for t in range(T))
    return {"steps": T, "lengths": [start + 1, start + T], "mean_us_per_step": total_ms * 1e3 / T,
            "GBps": total_bytes / (total_ms * 1e-3) / 1e9,
            "launches": T * ds.launches_per_step(),
            "timing": f"{len(graphs)} graphs of {chunk} steps replayed back to back, events around them"}


class HostStep:
    """End to end: every step's inputs come from pinned host memory and its tokens go back to the host.

    A step's inputs (every layer's q, q_cross, k_new, v_new, the logits, positions and lengths) are staged in
    one pinned host buffer and move in one copy.  Inputs and drawn tokens are double-buffered on the device,
    as a serving loop would do it: while step i runs on the compute stream, a copy stream reads back step
    i - 1's tokens and brings step i + 1's inputs into the other buffer set (the one step i - 1 used, once
    that step has finished).  Every copy and every token read-back is inside the timed region.  When the step
    rotates copies of the layers' buffers (batch 1), every copy reads the same staged inputs; only the caches
    and the description K/V rotate."""

    KEYS = ("q", "qx", "kn", "vn")

    def __init__(self, ds: DeviceStep):
        self.ds = ds
        srcs = [(("layer", l, k), L[k]) for l, L in enumerate(ds.layers) for k in self.KEYS]
        srcs += [(("logits",), ds.logits), (("pos",), ds.pos), (("seq",), ds.seq)]
        offs, total = [], 0
        for _, t in srcs:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256   # 256-byte aligned views
        self.h_flat = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.sets = []
        for _ in range(2):
            flat = torch.empty(total, dtype=torch.uint8, device=ds.dev)
            views = {}
            for (name, t), o in zip(srcs, offs):
                n = t.numel() * t.element_size()
                views[name] = flat[o:o + n].view(t.dtype).view(t.shape)
            self.sets.append({"flat": flat, "views": views, "tokens": torch.empty_like(ds.tokens)})
        for (name, t), o in zip(srcs, offs):   # the host copy of the inputs
            n = t.numel() * t.element_size()
            self.h_flat[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        self.h_tokens = torch.empty_like(ds.tokens, device="cpu").pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for _, t in srcs)
        self.d2h = self.h_tokens.numel() * 4
        self.copy_stream = torch.cuda.Stream()
        self._orig = ([{l: {k: L[k] for k in self.KEYS} for l, L in enumerate(layers)} for layers in ds.sets],
                      ds.logits, ds.pos, ds.seq, ds.tokens)

    def _use(self, st):
        ds, views = self.ds, st["views"]
        for layers in ds.sets:
            for l, L in enumerate(layers):
                for k in self.KEYS:
                    L[k] = views[("layer", l, k)]
        ds.logits, ds.pos, ds.seq, ds.tokens = views[("logits",)], views[("pos",)], views[("seq",)], st["tokens"]

    def _restore(self):
        ds = self.ds
        sets, ds.logits, ds.pos, ds.seq, ds.tokens = self._orig
        for layers, saved in zip(ds.sets, sets):
            for l, L in enumerate(layers):
                L.update(saved[l])

    def run_steps(self, K: int):
        """K steps: compute on the current stream, input copies on the copy stream, ordered by events."""
        main, side = torch.cuda.current_stream(), self.copy_stream
        side.wait_stream(main)
        copied = [torch.cuda.Event() for _ in range(K)]
        done = [torch.cuda.Event() for _ in range(K)]
        with torch.cuda.stream(side):
            for i in range(min(2, K)):
                self.sets[i % 2]["flat"].copy_(self.h_flat, non_blocking=True)
                copied[i].record(side)
        for i in range(K):
            main.wait_event(copied[i])
            self._use(self.sets[i % 2])
            self.ds.run(i)
            done[i].record(main)
            with torch.cuda.stream(side):
                side.wait_event(done[i])              # step i has drawn its tokens and read its inputs
                self.h_tokens.copy_(self.sets[i % 2]["tokens"], non_blocking=True)
                if i + 2 < K:
                    self.sets[i % 2]["flat"].copy_(self.h_flat, non_blocking=True)
                    copied[i + 2].record(side)
        main.wait_stream(side)
        self._restore()


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleSample:
    """A bounded sample of one decode step for the CPU oracle: `rows` batch rows of layer 0
    (self-attention over their paged/contiguous cache, cross-attention) and the sampler of those rows."""

    def __init__(self, w: W.Workload, rows: int):
        import oracle

        self.oracle, self.w = oracle, w
        idx = np.arange(min(rows, w.B))
        self.sub = W.Workload(w.index, w.name, 1, len(idx), w.layout, w.seq_len[idx], w.cap, w.enc_len[idx],
                              w.Lc_max, w.temperature, w.top_k, w.logit_std, w.seeds[idx], w.steps[idx],
                              H=w.H, D=w.D, C=w.C, V=w.V, ldv=w.ldv, pad_id=w.pad_id, ties=w.ties)
        s = self.sub
        cache = W.make_self_cache(s, 0, filled_len=s.seq_len)
        self.k, self.v = W.bits(cache.k), W.bits(cache.v)
        self.table = cache.block_table.numpy() if cache.block_table is not None else None
        kx, vx = W.make_cross_kv(s, 0)
        self.kx, self.vx = W.bits(kx), W.bits(vx)
        q, qx, _, _ = W.make_step_inputs(s, 0)
        self.q, self.qx = W.bits(q), W.bits(qx)
        self.logits = W.make_logits(s).numpy()
        self.scale = 1.0 / math.sqrt(s.D)
        b = step_bytes(s)
        self.bytes = b["self"] + b["cross"] + b["sampler"]

    def run(self, threads: int):
        s, o = self.sub, self.oracle
        jobs = []
        for b in range(s.B):
            for h in range(s.H):
                if self.table is not None:
                    jobs.append(lambda b=b, h=h: o.attn_paged_row(self.q[b, h], self.k, self.v, self.table[b], h,
                                                                  int(s.seq_len[b]), self.scale))
                else:
                    jobs.append(lambda b=b, h=h: o.attn_contiguous_row(self.q[b, h], self.k[b, h], self.v[b, h],
                                                                       int(s.seq_len[b]), self.scale))
                jobs.append(lambda b=b, h=h: o.attn_contiguous_row(self.qx[b, h], self.kx[b, h], self.vx[b, h],
                                                                   int(s.enc_len[b]), self.scale))
            for c in range(s.C):
                jobs.append(lambda b=b, c=c: o.sample_row(self.logits[b, c, : s.V], s.temperature, s.top_k,
                                                          int(s.seeds[b]), b, c, int(s.steps[b]), s.pad_id))
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda f: f(), jobs))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(w: W.Workload, steps: int, warmup: int = 0, min_seconds: float = 0.0):
    """Time the oracle on one layer of every batch row (self + cross attention of all heads) plus the
    sampler of every row, `steps` times (more while under min_seconds), with one thread per host core."""
    cores = host_cores()
    sample = OracleSample(w, w.B)
    for _ in range(warmup):
        sample.run(cores)
    t0 = time.perf_counter()
    n = 0
    while n < steps or time.perf_counter() - t0 < min_seconds:
        sample.run(cores)
        n += 1
    dt = time.perf_counter() - t0
    gbs = sample.bytes * n / dt / 1e9
    desc = (f"one layer of all {sample.sub.B} batch rows (self-attention over {w.layout} KV + cross-attention, "
            f"all {w.H} heads) plus the sampler of every row and codebook, {n} repetition(s) in {dt:.1f} s, "
            f"jobs per (row, head) and per (row, codebook) on a thread pool of {cores}")
    return dict(value=gbs, unit="GB/s", cores=cores, kind="oracle", sample=desc,
                seconds=dt, reps=n, bytes_per_step=sample.bytes, hardware_threads=os.cpu_count(),
                one_thread_workload1=time_oracle_one_thread())


def time_oracle_one_thread(min_seconds: float = 0.5) -> dict:
    """The oracle on the smallest workload (one layer, batch 1, 64 + 64 keys, the sampler) on one thread."""
    w1 = W.make_workload(1)
    sample = OracleSample(w1, w1.B)
    sample.run(1)
    t0, n = time.perf_counter(), 0
    while time.perf_counter() - t0 < min_seconds:
        sample.run(1)
        n += 1
    dt = time.perf_counter() - t0
    return {"us_per_step": dt / n * 1e6, "GBps": sample.bytes * n / dt / 1e9, "reps": n}


# ---------------------------------------------------------------------------
# one workload, measured on the GPU
# ---------------------------------------------------------------------------
SUB_WORKLOADS = ("1", "2", "3", "4", "4e", "5e")   # measured after the headline workload in the default run


def rotation_copies(step_b: int) -> int:
    """Copies of the layers' buffers a step rotates through so that the bytes between two uses of the same
    buffer are at least 3x L2; 1 when one step already is, or when it would take more than 8 copies (a step
    far smaller than L2, whose figure is then a warm-L2 one)."""
    if step_b >= 3 * L2_BYTES:
        return 1
    n = math.ceil(3 * L2_BYTES / step_b)
    return n if n <= 8 else 1


def l2_note(step_b: int, copies: int) -> str:
    if copies > 1:
        return (f"{copies} copies of every layer's caches and inputs used in turn: {copies * step_b / 1e6:.0f} MB "
                f"between two uses of the same data (>= 3x the 129 MB L2)")
    if step_b > L2_BYTES:
        return "inputs larger than L2 (%.1f GB per step vs 129 MB)" % (step_b / 1e9)
    return "inputs smaller than L2 (%.2f MB per step): warm-L2 figure" % (step_b / 1e6)


def workload_config(w: W.Workload, sb: dict, fp8: bool, ws: int, copies: int) -> dict:
    return {"workload": f"{w.index}: {w.name}", "batch": w.B, "layers": w.layers,
            "heads": w.H, "head_dim": w.D, "kv_layout": w.layout, "kv_dtype": "e4m3" if fp8 else "bf16",
            "codebooks": w.C, "vocab": w.V, "top_k": w.top_k, "temperature": w.temperature,
            "self_len_mean": float(w.seq_len.mean()), "self_len_max": int(w.seq_len.max()),
            "cross_len_mean": float(w.enc_len.mean()), "parallelism": f"replicas x{ws}",
            "bytes_per_step": sb["step"], "l2": l2_note(sb["step"], copies)}


def measure(w: W.Workload, K: int, warmup: int, dev, rank: int, ws: int, dist, *, fused=True, fp8=False,
            copies=1, eager=False, decoder_ends=False, standalone_self=False, e2e=False, long_output=False,
            gpu_index=0) -> dict:
    """Time K decode steps of workload w (and the dominant kernel, the sampler and the optional extras on their
    own), with an nvidia-smi clock record over the timed regions."""
    kvb = 1 if fp8 else 2
    sb = step_bytes(w, kv_bytes=kvb)
    ds = DeviceStep(w, dev, rank, fused=fused, fp8=fp8, copies=copies)
    if decoder_ends:
        ds.make_decoder_ends(rank)
    torch.cuda.synchronize()
    for i in range(max(3, warmup)):
        ds.run(i)
    torch.cuda.synchronize()
    assert int(ds.err.item()) == 0, "device error flag set during warm-up"
    K = max(K, copies) // copies * copies   # every copy is used equally often

    # The timed region is K decode steps, captured as one CUDA graph (the page's own way of removing launch
    # overhead) with no event nodes inside it; eager launches them one by one.  The dominant kernel's average
    # launch duration is then timed the same way on its own: a graph of its K x layers launches of the timed
    # steps, back to back (same arguments), bracketed by events; likewise the sampler's K launches.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cs):
            fn()
        torch.cuda.current_stream().wait_stream(cs)
        g.replay()                                         # untimed: instantiation and first-touch costs
        torch.cuda.synchronize()
        return g

    regions = {"step": lambda: [ds.run(i) for i in range(K)],
               "dominant": lambda: [ds.run_dominant(i) for i in range(K)],
               "sampler": lambda: [ds.run_sampler_only() for _ in range(K)]}
    if decoder_ends:
        regions["lm_head"] = lambda: [ds.run_lm_head(i) for i in range(K)]
        regions["embed"] = lambda: [ds.run_embed(i) for i in range(K)]
    if standalone_self and fused:
        regions["self_attn"] = lambda: [ds.run_self_attn(l, i) for i in range(K) for l in range(w.layers)]
    graphs = None if eager else {k: capture(f) for k, f in regions.items()}

    def timed(name):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        e0.record()
        if graphs is not None:
            graphs[name].replay()
        else:
            regions[name]()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    with ClockSampler(gpu_index) as clk:
        t_ms = {name: timed(name) for name in regions}

        # Regions of a few milliseconds (batch 1) are shorter than the clock sampling interval: keep the GPU on
        # the same steps (untimed replays, idempotent: same appends, no step advance) until the sampler has seen
        # them.
        def replay_steps():
            if graphs is not None:
                graphs["step"].replay()
            else:
                regions["step"]()
            torch.cuda.synchronize()

        clk.hold(replay_steps)
    barrier(dist)
    ms = max_over_ranks(dist, t_ms["step"] / K, dev)
    dom_ms = t_ms["dominant"] / (K * w.layers)
    peaks, peak_kind = measured_peaks()
    dom_bytes = sb["self"] + sb["cross"] + sb["append"] if fused else sb["self"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    kname = "decode_attn_kernel<fused>" if fused else "decode_attn_kernel"
    traffic = committed_traffic(f"{kname} workload {w.index} {'e4m3' if fp8 else 'bf16'}")
    drawing = int(sum(int(w.steps[b]) > c for b in range(w.B) for c in range(w.C)))
    r = {"value": sb["step"] * ws / (ms * 1e-3) / 1e9, "ms_per_step": ms, "us_per_step": ms * 1e3,
         "layer_us" if fused else "self_attn_us": dom_ms * 1e3,
         "sampler_us": t_ms["sampler"] / K * 1e3, "sampler_draws": drawing,
         "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": achieved / peaks["hbm_gbs"],
                      "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                      "kernel": kname + (" (dr_decode_layer: append + self + cross)" if fused
                                         else " (dr_decode_self_attn)"),
                      "peak_kind": peak_kind, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                      "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_us": dom_ms * 1e3},
         "config": workload_config(w, sb, fp8, ws, copies), "steps": K,
         "gpu_launches": ds.launches_per_step() * K, "launch_mode": "eager" if eager else "cuda_graph"}
    if "self_attn" in t_ms:
        sa_ms = t_ms["self_attn"] / (K * w.layers)
        sa = sb["self"] / (sa_ms * 1e-3) / 1e9
        sa_traffic = committed_traffic(f"decode_attn_kernel workload {w.index} {'e4m3' if fp8 else 'bf16'}")
        r["self_attn_standalone"] = {"us": sa_ms * 1e3, "achieved": sa, "frac": sa / peaks["hbm_gbs"],
                                     "frac_of_nominal_8tbs": sa / NOMINAL_HBM_GBS,
                                     "algorithmic_bytes_per_launch": sb["self"],
                                     "traffic": sa_traffic["dram_bytes_per_launch"] if sa_traffic else None,
                                     "kernel": "decode_attn_kernel (dr_decode_self_attn)"}
    if decoder_ends:
        r["decoder_ends"] = {
            "lm_head": {"us": t_ms["lm_head"] / K * 1e3, "batch": w.B, "K": 1024, "N": w.C * w.V,
                        "weight_GBps": w.C * w.V * 1024 * 2 / (t_ms["lm_head"] / K * 1e-3) / 1e9,
                        "weights": f"{HEAD_COPIES} copies used in turn (more than L2)"},
            "embed": {"us": t_ms["embed"] / K * 1e3, "rows_gathered": w.B * w.C, "Dm": 1024,
                      "tables": f"{HEAD_COPIES} copies used in turn (more than L2)"}}
    r["clocks"] = clk.summary()

    if e2e:
        # End to end: every step copies its inputs in from pinned host memory and its tokens back out, the next
        # step's copies overlapping this step's kernels.  In graph mode the K steps, with their copies on a
        # second stream, are one graph replayed once.
        hs = HostStep(ds)
        hs.run_steps(2)
        torch.cuda.synchronize()
        g_e2e = capture(lambda: hs.run_steps(K)) if graphs is not None else None
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        if g_e2e is not None:
            g_e2e.replay()
        else:
            hs.run_steps(K)
        e1.record()
        torch.cuda.synchronize()
        ems = max_over_ranks(dist, e0.elapsed_time(e1) / K, dev)
        r["e2e"] = {"value": sb["step"] * ws / (ems * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ems,
                    "h2d_bytes_per_step": hs.h2d, "d2h_bytes_per_step": hs.d2h,
                    "mode": ("cuda_graph with copy nodes" if g_e2e is not None else "eager") +
                            ", one input copy per step, inputs and tokens double-buffered: copies overlap the "
                            "previous step"}

    # the long-output workload: also the whole growing run, not only its last (longest) step, and the same
    # number of steps growing from there to the cache's capacity
    if long_output and w.n_steps > 1 and not eager:
        with ClockSampler(gpu_index) as clk2:
            lo = time_long_output(ds, kv_bytes=kvb)
            if 2 * w.n_steps <= w.cap:
                lo["continued"] = time_long_output(ds, kv_bytes=kvb, start=w.n_steps)
        lo["clocks"] = clk2.summary()
        lo["l2"] = (f"{copies} copies of every layer's caches used in turn" if copies > 1 else "one copy")
        r["long_output"] = lo

    assert int(ds.err.item()) == 0, "device error flag set during the timed steps"
    del ds, graphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return r


def sub_workload(name: str):
    """'4' -> workload 4 with a bf16 cache; '4e' -> the same with an e4m3 cache."""
    return int(name.rstrip("e")), name.endswith("e")


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps one by one instead of a CUDA graph")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="self-attention cache format (fp8 = OCP E4M3 codes with per-layer scales)")
    ap.add_argument("--unfused", action="store_true",
                    help="three launches per layer (append, self, cross) instead of one dr_decode_layer launch")
    ap.add_argument("--copies", type=int, default=0,
                    help="copies of the layers' buffers rotated over the steps (0: enough for 3x L2 at batch 1)")
    ap.add_argument("--sub", default="auto",
                    help="workloads measured after the headline one, comma-separated ('4e' = workload 4 with an "
                         "e4m3 cache); 'auto': %s after the default workload 5 run, none otherwise; 'none'"
                         % ",".join(SUB_WORKLOADS))
    args = ap.parse_args()
    ws, rank, local = dist_env()
    w = W.make_workload(args.workload)
    if args.layers > 0:
        w = dataclasses.replace(w, layers=args.layers)
    fp8 = args.kv == "fp8"
    sb = step_bytes(w, kv_bytes=1 if fp8 else 2)
    copies = args.copies if args.copies > 0 else rotation_copies(sb["step"])
    config = workload_config(w, sb, fp8, ws, copies)

    if args.impl == "reference":
        if rank != 0:
            return
        r = time_oracle(w, max(1, args.steps), warmup=min(args.warmup, 1))
        steps = r["reps"]
        ms = r["seconds"] / steps * 1e3
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": ws,
                "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
                "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample", "hardware_threads",
                                                   "one_thread_workload1")},
                "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")

    head = measure(w, args.steps, args.warmup, dev, rank, ws, dist, fused=not args.unfused, fp8=fp8,
                   copies=copies, eager=args.eager, decoder_ends=True, e2e=not args.no_e2e,
                   long_output=True, standalone_self=True, gpu_index=local)

    if args.sub == "auto":
        subs = list(SUB_WORKLOADS) if args.workload == 5 and args.layers == 0 and not args.unfused else []
    else:
        subs = [x for x in args.sub.split(",") if x and x != "none"]
    sub = {}
    for name in subs:
        idx, sfp8 = sub_workload(name)
        sw = W.make_workload(idx)
        scopies = rotation_copies(step_bytes(sw, kv_bytes=1 if sfp8 else 2)["step"])
        r = measure(sw, args.steps, args.warmup, dev, rank, ws, dist, fp8=sfp8, copies=scopies, eager=args.eager,
                    standalone_self=idx == 4, long_output=idx == 3, e2e=name == "2" and not args.no_e2e,
                    decoder_ends=name == "2", gpu_index=local)
        sub[name] = {k: r[k] for k in ("config", "steps", "us_per_step", "value", "layer_us", "sampler_us",
                                       "sampler_draws", "roofline", "clocks", "e2e", "decoder_ends") if k in r}
        sub[name]["unit"] = "GB/s"
        for k in ("self_attn_standalone", "long_output"):
            if k in r:
                sub[name][k] = r[k]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r = time_oracle(w, 1, min_seconds=10.0)
        cpu = {k: r[k] for k in ("value", "unit", "cores", "kind", "sample", "hardware_threads",
                                 "one_thread_workload1")}

    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": ws, "steps": head["steps"],
                "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": head["config"], "us_per_step": head["us_per_step"]}
        for k in ("layer_us", "self_attn_us", "sampler_us", "sampler_draws", "roofline"):
            if k in head:
                line[k] = head[k]
        line["cpu_baseline"] = cpu
        line["e2e"] = head.get("e2e")
        line["decoder_ends"] = head["decoder_ends"]
        line["gpu_launches"] = head["gpu_launches"]
        line["launch_mode"] = head["launch_mode"]
        line["kernel_timing"] = ("dominant kernel and sampler: K x layers (K) launches of the timed steps, back to "
                                 "back in their own graph, events around it")
        line["clocks"] = head["clocks"]
        if "self_attn_standalone" in head:
            line["self_attn_standalone"] = head["self_attn_standalone"]
        if "long_output" in head:
            line["long_output"] = head["long_output"]
        if sub:
            line["workloads"] = sub
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
