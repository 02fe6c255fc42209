#!/usr/bin/env python3
"""Decode-step select+attend benchmark (token-level KV selection, one GB300).

A step is one pass of the whole hot path over one batch: Selection Cache
check, paged score + head soft vote for the sequences that miss, selection
united with sinks and window, and sparse attention, for every sequence and
layer of the workload. The headline workload is the Llama-3-8B attention
geometry at N = 131072 (batch 1, 32 query / 8 KV heads, d 128, bf16 KV,
k 2048 + 4 sinks + 512 local, theta 0.9, a 64-step AR(1) query trajectory);
timed steps cycle through that trajectory with a fresh Selection Cache at the
start of each pass. Inputs are synthetic and already resident in HBM; L2 is
flushed before every timed step, outside the step's events (a 256 MB write,
then a 256 MB read so that no dirty line of the flush is left to be written
back inside the step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

prints one JSON line. Under torchrun every rank runs its own copy of the
workload (independent problems, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode select+attend steps/s at N=128K and 1M; achieved HBM GB/s vs peak"
UNIT = "steps/s"
L2_FLUSH_BYTES = 256 << 20
TRAJ = 64


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1920)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true", help="skip the 1M, miss-only and hit-only passes")
    p.add_argument("--cpu-baseline-only", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--case", choices=sorted(CASES),
                   help="run --steps decode steps of one workload and exit (for ncu captures; no timing)")
    p.add_argument("--phases", action="store_true",
                   help="with --case: print CTA 0's phase timestamps of each step (persistent kernel)")
    return p.parse_args(argv)


# workload index, theta for the profiling cases
CASES = {"n128k": (1, 0.9), "n128k-miss": (1, 2.0), "n1m-miss": (3, 2.0), "n1m-1layer-miss": ("3x1", 2.0),
         "n256k-1layer-miss": ("3x1@256k", 2.0), "qwen-b8-miss": (2, 2.0), "topp-b4": (4, 0.9),
         "topp-b4-miss": (4, 2.0), "topp-b4-64k-miss": ("4@64k", 2.0),
         "prefill-n128k-c512": ("prefill", None)}


def case_main(args):
    """Plain decode steps of one workload (graph replays, no flush, no timing)."""
    import torch

    import workloads as W
    cfg, theta = CASES[args.case]
    if cfg == "prefill":
        # the 128K workload's 512-query prefill chunk, --steps calls of ts_prefill_chunk
        import token_level_sparse_gb300 as T
        sp = W.spec(1, steps=512)
        wl = W.generate(sp, "cuda:0")
        ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1],
                        wl.num_pages)
        q = torch.stack([wl.q[i][0] for i in range(512)], dim=1).contiguous()
        idx = torch.zeros(1, sp.k + sp.n_sink + sp.n_local, dtype=torch.int32, device="cuda:0")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        out = torch.zeros(1, 512, sp.n_q_heads, sp.head_dim, device="cuda:0")
        prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
        for _ in range(args.steps):
            ctx.prefill_chunk(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, wl.seq_lens(0), prm, idx, cnt, out)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        print(f"case {args.case}: {args.steps} chunks")
        return
    if cfg == "3x1":
        sp = W.spec(3, layers=1)
    elif cfg == "3x1@256k":
        sp = W.spec(3, layers=1, n0=(262144,))
    elif cfg == "4@64k":
        sp = W.spec(4, n0=(65536,) * 4)
    else:
        sp = W.spec(cfg)
    b = DecodeBench(sp, "cuda:0", theta=theta)
    if args.phases:
        for i in range(args.steps):
            b.run(1, 0, flush=True, start=i)
            print_phases(b, i)
    else:
        b.run(args.steps, 0, flush=False)
    torch.cuda.synchronize()
    print(f"case {args.case}: {args.steps} steps, kernels per step {b.kernels_per_step}")


# phase boundaries the persistent kernel records (CTA 0, %globaltimer) when it ends a phase
PHASES = {0: "start", 1: "setup", 5: "lengths", 6: "cache-test", 7: "partition", 2: "scanned",
          3: "stats", 4: "scan-barrier", 13: "vote-partials", 14: "vote-norm", 20: "votes",
          28: "hist0", 29: "hist1", 30: "hist2", 21: "levels", 22: "candidates", 23: "flags",
          10: "gathered", 15: "att-scores", 16: "att-weights", 9: "rounds", 11: "attended", 24: "partials", 25: "last-barrier",
          26: "merged", 27: "end", 17: "last-cta-start", 18: "last-cta-end",
          32: "v-chunk", 33: "h0-start", 34: "h0-zeroed", 35: "h0-counted", 36: "h0-barrier",
          37: "h1-start", 38: "h1-zeroed", 39: "h1-counted", 40: "h1-barrier", 41: "h2-start",
          42: "h2-zeroed", 43: "h2-counted", 44: "h2-barrier", 45: "coarse", 46: "fine", 47: "classified",
          48: "cand-barrier", 49: "cand-fetched", 50: "ranked", 51: "att-q", 52: "att-fixed", 53: "att-own",
          54: "merge-fetched", 55: "counts", 56: "scanned-last", 57: "votes-last", 58: "classified-last",
          59: "flags-last", 8: "r1-listed", 12: "r1-gathered", 19: "r1-weights", 31: "r1-done"}


def print_phases(b, step):
    """One line: microseconds since kernel start at each recorded phase boundary (last layer)."""
    ph = b.T.ts_debug_phase_ns(b.ctx.handle)
    t0 = ph[0]
    pts = sorted((v - t0, i) for i, v in enumerate(ph) if v and i in PHASES and v >= t0)
    hit = bool(b.hit[b.sp.layers - 1][0])
    last = " ".join(f"{PHASES[i - 4]}-cta {ph[i] & 255}" for i in (61, 62, 63) if ph[i])
    if ph[60]:
        last += f" most-crossing-per-warp {ph[60] >> 32} (candidates {(ph[60] >> 8) & 0xffffff}, cta {ph[60] & 255})"
    print(f"step {step} hit={hit}: " + " ".join(f"{PHASES[i]} {dt / 1000:.1f}" for dt, i in pts) + " " + last)


# ------------------------------------------------------------ distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Largest x over the ranks (x itself when running alone)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    f"--loop-ms={period_ms}", f"--id={gpu_id}"]
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), active=f[4],
                                 hw=f[5], hwth=f[6], swth=f[7], swpc=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 1.2 * min(x["power"] for x in rows)] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwth", "hw_thermal_slowdown"),
                              ("swth", "sw_thermal_slowdown"), ("swpc", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "power_w_max": max(r["power"] for r in rows)}


# ----------------------------------------------------------- the GPU arm

def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def score_traffic():
    """Per-launch DRAM bytes of the score kernel from the committed ncu summary,
    or None when absent or taken on another revision of the kernel source."""
    src = open(os.path.join(ROOT, "token_level_sparse_gb300", "csrc", "ts_score.cu"), "rb").read()
    sha = hashlib.sha256(src).hexdigest()
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    for fn in sorted(os.listdir(prof)):
        if not fn.endswith(".md"):
            continue
        text = open(os.path.join(prof, fn)).read()
        m = re.search(r"traffic_bytes_per_launch_n128k:\s*([0-9.e+]+)\s+score_source_sha256:\s*([0-9a-f]{64})", text)
        if m and m.group(2) == sha:
            return float(m.group(1))
    return None


STEP_SOURCES = ("ts_step.cu", "ts_tc.cuh", "ts_common.cuh", "ts_internal.h")


def step_source_sha256() -> str:
    """Digest of the sources the persistent step kernel is compiled from."""
    h = hashlib.sha256()
    for fn in STEP_SOURCES:
        h.update(open(os.path.join(ROOT, "token_level_sparse_gb300", "csrc", fn), "rb").read())
    return h.hexdigest()


def step_traffic(tag="n128k"):
    """Per-launch DRAM bytes of the persistent step kernel on a miss step (tag n128k: the 128K
    workload; n1m: one 1M-token layer) from the committed ncu summaries, or None when absent or
    taken on another kernel revision."""
    sha = step_source_sha256()
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    for fn in sorted(os.listdir(prof)):
        if fn.endswith(".md"):
            m = re.search(r"step_traffic_bytes_per_launch_" + tag +
                          r":\s*([0-9.e+]+)\s+step_source_sha256:\s*([0-9a-f]{64})",
                          open(os.path.join(prof, fn)).read())
            if m and m.group(2) == sha:
                return float(m.group(1))
    return None


class DecodeBench:
    """One workload on one GPU: buffers, a captured CUDA graph of one decode step
    (all layers), and the timed loop."""

    def __init__(self, sp, device, theta, seed_offset=0):
        import torch

        import token_level_sparse_gb300 as T
        import workloads as W
        from dataclasses import replace
        self.T, self.torch = T, torch
        sp = replace(sp, seed=sp.seed + seed_offset)
        self.sp = sp
        self.dev = device
        self.wl = wl = W.generate(sp, device)
        self.theta = theta
        B, L, H, d = sp.batch, sp.layers, sp.n_q_heads, sp.head_dim
        self.ctx = T.Context(H, sp.n_kv_heads, d, T.TS_KV_BF16 if sp.kv_dtype == "bf16" else T.TS_KV_F32, B,
                             wl.page_table.shape[1], wl.num_pages)
        topp = sp.mode == "topp"
        # top-p keeps a data-dependent count, up to every cached token
        cap = self.ctx.max_tokens if topp else sp.k + sp.n_sink + sp.n_local
        self.cache = self.ctx.cache(L, self.ctx.max_tokens if topp else sp.k)
        self.params = T.params(mode=T.TS_SELECT_TOPP if topp else T.TS_SELECT_TOPK, k=sp.k, top_p=sp.top_p,
                               n_sink=sp.n_sink, n_local=sp.n_local, theta=theta)
        z = dict(device=device)
        # the step's queries (every layer) and lengths in one device block, so that the end-to-end
        # loop moves them with one copy
        nq = B * H * d
        self.in_buf = torch.zeros(L * nq + B, dtype=torch.int32, **z)
        self.q_buf = [self.in_buf[l * nq:(l + 1) * nq].view(torch.float32).view(B, H, d) for l in range(L)]
        self.seq_buf = self.in_buf[L * nq:]
        self.seq_all = torch.stack([wl.seq_lens(t) for t in range(sp.steps)])
        self.idx = [torch.zeros(B, cap, dtype=torch.int32, **z) for _ in range(L)]
        self.count = [torch.zeros(B, dtype=torch.int32, **z) for _ in range(L)]
        self.out = [torch.zeros(B, H, d, **z) for _ in range(L)]
        self.lse = [torch.zeros(B, H, **z) for _ in range(L)]
        self.hit = [torch.zeros(B, dtype=torch.uint8, **z) for _ in range(L)]
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, **z)
        self.flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, **z)
        self.flush_sink = torch.zeros((), dtype=torch.float32, **z)
        self.graph = None
        self.pattern = {}      # trajectory step -> its hits and bytes, from run()

    def flush_l2(self):
        """Evicts L2 before a timed step: a write of a buffer larger than L2, then a read of
        another one, so that the dirty lines of the write are written back here, outside the
        step's events, and the step starts with an L2 of clean lines it does not use."""
        self.flush.zero_()
        self.torch.sum(self.flush_r, 0, out=self.flush_sink)

    def _launch(self, l, q=None, seq=None):
        T = self.T
        wl = self.wl
        T.ts_decode_step(self.ctx.handle, self.cache.handle, l, self.q_buf[l] if q is None else q, wl.k_pool[l],
                         wl.v_pool[l], wl.page_table, self.seq_buf if seq is None else seq, self.sp.batch,
                         self.params, None, 0, self.idx[l], self.idx[l].stride(0), self.count[l], self.out[l],
                         self.lse[l], self.hit[l])

    def _stage(self, t):
        for l in range(self.sp.layers):
            self.q_buf[l].copy_(self.wl.q[t][l])
        self.seq_buf.copy_(self.seq_all[t])

    def capture(self):
        torch, T = self.torch, self.T
        self._stage(0)
        for l in range(self.sp.layers):      # first launch on this device, outside the capture
            self._launch(l)
        torch.cuda.synchronize()
        self.cache.reset()
        T.ts_profile_enable(self.ctx.handle, True)
        T.ts_profile_read(self.ctx.handle, keep=False)
        k0 = T.ts_kernel_count(self.ctx.handle)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l in range(self.sp.layers):
                self._launch(l)
        torch.cuda.synchronize()
        self.kernels_per_step = T.ts_kernel_count(self.ctx.handle) - k0
        self.graph = g

    def step_bytes(self, t, counts, misses):
        """Algorithmic HBM bytes of step t: K scanned for every missing (seq, layer)
        plus the K and V rows gathered for every selected token."""
        sp = self.sp
        row = sp.n_kv_heads * sp.head_dim * (2 if sp.kv_dtype == "bf16" else 4)
        scan = sum(int(n) * row for (l, b), m in misses.items() if m for n in [self.wl.n0[b] + t])
        gather = sum(int(c) * row * 2 for c in counts)
        return scan, gather

    def run(self, steps, warmup, flush=True, start=0):
        """Runs warmup + steps graph replays (trajectory steps from `start`); returns per-step
        device times and kernel times."""
        torch, T = self.torch, self.T
        if self.graph is None:
            self.capture()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        rec = []
        L, B = self.sp.layers, self.sp.batch
        for i in range(warmup + steps):
            t = (start + i) % self.sp.steps
            if t == 0:
                self.cache.reset()
            self._stage(t)
            if flush:
                self.flush_l2()
            timed = i >= warmup
            if timed:
                ev[i - warmup][0].record()
            self.graph.replay()
            if timed:
                ev[i - warmup][1].record()
            torch.cuda.synchronize()
            prof = T.ts_profile_read(self.ctx.handle, keep=True)
            if timed:
                hits = {(l, b): bool(self.hit[l][b]) for l in range(L) for b in range(B)}
                counts = [int(c) for l in range(L) for c in self.count[l].tolist()]
                misses = {k: not v for k, v in hits.items()}
                scan, gather = self.step_bytes(t, counts, misses)
                rec.append(dict(t=t, ms=ev[i - warmup][0].elapsed_time(ev[i - warmup][1]), prof=prof,
                                any_miss=any(misses.values()), n_miss=sum(misses.values()), scan=scan,
                                gather=gather))
                self.pattern[t] = dict(any_miss=any(misses.values()), n_miss=sum(misses.values()), scan=scan,
                                       gather=gather)
        st = T.ts_get_status(self.ctx.handle)
        if st != 0:
            raise RuntimeError(f"device status {T.STATUS.get(st, st)}")
        return rec

    def run_async(self, steps, warmup, flush=True, start=0):
        """The same steps enqueued back to back, the host never waiting for the device: one
        captured graph per trajectory step reads that step's query and lengths in place (no
        staging copies), so the host only flushes L2, records the events and replays, and the
        events around each replay see the step's device time rather than the host's launch
        latency. The kernels are deterministic and the cache restarts with every pass, so each
        trajectory step hits and selects as in the loop of run(), which must have covered it."""
        torch = self.torch
        if self.graph is None:
            self.capture()
        if not hasattr(self, "graphs"):
            self.T.ts_profile_enable(self.ctx.handle, False)   # no per-kernel event nodes in these graphs
            self.graphs = []
            for t in range(self.sp.steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for l in range(self.sp.layers):
                        self._launch(l, self.wl.q[t][l], self.seq_all[t])
                self.graphs.append(g)
            torch.cuda.synchronize()
            self.T.ts_profile_enable(self.ctx.handle, True)
        n = warmup + steps
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            t = (start + i) % self.sp.steps
            if t == 0:
                self.cache.reset()
            if flush:
                self.flush_l2()
            ev[i][0].record()
            self.graphs[t].replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        st = self.T.ts_get_status(self.ctx.handle)
        if st != 0:
            raise RuntimeError(f"device status {self.T.STATUS.get(st, st)}")
        rec = []
        for i in range(warmup, n):
            t = (start + i) % self.sp.steps
            r = dict(self.pattern[t])
            r.update(t=t, ms=ev[i][0].elapsed_time(ev[i][1]), prof={})
            rec.append(r)
        return rec

    def e2e(self, steps):
        """The same decode steps through the public calls with host buffers: every step copies one
        packed pinned block (the queries of every layer, the lengths, and the new token's K/V rows
        of every layer and sequence) to the device, appends the K/V rows to the paged pools
        (ts_append_kv), runs ts_decode_step per layer, and reads every layer's attention output
        back in one copy."""
        torch, T = self.torch, self.T
        wl, sp = self.wl, self.sp
        L, B, H, Hkv, d = sp.layers, sp.batch, sp.n_q_heads, sp.n_kv_heads, sp.head_dim
        P = sp.page_size
        kvb = 2 if sp.kv_dtype == "bf16" else 4
        nq, nkv = L * B * H * d * 4, L * B * Hkv * d * kvb

        def up16(x):
            return (x + 15) // 16 * 16
        o_seq = nq
        o_k = up16(o_seq + B * 4)
        o_v = up16(o_k + nkv)
        size = up16(o_v + nkv)
        dev = wl.page_table.device
        blk_dev = torch.zeros(size, dtype=torch.uint8, device=dev)
        q_dev = blk_dev[:nq].view(torch.float32).view(L, B, H, d)
        seq_dev = blk_dev[o_seq:o_seq + B * 4].view(torch.int32)
        kdt = torch.bfloat16 if kvb == 2 else torch.float32
        k_dev = blk_dev[o_k:o_k + nkv].view(kdt).view(L, B, Hkv, d)
        v_dev = blk_dev[o_v:o_v + nkv].view(kdt).view(L, B, Hkv, d)
        pt_host = wl.page_table.cpu()
        blocks = []
        for t in range(sp.steps):
            h = torch.zeros(size, dtype=torch.uint8)
            h[:nq] = torch.stack([wl.q[t][l].cpu() for l in range(L)]).reshape(-1).view(torch.uint8)
            h[o_seq:o_seq + B * 4] = self.seq_all[t].cpu().view(torch.uint8)
            ks, vs = [], []
            for l in range(L):
                for b in range(B):
                    pos = wl.n0[b] + t - 1           # the current token: the last cached position
                    page, slot = int(pt_host[b, pos // P]), pos % P
                    ks.append(wl.k_pool[l][page, :, slot, :].cpu())
                    vs.append(wl.v_pool[l][page, :, slot, :].cpu())
            h[o_k:o_k + nkv] = torch.stack(ks).reshape(-1).view(torch.uint8)
            h[o_v:o_v + nkv] = torch.stack(vs).reshape(-1).view(torch.uint8)
            blocks.append(h.pin_memory())
        out_dev = torch.zeros(L, B, H, d, device=dev)
        out_host = torch.empty(L, B, H, d).pin_memory()
        ctxh, cacheh = self.ctx.handle, self.cache.handle
        self.cache.reset()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            t = i % sp.steps
            if t == 0:
                self.cache.reset()
            blk_dev.copy_(blocks[t], non_blocking=True)
            for l in range(L):
                T.ts_append_kv(ctxh, k_dev[l], v_dev[l], wl.page_table, seq_dev, B, wl.k_pool[l], wl.v_pool[l])
                T.ts_decode_step(ctxh, cacheh, l, q_dev[l], wl.k_pool[l], wl.v_pool[l], wl.page_table, seq_dev, B,
                                 self.params, None, 0, self.idx[l], self.idx[l].stride(0), self.count[l],
                                 out_dev[l], self.lse[l], self.hit[l])
            out_host.copy_(out_dev, non_blocking=True)
            torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        st = T.ts_get_status(ctxh)
        if st != 0:
            raise RuntimeError(f"device status {T.STATUS.get(st, st)}")
        res = dict(value=steps / wall, unit=UNIT, h2d_bytes_per_step=size, d2h_bytes_per_step=out_host.numel() * 4,
                   steps=steps, note="per step: one packed pinned H2D copy (queries, lengths, new K/V rows), "
                                     "ts_append_kv and ts_decode_step per layer, one D2H copy of the outputs; no graph")
        # the same steps with each trajectory step's calls (the same copies and calls, all stream-
        # ordered) captured once as a CUDA graph and replayed: the host launches one graph per step
        # and waits for it
        try:
            T.ts_profile_enable(ctxh, False)
            graphs = []
            for t in range(sp.steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    blk_dev.copy_(blocks[t], non_blocking=True)
                    for l in range(L):
                        T.ts_append_kv(ctxh, k_dev[l], v_dev[l], wl.page_table, seq_dev, B, wl.k_pool[l],
                                       wl.v_pool[l])
                        T.ts_decode_step(ctxh, cacheh, l, q_dev[l], wl.k_pool[l], wl.v_pool[l], wl.page_table,
                                         seq_dev, B, self.params, None, 0, self.idx[l], self.idx[l].stride(0),
                                         self.count[l], out_dev[l], self.lse[l], self.hit[l])
                    out_host.copy_(out_dev, non_blocking=True)
                graphs.append(g)
            self.cache.reset()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(steps):
                t = i % sp.steps
                if t == 0:
                    self.cache.reset()
                graphs[t].replay()
                torch.cuda.synchronize()
            gwall = time.perf_counter() - t0
            st = T.ts_get_status(ctxh)
            if st == 0:
                res["graph"] = {"value": steps / gwall, "unit": UNIT,
                                "note": "the same copies and calls per step, captured once per trajectory step as a "
                                        "CUDA graph and replayed; the host waits for each step"}
        except Exception as e:  # noqa: BLE001 - the eager number stands
            res["graph"] = {"value": None, "error": str(e)[:200]}
        return res


def summarise(bench, rec, peak_gbs):
    """Headline numbers of a timed loop."""
    ms = [r["ms"] for r in rec]
    total_ms = sum(ms)
    miss = [r for r in rec if r["any_miss"]]
    fused = rec and rec[0]["prof"].get("step", (0.0, 0))[1] > 0
    timed_kernels = bool(rec and rec[0]["prof"])
    if not timed_kernels:
        score_ms = score_launches = scan_bytes = 0
    elif fused:
        # one persistent kernel per (step, layer): its bytes are the scan plus the gather
        score_ms = sum(r["prof"]["step"][0] for r in miss)
        score_launches = sum(r["prof"]["step"][1] for r in miss)
        scan_bytes = sum(r["scan"] + r["gather"] for r in miss)
    else:
        score_ms = sum(r["prof"]["score"][0] for r in miss)
        score_launches = sum(r["n_miss"] for r in miss)   # launches that scanned (one per missing layer)
        scan_bytes = sum(r["scan"] for r in miss)
    out = {"fused": bool(fused)}
    out.update(steps=len(rec), ms_per_step=total_ms / len(rec), value=1000.0 * len(rec) / total_ms,
               hit_rate=1.0 - sum(r["n_miss"] for r in rec) / (len(rec) * bench.sp.layers * bench.sp.batch))
    if miss and score_ms > 0:
        out["score_gbs"] = scan_bytes / (score_ms * 1e-3) / 1e9
        out["score_us_per_launch"] = 1000.0 * score_ms / max(1, score_launches)
        out["scan_bytes_per_launch"] = scan_bytes / max(1, score_launches)
    alg = sum(r["scan"] + r["gather"] for r in rec)
    out["step_gbs"] = alg / (total_ms * 1e-3) / 1e9
    # the least any implementation moves: K once for the scores, V of the selected tokens (their K
    # rows need not be read again when the scan's logits are kept, as the range attention does)
    out["min_step_gbs"] = sum(r["scan"] + r["gather"] / 2 for r in rec) / (total_ms * 1e-3) / 1e9
    if miss:
        mt = sum(r["ms"] for r in miss)
        out["miss_step_gbs"] = sum(r["scan"] + r["gather"] for r in miss) / (mt * 1e-3) / 1e9
        out["miss_ms_per_step"] = mt / len(miss)
        out["miss_steps"] = len(miss)
    hits = [r for r in rec if not r["any_miss"]]
    if hits:
        out["hit_ms_per_step"] = sum(r["ms"] for r in hits) / len(hits)
    fam = {}
    for r in rec:
        for k, (m, n) in r["prof"].items():
            fam[k] = fam.get(k, 0.0) + m
    out["kernel_ms_per_step"] = {k: v / len(rec) for k, v in fam.items()}
    if peak_gbs:
        out["step_frac_of_peak"] = out["step_gbs"] / peak_gbs
        out["min_frac_of_peak"] = out["min_step_gbs"] / peak_gbs
    return out


KERNEL_KEYS = ("fused", "score_gbs", "score_us_per_launch", "scan_bytes_per_launch", "kernel_ms_per_step")


def timed(bench, steps, warmup, peak_gbs, flush=True):
    """Step numbers from the back-to-back loop, per-launch kernel numbers from a loop that
    synchronises after every step (the kernel's own events are re-recorded by every replay)."""
    k = summarise(bench, bench.run(max(steps, bench.sp.steps), 3, flush=flush), peak_gbs)
    s = summarise(bench, bench.run_async(steps, warmup, flush=flush), peak_gbs)
    s.update({key: k[key] for key in KERNEL_KEYS if key in k})
    return s


def cpu_baseline_subprocess():
    """Times the CPU oracle in a fresh interpreter (no CUDA context) on the host cores."""
    env = dict(os.environ)
    n = str(os.cpu_count() or 1)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env.setdefault(k, n)
    env["CUDA_VISIBLE_DEVICES"] = ""
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-only"], env=env,
                           capture_output=True, text=True, timeout=600)
        for line in r.stdout.splitlines()[::-1]:
            if line.startswith("{"):
                return json.loads(line)
        return {"value": None, "error": (r.stderr or r.stdout)[-300:]}
    except Exception as e:  # noqa: BLE001
        return {"value": None, "error": str(e)[:300]}


def oracle_steps(max_seconds=20.0, min_steps=2, head_groups=None, steps=None, warmup=0):
    """Oracle decode steps over the 128K trajectory on CPU-generated inputs of the same
    recipe. head_groups limits scoring and attention to the first KV-head groups (a
    sample; the time then scales with the number of groups). Returns (per-step seconds,
    cpu seconds, wall seconds)."""
    import numpy as np

    import oracle as O
    import workloads as W
    sp = W.spec(1)
    wl = W.generate(sp, "cpu")
    kp, vp = W.host_copy(wl.k_pool[0]), W.host_copy(wl.v_pool[0])
    pt = W.host_copy(wl.page_table)[0]
    qs = [W.host_copy(wl.q[t][0])[0] for t in range(sp.steps)]
    if head_groups is not None:
        G = sp.n_q_heads // sp.n_kv_heads
        kp, vp = kp[:, :head_groups], vp[:, :head_groups]
        qs_s = [q[:head_groups * G] for q in qs]
    else:
        qs_s = qs
    times = []
    c0, w0 = os.times(), time.perf_counter()
    i = 0
    while True:
        t = i % sp.steps
        if t == 0:
            decide = O.CacheState()      # decisions on the full query, as on the GPU
            state = O.CacheState()       # the oracle's own state on the (sampled) heads
        s0 = time.perf_counter()
        hit, _ = O.cache_decision(decide, qs[t], sp.theta)
        O.decode_step(state, qs_s[t], kp, vp, pt, wl.n0[0] + t, k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local,
                      theta=-math.inf if hit else math.inf)
        if not hit:
            decide.first, decide.cq = False, np.asarray(qs[t], dtype=np.float64).copy()
        dt = time.perf_counter() - s0
        if i >= warmup:
            times.append(dt)
        i += 1
        if steps is not None:
            if i >= warmup + steps:
                break
        elif len(times) >= min_steps and (time.perf_counter() - w0) >= max_seconds:
            break
    c1, w1 = os.times(), time.perf_counter()
    return times, (c1.user + c1.system) - (c0.user + c0.system), w1 - w0


def cpu_model():
    """The host CPU's model name (lscpu), else the platform's processor string."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:  # noqa: BLE001
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_replica(_):
    """One process of the all-cores CPU baseline: its own copy of the 128K trajectory."""
    import torch
    torch.set_num_threads(1)             # one core per replica
    times, cpu_s, wall = oracle_steps(max_seconds=12.0, min_steps=2)
    return len(times), sum(times), cpu_s, wall


def cpu_baseline_main():
    times, cpu_s, wall = oracle_steps(max_seconds=15.0, min_steps=3)
    cores1 = max(1, round(cpu_s / wall)) if wall > 0 else 1
    one = len(times) / sum(times)
    # every host core: independent replicas of the trajectory (sequences are independent), one
    # process each (spawned: no state shared with this process)
    n = os.cpu_count() or 1
    value, cores, nsteps = one, cores1, len(times)
    try:
        import multiprocessing as mp
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"          # inherited by the spawned replicas
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_oracle_replica, range(n))
        value = sum(r[0] / r[1] for r in res)
        cores = max(1, round(sum(r[2] for r in res) / max(r[3] for r in res)))
        nsteps = sum(r[0] for r in res)
    except Exception:  # noqa: BLE001 - keep the one-core number
        pass
    print(json.dumps({"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                      "threads_available": n, "cpu_model": cpu_model(), "value_1core": one, "cores_1core": cores1,
                      "sample": f"steps of the 128K trajectory (theta 0.9), full heads, fp64 numpy oracle on "
                                f"CPU-generated inputs of the same recipe: {nsteps} steps over {n} processes "
                                f"(one replica each, about 12 s), and {len(times)} steps in one process for "
                                f"value_1core; cores = process CPU time / wall time"}))


def reference_main(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    groups = 1
    times, cpu_s, wall = oracle_steps(head_groups=groups, steps=args.steps, warmup=args.warmup)
    sp_groups = 8
    per_step = sum(times) / len(times) * (sp_groups / groups)
    v = 1.0 / per_step
    cores = max(1, round(cpu_s / wall)) if wall > 0 else 1
    sample = (f"each step: the CPU oracle's decode step of the 128K trajectory (theta 0.9) restricted to "
              f"{groups} of 8 KV-head groups (4 of 32 query heads), scaled by 8 to the full step")
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * per_step,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic",
                      "config": {"workload": "llama3-8b-gqa-n128k (B1, H32/Hkv8, d128, bf16 KV, N0=131072, "
                                             "k2048+4+512, theta 0.9)", "parallelism": "host cores"},
                      "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                       "sample": sample},
                      "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def _event_ms(fn, iters, warmup):
    """Mean device time (ms) of fn() over iters calls after warmup calls, CUDA events on the
    current stream, synchronised on both sides."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def prefill_extra(dev, peaks, c=512):
    """ts_prefill_chunk on the 128K workload with a chunk of c queries: the whole call (mean query,
    persistent score + selection, tensor-core causal chunk attention) and the chunk attention's
    own launch, against the dense bf16 tensor peak. Useful FLOPs count 2 x 2 x d per visible
    (query, head, token): the scores and the weighted values, nothing for the extra query terms,
    the second pass or the weight terms."""
    import torch
    import token_level_sparse_gb300 as T
    import workloads as W
    sp = W.spec(1, steps=c)
    wl = W.generate(sp, dev)
    B, H, d = 1, sp.n_q_heads, sp.head_dim
    ctx = T.Context(H, sp.n_kv_heads, d, T.TS_KV_BF16, B, wl.page_table.shape[1], wl.num_pages)
    q = torch.stack([wl.q[i][0] for i in range(c)], dim=1).contiguous()
    idx = torch.zeros(B, sp.k + sp.n_sink + sp.n_local, dtype=torch.int32, device=dev)
    cnt = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.zeros(B, c, H, d, device=dev)
    lse = torch.zeros(B, c, H, device=dev)
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
    seq = wl.seq_lens(0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)

    def call():
        flush.zero_()
        ctx.prefill_chunk(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt, out, lse)

    call()
    torch.cuda.synchronize()
    ids = idx[0, :int(cnt[0])].cpu()
    n = wl.n0[0]
    vis = sum(int((ids <= n - c + i).sum()) for i in range(c))
    flops = 4.0 * vis * H * d
    ms_flush = _event_ms(lambda: flush.zero_(), 10, 3)
    ms = _event_ms(call, 10, 3) - ms_flush
    T.ts_profile_enable(ctx.handle, True)
    T.ts_profile_read(ctx.handle)
    for _ in range(10):
        call()
    torch.cuda.synchronize()
    prof = T.ts_profile_read(ctx.handle)
    att_ms, att_n = prof["attend"]
    step_ms, step_n = prof["step"]
    peak = peaks.get("bf16_tflops", 1925.7) if peaks else 1900.0
    att_tf = flops / (att_ms / att_n * 1e-3) / 1e12 if att_n else None
    st = T.ts_get_status(ctx.handle)
    ctx.close()
    return {"value": 1000.0 / ms, "unit": "chunks/s", "ms_per_chunk": ms, "chunk": c, "selected": int(cnt[0]),
            "useful_gflop": flops / 1e9, "attend_us": 1000.0 * att_ms / max(1, att_n),
            "select_us": 1000.0 * step_ms / max(1, step_n),
            "roofline": {"bound": "tensor", "achieved": att_tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": att_tf / peak if att_tf else None,
                         "kernel": "chunk_attend_kernel (tcgen05, causal, two passes)",
                         "peak_source": "measured bf16_tflops (burst)" if peaks else "fallback"},
            "status": st, "l2": "flushed before every call (256 MB write, outside the attend events)"}


def ablation_extra(dev, fn_name):
    """Decode steps of the 128K trajectory with an ablation selection function (multi-kernel path,
    no cache: every step scores and selects)."""
    import torch
    import token_level_sparse_gb300 as T
    import workloads as W
    sp = W.spec(1, steps=8)
    wl = W.generate(sp, dev)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    fn = {"logit_sum": T.TS_SCORE_LOGIT_SUM, "hard_vote": T.TS_SCORE_HEAD_HARD_VOTE}[fn_name]
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0, score_fn=fn)
    idx = torch.zeros(1, sp.k + sp.n_sink + sp.n_local, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.zeros(1, sp.n_q_heads, sp.head_dim, device=dev)
    vote = torch.zeros(1, ctx.max_tokens, device=dev)
    seq = wl.seq_lens(0)
    q = wl.q[0][0]
    ms = _event_ms(lambda: ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt, out,
                                           vote=vote), 10, 3)
    st = T.ts_get_status(ctx.handle)
    ctx.close()
    return {"value": 1000.0 / ms, "unit": UNIT, "ms_per_step": ms, "status": st,
            "l2": "not flushed: inputs larger than L2 (268 MB of K per step)"}


def page1_extra(dev):
    """Miss steps of the 128K trajectory on a token-granular pool (one token per page), which
    runs the separate kernels, beside the same separate kernels on 16-token pages."""
    import os
    import torch
    import token_level_sparse_gb300 as T
    import workloads as W
    res = {}
    for P in (1, 16):
        sp = W.spec(1, steps=4, page_size=P)
        wl = W.generate(sp, dev)
        prev = os.environ.get("TOKENSELECT_MULTI_KERNEL")
        os.environ["TOKENSELECT_MULTI_KERNEL"] = "1"
        try:
            ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1],
                            wl.num_pages, page_size=P)
        finally:
            if prev is None:
                del os.environ["TOKENSELECT_MULTI_KERNEL"]
            else:
                os.environ["TOKENSELECT_MULTI_KERNEL"] = prev
        prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
        idx = torch.zeros(1, sp.k + sp.n_sink + sp.n_local, dtype=torch.int32, device=dev)
        cnt = torch.zeros(1, dtype=torch.int32, device=dev)
        out = torch.zeros(1, sp.n_q_heads, sp.head_dim, device=dev)
        seq = wl.seq_lens(0)
        q = wl.q[0][0]
        ms = _event_ms(lambda: ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, seq, prm, idx, cnt,
                                               out), 10, 3)
        res[f"page_size_{P}"] = {"value": 1000.0 / ms, "unit": UNIT, "ms_per_step": ms,
                                 "status": T.ts_get_status(ctx.handle)}
        ctx.close()
        del wl
        torch.cuda.empty_cache()
    res["path"] = "separate kernels (cache check, score, vote, select, attend), every step a miss"
    res["l2"] = "not flushed: inputs larger than L2 (268 MB of K per step)"
    return res


OVERLAP_RHOS = (0.5, 0.7, 0.8, 0.85, 0.9, 0.925, 0.95, 0.975, 0.99, 0.999)


def overlap_pairs(wl, rhos, draws, dev, seed=7):
    """(rho, cosine, q1, q2) pairs: q2 = rho q1 + sqrt(1 - rho^2) eps with eps ~ N(0, 1) per element
    (the workload's AR(1) step), rounded to bf16 values like the workload's queries."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    q1 = wl.q[0][0]
    out = []
    for rho in rhos:
        for _ in range(draws):
            eps = torch.randn(q1.shape, generator=g, device=dev)
            q2 = (rho * q1 + math.sqrt(1.0 - rho * rho) * eps).to(torch.bfloat16).to(torch.float32).contiguous()
            c = float(torch.nn.functional.cosine_similarity(q1.reshape(1, -1), q2.reshape(1, -1)))
            out.append((rho, c, q1, q2))
    return out


def selected_part(T, ctx, wl, sp, q, idx, cnt, prm):
    """The top-k part (without sinks and window) of one fresh selection through ts_decode_step."""
    import torch
    out = torch.zeros(1, sp.n_q_heads, sp.head_dim, device=q.device)
    ctx.decode_step(q, wl.k_pool[0], wl.v_pool[0], wl.page_table, wl.seq_lens(0), prm, idx, cnt, out)
    ids = idx[0, :int(cnt[0])].cpu().numpy()
    n = wl.n0[0]
    s_end, ls = min(sp.n_sink, n), max(min(sp.n_sink, n), n - sp.n_local)
    return ids[(ids >= s_end) & (ids < ls)]


def overlap_extra(dev, draws=4):
    """Selection overlap against query cosine on the 128K workload (the TokenSelect review's
    figure 3(b), on synthetic keys): for queries at a range of cosines to a base query, the
    fraction of the base query's top-k part that the other query selects too."""
    import numpy as np
    import torch
    import token_level_sparse_gb300 as T
    import workloads as W
    sp = W.spec(1, steps=1)
    wl = W.generate(sp, dev)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    prm = T.params(k=sp.k, n_sink=sp.n_sink, n_local=sp.n_local, theta=2.0)
    idx = torch.zeros(1, sp.k + sp.n_sink + sp.n_local, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    base = selected_part(T, ctx, wl, sp, wl.q[0][0], idx, cnt, prm)
    curve = {}
    for rho, c, _, q2 in overlap_pairs(wl, OVERLAP_RHOS, draws, dev):
        part = selected_part(T, ctx, wl, sp, q2, idx, cnt, prm)
        ov = float(np.intersect1d(base, part).size) / max(1, base.size)
        curve.setdefault(rho, []).append((c, ov))
    st = T.ts_get_status(ctx.handle)
    ctx.close()
    return {"k": sp.k, "draws_per_point": draws, "status": st,
            "points": [{"rho": r, "cosine": float(np.mean([c for c, _ in v])),
                        "overlap": float(np.mean([o for _, o in v]))} for r, v in sorted(curve.items())]}


def recall_extra(dev, budget=2048):
    """Recall@budget of the best tokens by vote when the same budget is spent on blocks of
    1..128 tokens (the TokenSelect review's figure 2(b), on the 128K workload's needles)."""
    import numpy as np
    import torch
    import token_level_sparse_gb300 as T
    import workloads as W
    sp = W.spec(1, steps=1)
    wl = W.generate(sp, dev)
    ctx = T.Context(sp.n_q_heads, sp.n_kv_heads, sp.head_dim, T.TS_KV_BF16, 1, wl.page_table.shape[1], wl.num_pages)
    n = wl.n0[0]
    seq = wl.seq_lens(0)
    vote = torch.zeros(1, ctx.max_tokens, device=dev)
    ctx.score(wl.q[0][0], wl.k_pool[0], wl.page_table, seq, vote)
    idx = torch.zeros(1, budget + 128, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    v = vote.cpu().numpy()[0, :n].astype(np.float64)
    top = set(np.argsort(-v, kind="stable")[:budget].tolist())
    pts = []
    for block in (1, 2, 4, 8, 16, 32, 64, 128):
        ctx.select_blocks(vote, seq, block, budget, idx, cnt)
        sel = idx[0, :int(cnt[0])].cpu().numpy()
        pts.append({"block": block, "recall": len(top.intersection(sel.tolist())) / budget})
    st = T.ts_get_status(ctx.handle)
    ctx.close()
    return {"budget": budget, "points": pts, "status": st}


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_baseline_only:
        cpu_baseline_main()
        return
    if args.impl == "reference":
        reference_main(args)
        return
    if args.case:
        case_main(args)
        return
    import torch

    import workloads as W
    ws, rank, local = dist_env()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    cpu_base = cpu_baseline_subprocess() if rank == 0 else None      # before any CUDA work here
    torch.cuda.set_device(local)
    dist_init(ws, "nccl")
    dev = f"cuda:{local}"
    peaks = measured_peaks()
    peak_gbs = peaks.get("hbm_gbs") if peaks else 6800.0
    peak_src = "measured" if peaks else "fallback"

    sp = W.spec(1)
    bench = DecodeBench(sp, dev, theta=sp.theta, seed_offset=rank)
    bench.capture()
    barrier(ws)
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid).replace("GPU-", "")
    except Exception:  # noqa: BLE001
        gpu_id = str(local)
    # the persistent kernel's own launch time (events around it inside the graph), one step at a
    # time over the whole trajectory; this also records each trajectory step's hits and bytes
    sk = summarise(bench, bench.run(TRAJ, args.warmup), peak_gbs)
    bench.run_async(1, 3)                  # per-step graphs captured before the timed region
    with ClockSampler(gpu_id) as clk:
        t0 = time.perf_counter()
        rec = bench.run_async(args.steps, args.warmup)
        torch.cuda.synchronize()
        barrier(ws)
        wall = time.perf_counter() - t0
    s = summarise(bench, rec, peak_gbs)
    s.update({key: sk[key] for key in KERNEL_KEYS if key in sk})
    dev_s = max_over_ranks(s["ms_per_step"] * len(rec) / 1000.0, ws, dev)
    value = ws * len(rec) / dev_s

    e2e = bench.e2e(min(max(args.steps, 2 * TRAJ), 4 * TRAJ))
    e2e_v = max_over_ranks(1.0 / e2e["value"], ws, dev)
    e2e["value"] = ws / e2e_v

    extras = {}
    if not args.no_extras:
        for name, theta in (("miss_only", 2.0), ("hit_only", -1.0)):
            b2 = DecodeBench(sp, dev, theta=theta, seed_offset=rank)
            s2 = timed(b2, TRAJ, 3, peak_gbs)
            extras[name] = {k: s2[k] for k in ("value", "ms_per_step", "hit_rate", "step_gbs", "score_gbs",
                                              "miss_step_gbs") if k in s2}
            del b2
        torch.cuda.empty_cache()
        sp4 = W.spec(4)
        for name, theta in (("topp_b4_n256k_theta0.9", sp4.theta), ("topp_b4_n256k_miss_only", 2.0)):
            b4 = DecodeBench(sp4, dev, theta=theta, seed_offset=rank)
            s4 = timed(b4, sp4.steps, 3, peak_gbs, flush=False)
            extras[name] = {k: s4[k] for k in ("value", "ms_per_step", "hit_rate", "step_gbs", "score_gbs",
                                              "miss_step_gbs", "score_us_per_launch", "step_frac_of_peak",
                                              "min_step_gbs", "min_frac_of_peak") if k in s4}
            extras[name]["top_p"] = sp4.top_p
            extras[name]["bytes"] = ("step_gbs: K scan + K and V rows of every selected token; min_step_gbs: "
                                     "K scan + V rows of every selected token (dense selections attend over "
                                     "each CTA's range from the scan's logits and read no K row again)")
            extras[name]["l2"] = "not flushed: inputs larger than L2 (2.15 GB of K per step on a miss)"
            del b4
            torch.cuda.empty_cache()
        sp2 = W.spec(2)
        for name, theta in (("qwen_b8_theta0.9", sp2.theta), ("qwen_b8_miss_only", 2.0)):
            b2 = DecodeBench(sp2, dev, theta=theta, seed_offset=rank)
            s2 = timed(b2, sp2.steps, 3, peak_gbs, flush=False)
            extras[name] = {k: s2[k] for k in ("value", "ms_per_step", "hit_rate", "step_gbs", "score_gbs",
                                              "miss_step_gbs", "score_us_per_launch") if k in s2}
            if peak_gbs and "score_gbs" in s2:
                extras[name]["score_frac_of_peak"] = s2["score_gbs"] / peak_gbs
            extras[name]["l2"] = "not flushed: inputs larger than L2 (about 1 GB of K per step on a miss)"
            del b2
            torch.cuda.empty_cache()
        extras["prefill_n128k_c512"] = prefill_extra(dev, peaks)
        extras["selection_overlap_vs_cosine_n128k"] = overlap_extra(dev)
        extras["recall_vs_block_size_n128k"] = recall_extra(dev)
        extras["token_granular_pool_n128k"] = page1_extra(dev)
        torch.cuda.empty_cache()
        for fn_name in ("logit_sum", "hard_vote"):
            extras[f"ablation_{fn_name}_n128k"] = ablation_extra(dev, fn_name)
            torch.cuda.empty_cache()
        sp3 = W.spec(3)
        for name, theta in (("n1m_theta0.9", sp3.theta), ("n1m_miss_only", 2.0)):
            b3 = DecodeBench(sp3, dev, theta=theta, seed_offset=rank)
            s3 = timed(b3, 2 * sp3.steps, 3, peak_gbs, flush=False)
            extras[name] = {k: s3[k] for k in ("value", "ms_per_step", "hit_rate", "step_gbs", "score_gbs",
                                              "miss_step_gbs", "score_us_per_launch") if k in s3}
            if peak_gbs and "score_gbs" in s3:
                extras[name]["score_frac_of_peak"] = s3["score_gbs"] / peak_gbs
            extras[name]["l2"] = "not flushed: inputs larger than L2 (2.15 GB of K per layer on a miss)"
            del b3
            torch.cuda.empty_cache()

    if rank != 0:
        return
    clocks = clk.summary()
    traffic = score_traffic()
    kname = ("step_kernel (persistent: cache test, paged score, vote, select, attend; miss steps)"
             if s.get("fused") else "score_logits_kernel (paged dot product + per-CTA normaliser)")
    roof = {"bound": "hbm", "achieved": s.get("score_gbs"), "peak": peak_gbs, "unit": "GB/s",
            "frac": (s["score_gbs"] / peak_gbs) if s.get("score_gbs") else None,
            "traffic": traffic if not s.get("fused") else step_traffic(), "kernel": kname,
            "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": s.get("scan_bytes_per_launch"),
            "us_per_launch": s.get("score_us_per_launch")}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": len(rec), "warmup": args.warmup,
        "ms_per_step": s["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "llama3-8b-gqa-n128k: B1, H32/Hkv8, d128, bf16 KV in 16-token pages, "
                               "N0=131072 (+1 per step), k2048 + 4 sinks + 512 local, Selection Cache theta 0.9, "
                               "64-step AR(1) query trajectory cycled with a fresh cache each pass",
                   "l2": "flushed before every timed step (256 MB write, then 256 MB read: no dirty lines left; outside the step events)",
                   "launch": "one CUDA graph per step (cache check, score, vote, select, attend), steps "
                             "enqueued back to back; per-launch kernel times from a loop synchronised "
                             "after every step",
                   "parallelism": f"{ws} independent replica(s), no collective"},
        "hit_rate": s["hit_rate"], "step_gbs": s["step_gbs"], "miss_ms_per_step": s.get("miss_ms_per_step"),
        "hit_ms_per_step": s.get("hit_ms_per_step"), "kernel_ms_per_step": s["kernel_ms_per_step"],
        "roofline": roof, "cpu_baseline": cpu_base, "e2e": e2e,
        # the same kernel on the 1M-token, 8-layer workload's miss steps (per-launch bytes / time)
        "roofline_n1m": ({"bound": "hbm", "achieved": extras["n1m_miss_only"]["score_gbs"], "peak": peak_gbs,
                          "unit": "GB/s", "frac": extras["n1m_miss_only"]["score_gbs"] / peak_gbs,
                          "traffic": step_traffic("n1m"), "kernel": kname,
                          "us_per_launch": extras["n1m_miss_only"].get("score_us_per_launch")}
                         if "score_gbs" in extras.get("n1m_miss_only", {}) else None),
        "gpu_launches": bench.kernels_per_step * len(rec), "kernels_per_step": bench.kernels_per_step,
        "clocks": clocks, "timed_wall_s": wall, "extras": extras,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
