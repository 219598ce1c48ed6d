"""Throughput of XAttention BSA chunked prefill (estimate + select + attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload q06b_32k] [--tau 0.9]

One step = one layer's whole chunked prefill of the workload: for each chunk,
xattn_estimate -> xattn_select -> bsa_chunk_attention through the C ABI, on
one stream, inputs resident in HBM.  Prints one JSON line (rank 0).

Default workload: Qwen3-0.6B-like layer at 32K context (16 Q / 8 KV heads,
head_dim 128, 8 chunks of 4096 tokens, 128-token pages in a seeded random
permutation addressed through a [1, 256] block table, stride 8, tau 0.9).
Multi-GPU runs independent replicas (the path has no exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "prefill tokens/s per layer at 32K ctx (estimate+select+BSA), % of GB300 roofline"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(t_local_s, tokens_local, device, dist_mod=None):
    """Whole-job figures of N replicas: the slowest rank's timed seconds (MAX)
    and the tokens all ranks processed (SUM).  One process returns its own."""
    if dist_mod is None or not dist_mod.is_initialized() or dist_mod.get_world_size() == 1:
        return float(t_local_s), float(tokens_local)
    import torch
    t = torch.tensor([float(t_local_s)], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens_local)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    dist_mod.all_reduce(n, op=dist_mod.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def check_replicas(gpus, world_size):
    """--gpus N is the number of replicas the launcher started (WORLD_SIZE):
    one process per GPU, started by torch.distributed.run; a mismatch would
    time another number of GPUs than the line reports."""
    if gpus != world_size:
        raise SystemExit(f"bench.py: --gpus {gpus} but WORLD_SIZE={world_size}; start one "
                         f"process per GPU with python -m torch.distributed.run "
                         f"--nproc-per-node {gpus} bench.py --gpus {gpus}")


def workload_desc(name, tau):
    from xattention_block_sparse_gb300 import inputs as I
    c = I.CONFIGS[name]
    return (f"{name}: {c.H} Q / {c.Hkv} KV heads, head_dim {c.D}, {c.L}-token context in "
            f"{c.L // c.chunk} chunks of {c.chunk}, block {c.block}, stride {c.stride}, "
            f"tau {tau}, pages permuted via block_table [1, {c.L // c.block}]")


# ---------------------------------------------------------------------------
# Algorithmic work (per chunk): the counts the method must do
# ---------------------------------------------------------------------------

def chunk_work(cfg, c, chunk, n_sel):
    H, Hkv, D, S, Bk = cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block
    Lh, Lc = c * chunk, chunk
    rq, ch = Lc // S, Lh // S
    cells = H * (rq * ch + rq * (rq + 1) // 2)
    f_est = 2 * S * D * cells
    # estimation inputs read once (keys of every KV head, the chunk's queries);
    # the reshaped scores are an intermediate the kernels never store
    b_est_gemm = 2 * Hkv * D * (Lh + Lc) + 2 * H * Lc * D
    qb, kb = Lc // Bk, (Lh + Lc) // Bk
    b_bsum = 4 * H * qb * kb  # the block sums written
    f_att = 4 * H * D * Lc * (n_sel * Bk) + 4 * H * D * Lc * (Lc + 1) // 2
    b_att = 2 * 2 * Hkv * D * (n_sel * Bk + Lc) + 2 * 2 * H * Lc * D + 4 * H * Lc
    return dict(f_est=f_est, b_est=b_est_gemm, b_bsum=b_bsum, f_att=f_att, b_att=b_att,
                cells=cells)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.idx = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def source_sha(files):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "xattention_block_sparse_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_files, kernel_name):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel's files; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha(kernel_files)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_name \
                    and parts[1] == sha:
                return float(parts[2])
    return None


class Timed:
    """One workload resident on the device and its chunked prefill, timed step
    by step with CUDA events on one stream (estimate, select, attention of
    every chunk bracketed separately)."""

    def __init__(self, name, tau, dev, est_from_pages=False, per_kv_head=False, samples=0):
        import torch
        from xattention_block_sparse_gb300 import inputs as I
        from xattention_block_sparse_gb300 import runner as RN
        from xattention_block_sparse_gb300 import xattn as X
        self.torch, self.RN, self.X = torch, RN, X
        self.name, self.tau, self.dev = name, tau, dev
        self.est_from_pages, self.per_kv, self.samples = est_from_pages, per_kv_head, samples
        self.wl = wl = I.make_workload(name)
        self.cfg = cfg = wl.cfg
        self.L, self.chunk = cfg.L, cfg.chunk
        self.nchunk = cfg.L // cfg.chunk
        up = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev).view(
            torch.bfloat16)
        self.Q, self.K, self.V = up(wl.q_bits), up(wl.k_bits), up(wl.v_bits)
        self.KP, self.VP = up(wl.kpool_bits), up(wl.vpool_bits)
        self.BT = torch.from_numpy(wl.block_table).to(dev)
        self.seq = RN.SequencePrefill(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, self.L,
                                      self.chunk, self.BT, self.KP.shape[0],
                                      est_from_pages=est_from_pages, per_kv_head=per_kv_head,
                                      est_samples=samples)
        self.O = torch.empty((cfg.H, self.L, cfg.D), dtype=torch.bfloat16, device=dev)
        self.LSE = torch.empty((cfg.H, self.L), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.flush = torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev)

    def stages(self, c):
        """The three calls of chunk c: estimate, select, attention."""
        X, RN, cfg, b = self.X, self.RN, self.cfg, self.seq.bufs
        Q, K, V, KP, VP, st = self.Q, self.K, self.V, self.KP, self.VP, self.stream
        scale = RN.estimation_scale(cfg.D, cfg.stride)
        select = X.xattn_select_per_kv_head if self.per_kv else X.xattn_select
        attend = X.bsa_chunk_attention_per_kv_head if self.per_kv else X.bsa_chunk_attention
        p, t0 = self.seq.problems[c], c * self.chunk

        def est():
            if self.est_from_pages:
                X.xattn_estimate(p, Q[:, t0:], K[:, t0:], KP, scale, b.workspace, b.block_sums,
                                 st)
            elif self.samples:
                X.xattn_estimate_sampled(p, Q[:, t0:], K, [0], self.samples, scale, b.workspace,
                                         b.block_sums, st)
            else:  # keys in token order: K [Hkv, L, D] holds the history and the chunk
                X.xattn_estimate_seq(p, Q[:, t0:], K, [0], scale, b.workspace, b.block_sums, st)

        def sel():
            select(p, b.block_sums, self.tau, b.workspace, None, b.sel_idx, b.sel_page, b.n_sel,
                   st)

        def att():
            attend(p, Q[:, t0:], K[:, t0:], V[:, t0:], KP, VP, b.sel_page, b.n_sel,
                   1.0 / math.sqrt(cfg.D), b.workspace, self.O[:, t0:], self.LSE[:, t0:], st)

        return est, sel, att

    def step(self, ev=None):
        st = self.stream
        for c in range(self.nchunk):
            if ev is not None:
                ev[c][0].record(st)
            for i, fn in enumerate(self.stages(c)):
                fn()
                if ev is not None:
                    ev[c][i + 1].record(st)

    def stage_times(self, reps=5, rounds=3):
        """Milliseconds per step of each stage: for every chunk, the chunk's
        estimate and selection run once (so the buffers hold its selection),
        then each stage alone is timed as a CUDA graph of `reps` back-to-back
        calls (median of `rounds` replays), the way the step itself is timed:
        no host gaps between launches."""
        torch = self.torch
        tot = [0.0, 0.0, 0.0]
        st = self.stream
        for c in range(self.nchunk):
            fns = self.stages(c)
            with torch.cuda.stream(st):
                fns[0]()
                fns[1]()
            for i, fn in enumerate(fns):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=st, capture_error_mode="relaxed"):
                    for _ in range(reps):
                        fn()
                ts = []
                for _ in range(rounds):
                    with torch.cuda.stream(st):
                        e0, e1 = (torch.cuda.Event(enable_timing=True),
                                  torch.cuda.Event(enable_timing=True))
                        e0.record(st)
                        g.replay()
                        e1.record(st)
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) / reps)
                tot[i] += float(np.median(ts))
                del g
        return {"estimate_ms_per_step": tot[0], "select_ms_per_step": tot[1],
                "attention_ms_per_step": tot[2]}

    def selections(self):
        """History blocks attended per chunk (summed over KV heads and divided by
        their number for a selection per KV head): one untimed pass."""
        torch, n_sel = self.torch, []
        with torch.cuda.stream(self.stream):
            for c in range(self.nchunk):
                self.seq.run_chunk(c, self.Q, self.K, self.V, self.KP, self.VP, self.tau, self.O,
                                   self.LSE, stream=self.stream)
                n = self.seq.bufs.n_sel.view(-1).cpu().numpy()
                n_sel.append(float(n.mean()) if self.per_kv else int(n[0]))
        return n_sel

    def run(self, steps, warmup, sample_clocks=None, graph=True):
        """Eager steps (events around each step), then the timed steps: one
        replay per step of a CUDA graph of the whole step, so that the GPU never
        waits for the host between launches (eager launches of short kernels
        can outrun the host); then the stage times (stage_times, or the eager
        calls' events when no graph could be captured)."""
        torch = self.torch
        self.n_sel = self.selections()
        for _ in range(warmup):
            with torch.cuda.stream(self.stream):
                self.step()
        torch.cuda.synchronize()
        assert self.X.xattn_device_error() == 0
        events = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                   for _ in range(self.nchunk)] for _ in range(steps)]
        torch.cuda.synchronize()
        with torch.cuda.stream(self.stream):
            for s in range(steps):
                self.flush.zero_()  # L2 flush between steps (outside the step events)
                self.step(events[s])
        torch.cuda.synchronize()
        eager_ms = [events[s][0][0].elapsed_time(events[s][self.nchunk - 1][3])
                    for s in range(steps)]
        self.eager_ms = float(np.mean(eager_ms))
        eager_stage = [sum(events[s][c][i].elapsed_time(events[s][c][i + 1])
                           for s in range(steps) for c in range(self.nchunk)) / steps
                       for i in range(3)]
        self.graph, self.timing = None, "eager launches, events around each step"
        if graph:
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream, capture_error_mode="relaxed"):
                    self.step()
                torch.cuda.synchronize()
                self.graph = g
                self.timing = "one CUDA graph replay per step (the step's launches captured once)"
            except Exception as e:  # capture refused: time the eager launches
                self.timing += f" (graph capture failed: {type(e).__name__})"
        se = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        clk = ClockSampler(self.dev.index or 0) if sample_clocks else None
        t_wall = time.perf_counter()
        with torch.cuda.stream(self.stream):
            for s in range(steps):
                self.flush.zero_()
                se[s][0].record(self.stream)
                if self.graph is not None:
                    self.graph.replay()
                else:
                    self.step()
                se[s][1].record(self.stream)
        torch.cuda.synchronize()
        self.wall = time.perf_counter() - t_wall
        self.clocks = clk.stop() if clk else None
        assert self.X.xattn_device_error() == 0
        self.step_ms = [a.elapsed_time(b) for a, b in se]
        if self.graph is not None:
            self.stage = self.stage_times()
            self.stage_timing = "per chunk, each stage alone as a CUDA graph of 5 calls"
        else:
            self.stage = {"estimate_ms_per_step": eager_stage[0],
                          "select_ms_per_step": eager_stage[1],
                          "attention_ms_per_step": eager_stage[2]}
            self.stage_timing = "eager calls, CUDA events around each call"
        self.steps = steps
        return self

    def density(self):
        avail = sum(c * self.chunk // self.cfg.block for c in range(self.nchunk))
        return sum(self.n_sel) / max(1, avail)

    def work(self):
        return [chunk_work(self.cfg, c, self.chunk, self.n_sel[c]) for c in range(self.nchunk)]

    def summary(self, peaks):
        """Rates of the timed run: tokens/s, the attention's algorithmic TFLOP/s
        per launch (on the FLOPs of the blocks it attends), the estimate's."""
        work = self.work()
        ms = float(np.mean(self.step_ms))
        f_att = sum(w["f_att"] for w in work)
        f_est = sum(w["f_est"] for w in work)
        att_launch_ms = self.stage["attention_ms_per_step"] / self.nchunk
        att_tflops = (f_att / self.nchunk) / (att_launch_ms * 1e-3) / 1e12
        est_tflops = f_est / (self.stage["estimate_ms_per_step"] * 1e-3) / 1e12
        return {"value": self.L / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
                "ms_per_step_eager": self.eager_ms, "timing": self.timing,
                "density": self.density(), "n_sel_per_chunk": self.n_sel,
                "attention": {"achieved_tflops": att_tflops,
                              "frac": att_tflops / peaks["bf16_tflops"],
                              "flops_per_step": f_att, "launch_ms": att_launch_ms},
                "estimate": {"achieved_tflops": est_tflops,
                             "frac": est_tflops / peaks["bf16_tflops"]},
                **self.stage}

    def release(self):
        for name in ("graph", "Q", "K", "V", "KP", "VP", "O", "LSE", "flush", "seq", "wl"):
            setattr(self, name, None)
        self.torch.cuda.empty_cache()


def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist
    from xattention_block_sparse_gb300 import runner as RN
    from xattention_block_sparse_gb300 import xattn as X

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from __graft_entry__ import build
    if rank == 0 or ws == 1:
        build()
    if ws > 1:
        dist.barrier()
    X.load_library()

    tau = args.tau
    T = Timed(args.workload, tau, dev, est_from_pages=args.est_from_pages)
    cfg, L, chunk, nchunk = T.cfg, T.L, T.chunk, T.nchunk
    if ws > 1:
        dist.barrier()
    T.run(args.steps, args.warmup, sample_clocks=True, graph=not args.eager)
    if ws > 1:
        dist.barrier()
    step_ms, stage, clocks, wall, n_sel = T.step_ms, T.stage, T.clocks, T.wall, T.n_sel
    ms = float(np.mean(step_ms))
    t_max, tokens = aggregate_over_ranks(sum(step_ms) / 1e3, L * args.steps, dev,
                                         dist if ws > 1 else None)

    work = T.work()
    K_ = args.steps
    b_bs = sum(w["b_bsum"] for w in work)
    peaks, peak_src = load_peaks()
    summ = T.summary(peaks)
    att_tflops = summ["attention"]["achieved_tflops"]
    att_launch_ms = summ["attention"]["launch_ms"]
    value = tokens / t_max

    # roofline of the step: algorithmic time at peak over measured time
    t_roof = sum(max(w["f_est"] / (peaks["bf16_tflops"] * 1e12),
                     (w["b_est"] + w["b_bsum"]) / (peaks["hbm_gbs"] * 1e9))
                 + max(w["f_att"] / (peaks["bf16_tflops"] * 1e12),
                       w["b_att"] / (peaks["hbm_gbs"] * 1e9)) for w in work)

    # end to end through the public API with host buffers
    e2e = run_e2e(args, T.wl, cfg, T.seq, tau, dev, T.stream, X, RN, torch, nchunk, chunk)
    density = T.density()
    wl = T.wl
    T.release()

    # the same step on the sparse workload (density near the pages' 32K figure):
    # the page gather at partial density, with the vote and with one block set
    # per KV head
    extra = {}
    if not args.skip_sparse:
        for key, per_kv, samples in (("sparse", False, 0), ("sparse_per_kv_head", True, 0),
                                     ("sparse_sampled_estimate", False, 4)):
            S_ = Timed("q06b_32k_sparse", tau, dev, per_kv_head=per_kv, samples=samples)
            S_.run(args.steps, args.warmup, graph=not args.eager)
            extra[key] = {"workload": workload_desc("q06b_32k_sparse", tau)
                          + (", one block set per KV head" if per_kv else ", majority vote")
                          + (f", history estimated from the first {samples} of each block's "
                             f"16 reshaped columns" if samples else ""),
                          **S_.summary(peaks)}
            S_.release()

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": K_,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_per_step_median": float(np.median(step_ms)),
        "ms_per_step_best": float(min(step_ms)),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 with RoPE theta 1e6; no model weights)",
        "config": {"workload": workload_desc(args.workload, tau), "tokens_per_step": L,
                   "chunks": nchunk, "l2": "flushed between steps (256 MiB write)",
                   "parallelism": f"replicas x{ws}", "timing": T.timing,
                   "stage_times": T.stage_timing},
        "ms_per_step_eager": T.eager_ms,
        "roofline": {"bound": "tensor", "kernel": "attn_tc_kernel (bsa_chunk_attention)",
                     "achieved": att_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": att_tflops / peaks["bf16_tflops"],
                     "frac_sustained": att_tflops / peaks["bf16_tflops_sustained"],
                     "peak_source": peak_src,
                     "traffic": traffic_for(("attention.cu", "tc_common.cuh", "common.cuh"),
                                            "attn_tc_kernel"),
                     "launch_ms": att_launch_ms},
        "step_roofline": {"t_roof_ms": t_roof * 1e3, "t_meas_ms": ms,
                          "frac": t_roof * 1e3 / ms},
        "kernels": {"estimate": summ["estimate"],
                    "block_sum_bytes_per_step": b_bs, **stage},
        "density": density,
        "n_sel_per_chunk": n_sel,
        "clocks": clocks,
        "e2e": e2e,
        # per chunk, this library's kernels: score GEMM, block sums, select (+ vote),
        # attention -- the first chunk, with no history to select from, launches no
        # select (n_sel cleared) -- plus cudaMemsetAsync of counters (not counted)
        "gpu_launches": (4 * nchunk - 1) * K_,
        "wall_s_timed": wall,
        **extra,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args, wl, n_sel)
        print(json.dumps(line), flush=True)


def run_e2e(args, wl, cfg, seq, tau, dev, stream, X, RN, torch, nchunk, chunk):
    """Same metric through the public API with pinned HOST buffers: every step
    copies the layer's Q, K, V host->device chunk by chunk, the copies of later
    chunks overlapped with the compute of earlier ones, and O and LSE reach
    the host buffers within the step (`SequencePrefill.run_from_host`): copied
    back per chunk on a side stream, or, with --e2e-direct-out, written there
    by the attention kernel itself.  The page pools are this sequence's own
    keys and values: each chunk's K/V are stored into their pages on the
    device (xattn_store_kv) before the chunk's attention, so the history the
    next chunk reads is built in place rather than copied in.  Timed twice:
    steps one after the other ('serial'), and steps pipelined through two
    device buffer sets (runner.HostFedPipeline), the headline value."""
    pin = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(
        torch.bfloat16).pin_memory()
    L = cfg.L
    host = {"q": pin(wl.q_bits), "k": pin(wl.k_bits), "v": pin(wl.v_bits),
            "o": torch.empty((cfg.H, L, cfg.D), dtype=torch.bfloat16).pin_memory(),
            "lse": torch.empty((cfg.H, L), dtype=torch.float32).pin_memory()}
    devb = {k: torch.empty_like(t, device=dev) for k, t in host.items()}
    for name, bits in (("kpool", wl.kpool_bits), ("vpool", wl.vpool_bits)):
        devb[name] = torch.empty(bits.shape, dtype=torch.bfloat16, device=dev)
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v"))
    d2h = sum(host[k].numel() * host[k].element_size() for k in ("o", "lse"))
    h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    def one():
        seq.run_from_host(host, devb, tau, stream, h2d_stream, d2h_stream, store_kv=True,
                          out_direct=args.e2e_direct_out)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    # the step's launches and copies captured once (all three streams, joined
    # back into `stream` by run_from_host's events) and replayed every step:
    # every replay moves the step's bytes host -> device and back again
    graph, timing = None, "eager launches"
    if not args.eager:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                one()
            torch.cuda.synchronize()
            graph, timing = g, "one CUDA graph replay per step (copies and launches captured once)"
        except Exception as e:  # capture refused: time the eager calls
            timing += f" (graph capture failed: {type(e).__name__})"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, args.steps)
    e0.record(stream)
    for _ in range(steps):
        if graph is not None:
            with torch.cuda.stream(stream):
                graph.replay()
        else:
            one()
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    serial = {"value": L * steps / t, "ms_per_step": t * 1e3 / steps, "timing": timing,
              "overlap": "each step's copies wait for the step before to finish"}
    # Steps pipelined (runner.HostFedPipeline): a second device buffer set, so
    # the next step's Q, K, V cross while this one computes and this one's O
    # and LSE come back while the next one computes; every step still moves
    # all its bytes inside the timed region.  The K steps are captured as one
    # CUDA graph (launched eagerly they would be bound by the host's launch
    # rate) and timed as one replay.
    devb2 = {k: torch.empty_like(devb[k]) for k in ("q", "k", "v", "o", "lse")}
    devb2["kpool"], devb2["vpool"] = devb["kpool"], devb["vpool"]

    def many(n):
        pipe = RN.HostFedPipeline(seq, [devb, devb2], stream, h2d_stream, d2h_stream,
                                  store_kv=True, out_direct=args.e2e_direct_out)
        for _ in range(n):
            pipe.submit(host, tau)
        pipe.join()

    with torch.cuda.stream(stream):
        many(2)
    torch.cuda.synchronize()
    pipelined = None
    if not args.eager:
        try:
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp, stream=stream, capture_error_mode="relaxed"):
                many(steps)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                gp.replay()  # warm-up replay
            torch.cuda.synchronize()
            e0.record(stream)
            with torch.cuda.stream(stream):
                gp.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            tp = e0.elapsed_time(e1) / 1e3
            pipelined = {"value": L * steps / tp, "ms_per_step": tp * 1e3 / steps,
                         "timing": f"{steps} steps captured as one CUDA graph, one replay timed",
                         "overlap": "two device buffer sets: a step's copies overlap the "
                                    "neighbouring steps' compute"}
        except Exception as e:  # capture refused: report the serial steps only
            pipelined = None
            serial["pipelined"] = f"graph capture failed: {type(e).__name__}"
    head = pipelined if pipelined is not None else serial
    return {"value": head["value"], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": head["ms_per_step"],
            "timing": head["timing"], "pipelined": pipelined is not None,
            "serial": serial,
            "copies": "Q, K, V copied chunk by chunk on one side stream, overlapped with "
                      "earlier chunks' compute (a chunk's estimate waits for its Q and K, "
                      "its attention for V too); each chunk's K/V stored into its pool pages "
                      "on the device (xattn_store_kv) before its attention; "
                      + ("O and LSE written into the pinned host buffers by the attention "
                         "kernel itself (d2h bytes: those stores)" if args.e2e_direct_out else
                         "O and LSE read back per chunk on another side stream")}


# ---------------------------------------------------------------------------
# Oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_chunk_sample(wl, cfg, c, chunk, tau, rows_per_chunk, oracle):
    """Estimate + select on the whole chunk c; attention on `rows_per_chunk`
    evenly spread query rows, extrapolated to the chunk.  Returns
    (tokens represented, seconds, seconds measured)."""
    O = oracle
    t0, t1 = c * chunk, (c + 1) * chunk
    q = wl._f64_cache["q"]
    k = wl._f64_cache["k"]
    v = wl._f64_cache["v"]
    kp, vp = wl._f64_cache["kpool"], wl._f64_cache["vpool"]
    s0 = time.perf_counter()
    bs = O.estimate_request(q[:, t0:t1], k[:, t0:t1], kp, wl.block_table[0], t0, cfg.H, cfg.Hkv,
                            cfg.stride, cfg.block, O.default_estimation_scale(cfg.D, cfg.stride))
    _, _, pages = O.select_request(bs.astype(np.float32), tau, cfg.Hkv, t0 // cfg.block,
                                   wl.block_table[0])
    s1 = time.perf_counter()
    rows = np.linspace(0, chunk - 1, rows_per_chunk).astype(int)
    O.attend_request(q[:, t0:t1], k[:, t0:t1], v[:, t0:t1], kp, vp, pages, cfg.H, cfg.Hkv,
                     1 / math.sqrt(cfg.D), rows=rows)
    s2 = time.perf_counter()
    est = (s1 - s0) + (s2 - s1) * chunk / rows_per_chunk
    return chunk, est, s2 - s0


def _prep_oracle(wl):
    wl._f64_cache = {n: wl.f64(n) for n in ("q", "k", "v", "kpool", "vpool")}


def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max((i.get("num_threads", 0) for i in info), default=os.cpu_count())
    except Exception:
        return os.cpu_count()


def cpu_baseline(args, wl, n_sel):
    from oracle import xattn_oracle as O
    cfg = wl.cfg
    chunk = cfg.chunk
    nchunk = cfg.L // chunk
    _prep_oracle(wl)
    rows = 32
    tok = sec = meas = 0.0
    for c in range(nchunk):
        a, b, m = oracle_chunk_sample(wl, cfg, c, chunk, args.tau, rows, O)
        tok += a
        sec += b
        meas += m
    return {"value": tok / sec, "unit": "tokens/s", "cores": _blas_threads(),
            "host_cpus": os.cpu_count(), "kind": "oracle",
            "value_basis": "extrapolated",
            "measured_s": meas, "seconds_extrapolated": sec,
            "sample": (f"float64 oracle on all {nchunk} chunks: estimate + select in full, "
                       f"attention on {rows} of {chunk} query rows per chunk; value = "
                       f"{int(tok)} tokens / {sec:.1f} s, the attention time scaled linearly "
                       f"from the sampled rows to the chunk ({meas:.1f} s measured)")}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    from oracle import xattn_oracle as O
    from xattention_block_sparse_gb300 import inputs as I
    wl = I.make_workload(args.workload)
    cfg = wl.cfg
    chunk = cfg.chunk
    nchunk = cfg.L // chunk
    _prep_oracle(wl)
    rows = 16
    for s in range(args.warmup):
        oracle_chunk_sample(wl, cfg, s % nchunk, chunk, args.tau, rows, O)
    tok = sec = meas = 0.0
    for s in range(args.steps):
        a, b, m = oracle_chunk_sample(wl, cfg, s % nchunk, chunk, args.tau, rows, O)
        tok += a
        sec += b
        meas += m
    value = tok / sec
    cores = _blas_threads()
    steps = max(1, args.steps)
    sample = (f"each step: one chunk (chunk index = step mod {nchunk}), estimate + select in "
              f"full, attention on {rows} of {chunk} query rows; value = tokens / the "
              f"step's seconds with the attention scaled linearly to the chunk "
              f"({sec:.1f} s extrapolated, {meas:.1f} s measured)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "value_basis": "extrapolated",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        # measured wall time of each step's sample; the extrapolated chunk time beside it
        "ms_per_step": meas * 1e3 / steps, "ms_per_step_extrapolated": sec * 1e3 / steps,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, args.tau)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "value_basis": "extrapolated", "measured_s": meas,
                         "seconds_extrapolated": sec, "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="q06b_32k")
    ap.add_argument("--tau", type=float, default=0.9)
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of replays of a CUDA graph of the step")
    ap.add_argument("--skip-sparse", action="store_true",
                    help="time only the headline workload (no sparse-workload lines)")
    ap.add_argument("--e2e-direct-out", action="store_true",
                    help="end-to-end leg: the attention writes O and LSE into the pinned "
                         "host buffers itself instead of a copy back per chunk")
    ap.add_argument("--est-from-pages", action="store_true",
                    help="estimate from the history pages (xattn_estimate) instead of the "
                         "keys in token order (xattn_estimate_seq)")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    check_replicas(args.gpus, ws)
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
