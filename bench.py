"""Benchmark of the MARché decode-step hot path on the MAR-H-shaped workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

Workload (default ``--config mar_h``): batch 256 doubled to 512 rows for classifier-free
guidance, 16 heads, head dim 80, 320 tokens (256 image + 64 buffer), bf16; a cached step
has 4 generating + 4 just-decoded + top-32 refresh tokens (A = 40 active queries). The
inputs are seeded synthetic tensors; two independent input sets (each ~3.4 GB, far larger
than the 129 MB L2) alternate from step to step.

One bench step is one cached decode step through the two layers the hot path changes:
layer-2 full attention with the head-averaged score, the top-K refresh set and the
active set; layer-3 cache-aware attention of the active queries (their rows read in place
from the fresh Q/K/V, the KV-cache scatter in the same launch); the condition-cache apply.
``value`` = active-query tokens of the cache-aware layer (B' * A per step) over the device
time of the K timed steps, launched eagerly (each step keeps the GPU busy for ~0.8 ms,
far longer than its launches take on the host). ``roofline`` is the cache-aware launch,
timed with CUDA events around it inside the timed region. The other legs: the refresh
step (step % 3 == 0: full attention of both layers, the whole-cache overwrite, the
condition-cache update; B' * N tokens), the schedule average, per-call device times,
the active-set sweep (A = 2 % .. 50 % of N), the refresh-count sweep (K = 16 .. 64), the
512 px shape's tensor-bound full attention, the end-to-end leg through the C ABI with
pinned host buffers, and the fp64 oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "cache-aware attn active-query tok/s per layer; HBM GB/s & % roofline, 1 GB300"
UNIT = "tok/s"
DEFAULT_CONFIG = "mar_h"
N_SETS = 2
REFRESH_PERIOD = 3
K_SWEEP = (16, 32, 64)
# DRAM traffic per launch from committed ncu captures: one line per kernel and workload,
# keyed by a hash of the kernel's sources so that a capture of an older build is not used
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
KERNEL_SOURCES = {
    "attn_tc5": ["attn_tc5.cu", "attn_tc5_q96.cu", "tc5.cuh", "common.cuh", "attn.h", "tma_host.h"],
}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=ws)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.rows, self.proc = gpu, [], None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [r for t, r in self.rows if self.t0 and self.t1 and self.t0 <= t <= self.t1] or \
               [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- workload
def host_schedule(cfg, seed: int):
    """Generating and exclusion ([generating, just-decoded]) positions of one step, drawn
    from the image tokens and shared by the cond and uncond rows of an image."""
    pos = workloads.distinct_positions(cfg.B, cfg.G + cfg.J, cfg.n_buf, cfg.N, seed)
    pos = torch.cat([pos, pos], 0) if cfg.cfg else pos
    return pos[:, :cfg.G].contiguous(), pos.contiguous()


class InputSet:
    def __init__(self, cfg, s, device):
        ss = workloads.single_step(cfg, device=device, seed=cfg.seed * 100 + s)
        self.layer2 = (ss.Q2, ss.K2, ss.V2)
        self.layer3 = (ss.Q3, ss.K3, ss.V3)
        self.cache = (ss.Kc, ss.Vc)
        self.cond, self.uncond, self.residual = ss.cond, ss.uncond, ss.residual
        self.gen, self.exclude = (x.to(device) for x in host_schedule(cfg, 7000 + 17 * s))

    def host_copy(self):
        """Pinned host copies of the per-step inputs (for the end-to-end leg)."""
        pin = lambda x: x.detach().to("cpu").pin_memory()
        return {"layer2": [pin(x) for x in self.layer2], "layer3": [pin(x) for x in self.layer3],
                "gen": pin(self.gen), "exclude": pin(self.exclude), "cond": pin(self.cond)}


# Algorithmic bytes per call (bf16 = 2 bytes per element)
def bytes_full_attention(cfg):
    return 4 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2          # Q, K, V read + O write


def bytes_cache_aware(cfg, A):
    """Cached K/V read 4 (N - A) d, active Q/K/V read 6 A d, O write 2 A d per (b, h), positions."""
    per_bh = 4 * (cfg.N - A) * cfg.d + 6 * A * cfg.d + 2 * A * cfg.d
    return cfg.Bp * cfg.H * per_bh + cfg.Bp * A * 4


def bytes_scatter(cfg, A):
    """The fused KV-cache scatter: K and V rows of the active positions written, 4 A d per (b, h)."""
    return cfg.Bp * cfg.H * 4 * A * cfg.d


def kernel_build_key(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "cache_aware_attention_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the committed ncu
    summary, or None when there is none for the current build of the kernel."""
    key = kernel_build_key(kernel)
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and \
                        parts[1] == key and parts[2] == workload:
                    return float(parts[3])
    except OSError:
        pass
    return None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def graph_time(fn, n_sets: int, reps: int = 24) -> float:
    """Per-call device time (us) of fn(set index): one CUDA graph of `reps` back-to-back calls,
    the input sets rotating, replayed once to warm up and then timed with CUDA events on the
    replaying stream (host launch overhead excluded, the short gaps between kernels included)."""
    fn(0)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for r in range(reps):
            fn(r % n_sets)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) * 1e3 / reps


# ----------------------------------------------------------------------------- our arm
def config_from_args(args):
    cfg = workloads.CONFIGS[args.config]
    if cfg.G == 0:
        # a decode-loop config: its largest step (the cosine schedule's most generating tokens,
        # as many just decoded)
        g = max(workloads.cosine_schedule(cfg.n_img, cfg.steps))
        cfg = cfg.scaled(G=g, J=g)
    if args.rows:
        cfg = cfg.scaled(B=args.rows // 2 if cfg.cfg else args.rows)
    return cfg


def run_mine(args, ws, rank, local):
    import cache_aware_attention_gb300 as mar
    from cache_aware_attention_gb300 import _build
    from cache_aware_attention_gb300.step import DecodeStep, is_full_refresh

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    barrier(ws)
    mar.load()
    cfg = config_from_args(args)
    A = cfg.A
    sets = [InputSet(cfg, s, dev) for s in range(N_SETS)]
    # the caches hold finite values (seeded, as a refresh step leaves them), so the decode step
    # passes that guarantee to the cache-aware launch (MAR_CA_STALE_FINITE)
    step = DecodeStep(cfg.Bp, cfg.H, cfg.N, cfg.d, max(K_SWEEP + (cfg.K,)), max(cfg.sweep_A + (A, cfg.G + cfg.J + max(K_SWEEP))),
                      device=dev, max_gen=cfg.G, stale_finite=True)
    step.K = cfg.K
    if args.only:
        # profiling aid: one layer-2 select call (fills the score and the active set the
        # other calls read), then --reps calls of the named kind, input sets rotating
        calls, _ = step_calls(cfg, step, mar)
        calls = {k: v for k, v in calls.items() if not k.startswith(("_", "torch_"))}
        if args.only not in calls:
            raise SystemExit(f"--only: one of {sorted(calls)}")
        calls["attn_full_select"](sets[0])
        for r in range(args.reps):
            calls[args.only](sets[r % N_SETS])
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"only": args.only, "reps": args.reps, "config": args.config, "rows": cfg.Bp,
                              "status": "ok"}))
        return

    # cached steps are those with t % 3 != 0; refresh steps those with t % 3 == 0
    cached_t = [t for t in range(1, 3 * (args.warmup + args.steps) + 3) if not is_full_refresh(t)]

    def cached_step(i, events=None):
        t = cached_t[i]
        s = sets[i % N_SETS]
        kind = step.run(t, s.layer2, s.layer3, s.cache, s.gen, s.exclude, events=events)[0]
        assert kind == "cached"
        mar.mar_cfg_residual(mar.MAR_CFG_APPLY, s.cond, s.uncond, s.residual)

    clocks = ClockSampler(local)
    clocks.start()
    W, K = args.warmup, args.steps
    for i in range(W):
        cached_step(i)
    torch.cuda.synchronize()

    # timed region: exactly K cached steps, eager launches; events around each cache-aware launch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    ev0.record()
    for i in range(K):
        cached_step(W + i, events=evs[i])
    ev1.record()
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier(ws)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, ws)
    total_tokens = cfg.Bp * A * K * ws
    ca_us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    ca_mean = statistics.fmean(ca_us)
    assert mar.mar_status_read(step.status) == 0, "device reported an index error"

    legs = args.legs != "none"
    refresh = refresh_leg(args, cfg, sets, step, mar, is_full_refresh) if legs else None
    schedule = schedule_leg(cfg, sets, step, mar, is_full_refresh) if legs else None
    brk = breakdown(cfg, sets, step, mar) if legs else None
    sweep_a = sweep_active(cfg, sets, step, mar) if legs else None
    sweep_k = sweep_refresh_count(cfg, sets, step, mar) if legs else None
    e2e = end_to_end(args, cfg, sets, step, mar, cached_t) if legs else None
    clocks.stop()
    del sets
    torch.cuda.empty_cache()
    px = px512_leg(mar, dev) if legs and not args.no_px512 else None

    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    b_a3 = bytes_cache_aware(cfg, A)
    b_launch = b_a3 + bytes_scatter(cfg, A)
    wl = f"{args.config}-A{A}" + (f"-rows{cfg.Bp}" if args.rows else "")
    traffic = dram_traffic("attn_tc5", wl)
    roof = {"bound": "hbm",
            "kernel": f"attn_tc5_kernel<{cfg.d},0>: cache-aware attention, active rows read in place, fused "
                      f"KV-cache scatter ({cfg.Bp}x{cfg.H}, N={cfg.N}, d={cfg.d}, A={A})",
            "achieved": b_launch / (ca_mean * 1e-6) / 1e9, "peak": hbm, "unit": "GB/s",
            "frac": b_launch / (ca_mean * 1e-6) / 1e9 / hbm,
            "traffic": traffic,
            "algorithmic_bytes": b_launch,
            "bytes_note": "cached K/V 4(N-A)d + active Q/K/V 6Ad + O 2Ad per (b,h) + positions, plus the fused "
                          "scatter's 4Ad per (b,h)",
            "frac_without_scatter": b_a3 / (ca_mean * 1e-6) / 1e9 / hbm,
            "launch_us_mean": ca_mean, "launch_us_median": statistics.median(ca_us), "launches_timed": K,
            "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured copy)" if "hbm_gbs" in peaks
                           else "fallback 6800 GB/s",
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, committed capture of "
                              "this kernel build" if traffic else "no capture of this kernel build"}
    cpu = cpu_baseline(cfg, budget_s=args.cpu_seconds) if (rank == 0 and ws == 1 and legs and not args.no_cpu) \
        else None
    line = {
        "metric": METRIC, "value": total_tokens / (ms_max / 1e3), "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"MAR-H-shaped cached decode step ({cfg.B} images doubled to {cfg.Bp} rows for CFG, "
                               f"{cfg.H} heads, d={cfg.d}, {cfg.n_img}+{cfg.n_buf} tokens, {cfg.G} gen + {cfg.J} "
                               f"just-decoded + top-{cfg.K} refresh = {A} active)" if args.config == "mar_h"
                   else f"{args.config} cached decode step ({cfg.Bp} rows, {cfg.H} heads, d={cfg.d}, N={cfg.N}, A={A})",
                   "name": args.config, "B_rows": cfg.Bp, "heads": cfg.H, "head_dim": cfg.d, "tokens": cfg.N,
                   "active": A, "refresh_K": cfg.K,
                   "unit_tokens": "B'*A active queries of the cache-aware layer per cached step",
                   "step": "layer-2 full attention + score + top-K + active set; layer-3 cache-aware attention "
                           "(active rows read in place, fused scatter); condition-cache apply",
                   "l2": f"inputs larger than L2: {N_SETS} alternating input sets of "
                         f"~{(8 * bytes_full_attention(cfg) // 4) // 2**20} MB each, no flush",
                   "timing": "eager launches, CUDA events on the stream around the K timed steps"},
        "roofline": roof,
        "refresh_step": refresh,
        "schedule": schedule,
        "sweep_active": sweep_a,
        "sweep_refresh_k": sweep_k,
        "px512": px,
        "breakdown": brk,
        "e2e": e2e,
        "gpu_launches": 5 * K,
        "gpu_launches_note": "per cached step: layer-2 attention with the raw scores, score reduction, top-K, "
                             "cache-aware attention, condition cache",
        "cpu_baseline": cpu,
        "clocks": clocks.summary(),
        # The pages' own figures, end to end on whole images with trained models (one H100,
        # ImageNet 256): context only, not comparable with a per-step kernel figure.
        "context": {"marche_end_to_end_speedup_over_mar": {"B": 1.57, "L": 1.68, "H": 1.79},
                    "marche_speedup_stated_in_the_review": "1.57-1.72x",
                    "marche_cache_aware_attention_alone_mar_b": 1.55,
                    "lazymar_speedup": 2.83,
                    "source": "MARche notes: Main Results table, Speedup Component Breakdown; the MARche "
                              "review; LazyMAR notes: main results and ablation (token + condition cache)"},
    }
    if rank == 0:
        print(json.dumps(line))


def refresh_leg(args, cfg, sets, step, mar, is_full_refresh):
    """Refresh steps (t % 3 == 0), eager: device time per step and of the layer-3 launch."""
    n = max(12, args.steps // 10)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(3):
        s = sets[i % N_SETS]
        step.run(3 * i, s.layer2, s.layer3, s.cache, s.gen, s.exclude)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        s = sets[i % N_SETS]
        step.run(3 * i, s.layer2, s.layer3, s.cache, s.gen, s.exclude, events=evs[i])
        mar.mar_cfg_residual(mar.MAR_CFG_UPDATE, s.cond, s.uncond, s.residual)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    l3 = statistics.fmean(a.elapsed_time(b) * 1e3 for a, b in evs)
    b3 = bytes_full_attention(cfg) + 2 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2
    return {"ms_per_step": ms, "tok_s": cfg.Bp * cfg.N / (ms / 1e3), "unit_tokens": "B'*N (every token active)",
            "steps": n, "layer3_launch_us": l3, "layer3_gbs": b3 / (l3 * 1e-6) / 1e9,
            "layer3_bytes": b3, "launches_per_step": 3}


def schedule_leg(cfg, sets, step, mar, is_full_refresh, n: int = 30):
    """Decode steps following the refresh schedule (one refresh step in three), eager."""
    A = cfg.A
    for t in range(3):
        s = sets[t % N_SETS]
        step.run(t, s.layer2, s.layer3, s.cache, s.gen, s.exclude)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    cached_tokens = 0
    for t in range(3, 3 + n):
        s = sets[t % N_SETS]
        kind = step.run(t, s.layer2, s.layer3, s.cache, s.gen, s.exclude)[0]
        mode = mar.MAR_CFG_UPDATE if kind == "full" else mar.MAR_CFG_APPLY
        mar.mar_cfg_residual(mode, s.cond, s.uncond, s.residual)
        cached_tokens += cfg.Bp * A if kind == "cached" else 0
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"steps": n, "ms_per_step": ms / n, "refresh_every": REFRESH_PERIOD,
            "cached_step_tok_s": cached_tokens / (ms / 1e3),
            "note": "B'*A tokens of the cached steps over the time of all steps (refresh steps included)"}


def step_calls(cfg, step, mar, A=None, K=None):
    """The C-ABI calls of the step (and of the next rows), by name, each a function of one
    input set, with the algorithmic bytes of one call."""
    A = cfg.A if A is None else A
    K = cfg.K if K is None else K
    act = step.active(A)
    oa = step.dense(3, A)
    dev = step.score.device
    R = step.refresh_set(K)
    # dense active blocks for the two-call form (gather, then cache-aware attention)
    qa, ka, va = (torch.empty(cfg.Bp, cfg.H, A, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(3))
    cos_buf = torch.empty(cfg.Bp, cfg.N, dtype=torch.float32, device=dev)
    sel_idx = torch.empty(cfg.Bp, cfg.N, dtype=torch.int32, device=dev)
    sel_cnt = torch.empty(cfg.Bp, dtype=torch.int32, device=dev)
    # the cached positions of each row (the complement of the active set), for the context call
    cached_idx = torch.empty(cfg.Bp, cfg.N - A, dtype=torch.int64, device=dev)
    calls = {
        "attn_full": lambda s: mar.mar_attn_full(s.layer2[0], s.layer2[1], s.layer2[2], step.O2),
        "attn_full+score": lambda s: mar.mar_attn_full(s.layer2[0], s.layer2[1], s.layer2[2], step.O2,
                                                       gen_idx=s.gen, score_out=step.score,
                                                       workspace=step.workspace),
        "topk": lambda s: mar.mar_refresh_topk(step.score, s.exclude, K, out_idx=R, active_out=act),
        "attn_full_select": lambda s: mar.mar_attn_full_select(s.layer2[0], s.layer2[1], s.layer2[2], s.gen, s.exclude,
                                                               K, step.score, O=step.O2, out_idx=R,
                                                               active_out=act, workspace=step.workspace),
        "gather": lambda s: mar.mar_kv_gather(list(s.layer3), act, dsts=[qa, ka, va]),
        "cache_aware": lambda s: mar.mar_attn_cache_aware(qa, ka, va, s.cache[0], s.cache[1], act, O_A=oa,
                                                          fuse_scatter=True, stale_finite=step.stale_finite),
        "cache_aware_gather": lambda s: mar.mar_attn_cache_aware_gather(s.layer3[0], s.layer3[1], s.layer3[2],
                                                                        s.cache[0], s.cache[1], act, O_A=oa,
                                                                        fuse_scatter=True,
                                                                        stale_finite=step.stale_finite),
        # the same launch without the finite-cache guarantee: the stale V rows are zeroed first
        "cache_aware_gather_zeroed": lambda s: mar.mar_attn_cache_aware_gather(s.layer3[0], s.layer3[1],
                                                                               s.layer3[2], s.cache[0], s.cache[1],
                                                                               act, O_A=oa, fuse_scatter=True),
        "attn_full_refresh": lambda s: mar.mar_attn_full_refresh(s.layer3[0], s.layer3[1], s.layer3[2], s.cache[0],
                                                                 s.cache[1], step.O3),
        "cfg": lambda s: mar.mar_cfg_residual(mar.MAR_CFG_APPLY, s.cond, s.uncond, s.residual),
        # next rows, outside the step: KV-drift cosine of the layer-3 cache against the fresh
        # keys, the token cache's recompute set on those similarities, the shared refresh set
        "token_cosine": lambda s: mar.mar_token_cosine(s.cache[0], s.layer3[1], out=cos_buf),
        "select_recompute": lambda s: mar.mar_select_recompute(cos_buf, 0.999, s.exclude, out_idx=sel_idx,
                                                               out_count=sel_cnt),
        "topk_pairs": lambda s: mar.mar_refresh_topk_pairs(step.score, s.exclude, K, out_idx=R,
                                                           active_out=act),
        # context only (not this library): the concatenating alternative of MARché's Figure 7 --
        # gather the active rows and the cached rows, concatenate, PyTorch's fused attention,
        # then the cache update
        "torch_concat_sdpa (context)": lambda s: torch_concat_sdpa(s, act, cached_idx),
    }
    E = cfg.G + cfg.J
    algo = {"attn_full": bytes_full_attention(cfg),
            "attn_full+score": bytes_full_attention(cfg),
            "topk": cfg.Bp * cfg.N * 4 + cfg.Bp * (E + K) * 4,
            "attn_full_select": bytes_full_attention(cfg),
            "gather": 2 * 3 * cfg.Bp * cfg.H * A * cfg.d * 2,
            "cache_aware": bytes_cache_aware(cfg, A) + bytes_scatter(cfg, A),
            "cache_aware_gather": bytes_cache_aware(cfg, A) + bytes_scatter(cfg, A),
            "cache_aware_gather_zeroed": bytes_cache_aware(cfg, A) + bytes_scatter(cfg, A),
            "attn_full_refresh": bytes_full_attention(cfg) + 2 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2,
            "cfg": 3 * cfg.B * cfg.n_img * cfg.latent * 4,
            "token_cosine": 2 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2 + cfg.Bp * cfg.N * 4,
            "select_recompute": cfg.Bp * cfg.N * 4 * 2 + cfg.Bp * E * 4,
            "topk_pairs": cfg.Bp * cfg.N * 4 + cfg.Bp * (E + K) * 4,
            "torch_concat_sdpa (context)": bytes_cache_aware(cfg, A) + bytes_scatter(cfg, A)}
    calls["_cached_idx"] = cached_idx
    return calls, algo


def torch_concat_sdpa(s, act, cached_idx):
    """Cache-aware attention the concatenating way, with PyTorch ops (context only)."""
    import torch.nn.functional as F
    Q3, K3, V3 = s.layer3
    Kc, Vc = s.cache
    B, H, N, d = Q3.shape
    ia = act.long()[:, None, :, None].expand(-1, H, -1, d)
    ic = cached_idx[:, None, :, None].expand(-1, H, -1, d)
    qa, ka, va = (torch.gather(x, 2, ia) for x in (Q3, K3, V3))
    k = torch.cat([ka, torch.gather(Kc, 2, ic)], 2)
    v = torch.cat([va, torch.gather(Vc, 2, ic)], 2)
    o = F.scaled_dot_product_attention(qa, k, v)
    Kc.scatter_(2, ia, ka)
    Vc.scatter_(2, ia, va)
    return o


def breakdown(cfg, sets, step, mar):
    """Device time of each C-ABI call of the step (graph_time: 24 back-to-back calls)."""
    A = cfg.A
    calls, algo = step_calls(cfg, step, mar)
    cached_idx = calls.pop("_cached_idx")
    calls["attn_full_select"](sets[0])
    torch.cuda.synchronize()
    mask = torch.ones(cfg.Bp, cfg.N, dtype=torch.bool, device=cached_idx.device)
    mask.scatter_(1, step.active(A).long(), False)
    cached_idx.copy_(torch.nonzero(mask)[:, 1].view(cfg.Bp, cfg.N - A))
    out = {}
    for name, fn in calls.items():
        us = graph_time(lambda i: fn(sets[i]), N_SETS, reps=24 if not name.startswith("torch_") else 6)
        out[name] = {"us": us, "bytes": algo[name], "gbs": algo[name] / (us * 1e-6) / 1e9}
    out["score (difference)"] = {"us": out["attn_full+score"]["us"] - out["attn_full"]["us"]}
    flops_full = 4 * cfg.Bp * cfg.H * cfg.N * cfg.N * cfg.d
    out["attn_full"]["tflops"] = flops_full / (out["attn_full"]["us"] * 1e-6) / 1e12
    for k in ("cache_aware", "cache_aware_gather"):
        out[k]["tflops"] = 4 * cfg.Bp * cfg.H * A * cfg.N * cfg.d / (out[k]["us"] * 1e-6) / 1e12
    return out


def sweep_active(cfg, sets, step, mar):
    """The cache-aware launch (active rows read in place, fused scatter) across active-set
    sizes: tokens per second, algorithmic GB/s and the fraction of the measured HBM copy
    bandwidth, per point."""
    hbm = load_peaks().get("hbm_gbs", 6800.0)
    dev = step.score.device
    out = {}
    for A in cfg.sweep_A or (cfg.A,):
        acts = [workloads.distinct_positions(cfg.Bp, A, 0, cfg.N, 880 + 7 * A + s).to(dev) for s in range(N_SETS)]
        oa = step.dense(3, A)
        us = graph_time(lambda i: mar.mar_attn_cache_aware_gather(*sets[i].layer3, *sets[i].cache, acts[i], O_A=oa,
                                                                  fuse_scatter=True, stale_finite=step.stale_finite),
                        N_SETS)
        b = bytes_cache_aware(cfg, A) + bytes_scatter(cfg, A)
        out[str(A)] = {"active_frac": A / cfg.N, "us": us, "tok_s": cfg.Bp * A / (us * 1e-6),
                       "gbs": b / (us * 1e-6) / 1e9, "hbm_frac": b / (us * 1e-6) / 1e9 / hbm,
                       "hbm_frac_without_scatter": bytes_cache_aware(cfg, A) / (us * 1e-6) / 1e9 / hbm}
    return out


def sweep_refresh_count(cfg, sets, step, mar):
    """The layer-2 call of a cached step (attention, score, top-K, active set) and the top-K
    launch alone, across refresh counts K."""
    out = {}
    E = cfg.G + cfg.J
    for K in K_SWEEP:
        act = step.active(E + K)
        R = step.refresh_set(K)
        sel = graph_time(lambda i: mar.mar_attn_full_select(*sets[i].layer2, sets[i].gen, sets[i].exclude, K,
                                                            step.score, O=step.O2, out_idx=R, active_out=act,
                                                            workspace=step.workspace), N_SETS)
        tk = graph_time(lambda i: mar.mar_refresh_topk(step.score, sets[i].exclude, K, out_idx=R, active_out=act),
                        N_SETS)
        out[str(K)] = {"attn_full_select_us": sel, "topk_us": tk}
    return out


def px512_leg(mar, dev):
    """The 512 px shape (128 rows, 16 heads, d = 80, N = 1088): full attention is the one
    tensor-bound step (544 flop/B); its bf16 tensor throughput against the measured cuBLAS
    peaks, and the refresh and cache-aware calls on the same shape."""
    cfg = workloads.CONFIGS["px512"]
    peaks = load_peaks()
    burst = peaks.get("bf16_tflops", 1900.0)
    sust = peaks.get("bf16_tflops_sustained", 1700.0)
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    sets = [[workloads.normal(shape, 4400 + 10 * s + i, torch.bfloat16, dev) for i in range(5)] for s in range(2)]
    O = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    flops = 4 * cfg.Bp * cfg.H * cfg.N * cfg.N * cfg.d
    us = graph_time(lambda i: mar.mar_attn_full(*sets[i][:3], O), 2, reps=8)
    tf = flops / (us * 1e-6) / 1e12
    out = {"shape": f"{cfg.Bp}x{cfg.H}x{cfg.N}x{cfg.d}", "attn_full_us": us, "attn_full_tflops": tf,
           "tensor_frac_of_burst": tf / burst, "tensor_frac_of_sustained": tf / sust,
           "attn_full_hbm_gbs": bytes_full_attention(cfg) / (us * 1e-6) / 1e9,
           "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst) and bf16_tflops_sustained"}
    us_r = graph_time(lambda i: mar.mar_attn_full_refresh(*sets[i][:3], sets[i][3], sets[i][4], O), 2, reps=8)
    out["attn_full_refresh_us"] = us_r
    out["attn_full_refresh_tflops"] = flops / (us_r * 1e-6) / 1e12
    hbm = peaks.get("hbm_gbs", 6800.0)
    for A in (1 + 1 + cfg.K, 25 + 25 + cfg.K):
        acts = [workloads.distinct_positions(cfg.Bp, A, 0, cfg.N, 4500 + A + s).to(dev) for s in range(2)]
        oa = torch.empty(cfg.Bp, cfg.H, A, cfg.d, dtype=torch.bfloat16, device=dev)
        us_a = graph_time(lambda i: mar.mar_attn_cache_aware_gather(*sets[i][:3], sets[i][3], sets[i][4], acts[i],
                                                                    O_A=oa, fuse_scatter=True, stale_finite=True),
                          2, reps=8)
        b = bytes_cache_aware(cfg, A) + bytes_scatter(cfg, A)
        out[f"cache_aware_A{A}"] = {"us": us_a, "tok_s": cfg.Bp * A / (us_a * 1e-6), "gbs": b / (us_a * 1e-6) / 1e9,
                                    "hbm_frac": b / (us_a * 1e-6) / 1e9 / hbm}
    del sets
    torch.cuda.empty_cache()
    return out


def end_to_end(args, cfg, sets, step, mar, cached_t):
    """The same cached steps through the public API with host buffers: every step copies its
    inputs (layer-2 and layer-3 Q/K/V, the schedule's positions, the conditional output)
    from pinned host memory and reads its results (O_A, the active set, the unconditional
    output) back.

    The host-to-device copies of step t + 1 run on a copy stream while step t computes (the
    input sets alternate, and a set is overwritten only after the step that last read it
    has finished); each step's compute waits for its own inputs. The timed region starts
    before the first copy and ends after the last result is back."""
    host = sets[0].host_copy()
    A = cfg.A
    nstep = min(args.steps, 24)
    res_host = torch.empty(cfg.Bp, cfg.H, A, cfg.d, dtype=torch.bfloat16).pin_memory()
    act_host = torch.empty(cfg.Bp, A, dtype=torch.int32).pin_memory()
    unc_host = torch.empty(cfg.B, cfg.n_img, cfg.latent).pin_memory()
    main = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in range(N_SETS)]    # the set's last step has finished
    ready = [torch.cuda.Event() for _ in range(N_SETS)]   # the set holds the next step's inputs
    h2d = d2h = 0
    tokens = 0

    def copy_inputs(i):
        s = sets[i % N_SETS]
        copy_stream.wait_event(done[i % N_SETS])
        with torch.cuda.stream(copy_stream):
            for dst, src in zip(s.layer2 + s.layer3, host["layer2"] + host["layer3"]):
                dst.copy_(src, non_blocking=True)
            s.gen.copy_(host["gen"], non_blocking=True)
            s.exclude.copy_(host["exclude"], non_blocking=True)
            s.cond.copy_(host["cond"], non_blocking=True)
        ready[i % N_SETS].record(copy_stream)
        return sum(x.numel() * x.element_size() for x in host["layer2"] + host["layer3"]) + \
            host["gen"].numel() * 4 + host["exclude"].numel() * 4 + host["cond"].numel() * 4

    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(main)
    copy_stream.wait_event(ev0)
    h2d += copy_inputs(0)
    for i in range(nstep):
        if i + 1 < nstep:
            h2d += copy_inputs(i + 1)
        s = sets[i % N_SETS]
        main.wait_event(ready[i % N_SETS])
        kind, oa, act = step.run(cached_t[i], s.layer2, s.layer3, s.cache, s.gen, s.exclude)
        mar.mar_cfg_residual(mar.MAR_CFG_APPLY, s.cond, s.uncond, s.residual)
        res_host.copy_(oa, non_blocking=True)
        act_host.copy_(act, non_blocking=True)
        unc_host.copy_(s.uncond, non_blocking=True)
        done[i % N_SETS].record(main)
        d2h += res_host.numel() * 2 + act_host.numel() * 4 + unc_host.numel() * 4
        tokens += cfg.Bp * A
    ev1.record(main)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d // nstep,
            "d2h_bytes_per_step": d2h // nstep, "steps": nstep,
            "overlap": "next step's host-to-device copies on a second stream during this step's compute"}


# ----------------------------------------------------------------------------- oracle arm
def host_set(cfg, s):
    ss = workloads.single_step(cfg, device="cpu", seed=cfg.seed * 100 + s)
    gen, excl = host_schedule(cfg, 7000 + 17 * s)
    return {"layer2": (ss.Q2, ss.K2, ss.V2), "layer3": (ss.Q3, ss.K3, ss.V3), "cache": (ss.Kc, ss.Vc),
            "gen": gen, "exclude": excl}


def oracle_cached_step(s_host, rows, cfg):
    """The oracle's cached decode step on whole batch rows (all heads) of one input set:
    layer-2 full attention, the head-averaged score, the top-K refresh set, the cache-aware
    attention of the active rows and the cache scatter. Returns the active-query tokens."""
    import oracle
    A = cfg.A
    Q2, K2, V2 = s_host["layer2"]
    Q3, K3, V3 = s_host["layer3"]
    Kc, Vc = s_host["cache"]
    gen, excl = s_host["gen"], s_host["exclude"]
    for b in rows:
        sl = lambda x: x[b:b + 1]
        oracle.full_attn(sl(Q2), sl(K2), sl(V2))
        score = oracle.l2_score(sl(Q2), sl(K2), gen[b:b + 1])
        R = oracle.topk(score, excl[b:b + 1], cfg.K)
        act = np.concatenate([excl[b:b + 1].numpy(), R], 1).astype(np.int32)
        qa, ka, va = (torch.from_numpy(oracle.gather(sl(x), act).view(np.int16).copy())
                      .view(torch.bfloat16).reshape(1, cfg.H, A, cfg.d) for x in (Q3, K3, V3))
        oracle.cache_aware(qa, ka, va, sl(Kc), sl(Vc), act)
        oracle.scatter(ka, act, sl(Kc))
        oracle.scatter(va, act, sl(Vc))
    return len(rows) * A


def cpu_baseline(cfg, budget_s: float = 12.0):
    """The oracle, as it stands, on a bounded sample of the same workload: whole batch rows of
    one input set, one cached step each, until the budget is spent."""
    import oracle
    oracle.build()
    s = host_set(cfg.scaled(B=2), 0)          # two images = four rows of the same shape
    t0 = time.time()
    done, n = 0, 0
    while time.time() - t0 < budget_s and n < 4096:  # the time budget ends it (about 12 s)
        done += oracle_cached_step(s, [n % 4], cfg)
        n += 1
    el = time.time() - t0
    return {"value": done / el, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{n} row-steps (one batch row, all {cfg.H} heads, one cached step each) of the same "
                      f"workload, fp64 C oracle, {el:.1f} s"}


def oracle_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (os.cpu_count() or 1)


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = config_from_args(args)
    s = host_set(cfg.scaled(B=2), 0)
    t0 = time.time()
    oracle_cached_step(s, [0], cfg)
    per_row = max(time.time() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_rows = int(min(4, max(1, budget / per_row)))
    rows = list(range(n_rows))
    for _ in range(args.warmup):
        oracle_cached_step(s, rows, cfg)
    t0 = time.time()
    done = 0
    for _ in range(args.steps):
        done += oracle_cached_step(s, rows, cfg)
    el = time.time() - t0
    v = done / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{args.config} cached decode step, fp64 oracle on {n_rows} batch row(s) "
                                   f"(all heads) per step", "name": args.config, "rows_per_step": n_rows},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": f"{n_rows} batch row(s) x {cfg.H} heads per step, {args.steps} steps"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--rows", type=int, default=0, help="batch rows B' (default: the config's)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-px512", action="store_true", help="skip the 512 px leg")
    ap.add_argument("--legs", default="all", choices=["all", "none"],
                    help="none: only the warm-up and the timed steps (e.g. for a launch list)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", default=None,
                    help="profiling aid: run REPS calls of one C-ABI call kind of the step "
                         "(e.g. attn_full, cache_aware_gather) after one layer-2 select call; no timing")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--build-key", action="store_true", help="print the source key of the attention kernel")
    args = ap.parse_args()
    if args.build_key:
        print(kernel_build_key("attn_tc5"))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_mine(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
