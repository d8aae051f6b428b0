"""Benchmark of the MARché decode-step hot path on the MAR-B-shaped workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

Workload: batch 32 doubled to 64 rows for classifier-free guidance, 12 heads, head
dim 64, 320 tokens (256 image + 64 buffer), bf16, 4 generating + 4 just-decoded +
top-32 refresh tokens per cached step. Inputs are seeded synthetic tensors.

One bench step is one decode step through the two layers the hot path changes:
  cached step  : layer-2 full attention + head-averaged score, top-K refresh and
                 active-set build; layer-3 cache-aware attention reading its active rows
                 in place from the fresh Q/K/V, with the KV-cache scatter in the same
                 launch; condition-cache apply (uncond = cond - r);
  refresh step : (step % 3 == 0) layer-2 and layer-3 full attention, full cache
                 overwrite, condition-cache update (r = cond - uncond).
Timed steps continue the schedule after the warm-up steps. The unit is the active
query token of the cache-aware layer: B'*A per cached step, B'*N per refresh step
(every token is recomputed), so ``value`` = those tokens over the device time.

Three independent input sets (each with its own KV cache) rotate from step to step;
one set's step touches ~250 MB and the three together ~760 MB, so no step's inputs
are left in the 129 MB L2 by the previous step.
"""
from __future__ import annotations

import argparse
import json
import math
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
CONFIG = "mar_b"
N_SETS = 3
REFRESH_PERIOD = 3
GRAPH_PERIODS = 10   # schedule periods per replayed CUDA graph in the timed region
# DRAM bytes (read + write) of one full-attention launch on this workload, from the ncu
# capture summarised in profiles/attn_tc5_mar_b.md (dram__bytes_read.sum +
# dram__bytes_write.sum); None once the kernel has changed since that capture.
FULL_ATTN_DRAM_BYTES = 94.472192e6 + 7.936e6
# the same for one cache-aware launch with the active rows read in place and the fused
# scatter (A = 40)
CACHE_AWARE_DRAM_BYTES = 70.90688e6 + 1.603584e6


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
def host_schedule(cfg, n_steps_pool: int, seed: int):
    """Generating / just-decoded positions for a pool of steps (host side).

    The single-step workload fixes G = J = 4; positions are drawn from the image
    tokens, shared between the cond and uncond rows of an image."""
    out = []
    for s in range(n_steps_pool):
        pos = workloads.distinct_positions(cfg.B, cfg.G + cfg.J, cfg.n_buf, cfg.N, seed + s)
        pos = torch.cat([pos, pos], 0) if cfg.cfg else pos
        out.append((pos[:, :cfg.G].contiguous(), pos.contiguous()))   # gen, exclude = [gen, just]
    return out


class InputSet:
    def __init__(self, cfg, s, device):
        ss = workloads.single_step(cfg, device=device, seed=cfg.seed * 100 + s)
        self.layer2 = (ss.Q2, ss.K2, ss.V2)
        self.layer3 = (ss.Q3, ss.K3, ss.V3)
        self.cache = (ss.Kc, ss.Vc)
        self.cond, self.uncond, self.residual = ss.cond, ss.uncond, ss.residual
        sched = host_schedule(cfg, 1, 7000 + 17 * s)
        self.gen, self.exclude = (x.to(device) for x in sched[0])

    def host_copy(self):
        """Pinned host copies of the per-step inputs (for the end-to-end leg)."""
        pin = lambda x: x.detach().to("cpu").pin_memory()
        return {"layer2": [pin(x) for x in self.layer2], "layer3": [pin(x) for x in self.layer3],
                "gen": pin(self.gen), "exclude": pin(self.exclude), "cond": pin(self.cond),
                "residual": pin(self.residual), "uncond": pin(self.uncond)}


def bytes_full_attention(cfg):
    return 4 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2          # Q, K, V read + O write (bf16)


def bytes_cache_aware(cfg, A):
    per_bh = 4 * (cfg.N - A) * cfg.d + 6 * A * cfg.d + 2 * A * cfg.d   # cached K/V, Q/K/V_A, O_A
    return cfg.Bp * cfg.H * per_bh + cfg.Bp * A * 4


# ----------------------------------------------------------------------------- our arm
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
    cfg = workloads.CONFIGS[CONFIG]
    A = cfg.A
    sets = [InputSet(cfg, s, dev) for s in range(N_SETS)]
    step = DecodeStep(cfg.Bp, cfg.H, cfg.N, cfg.d, cfg.K, A, device=dev, max_gen=cfg.G)
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
            print(json.dumps({"only": args.only, "reps": args.reps, "status": "ok"}))
        return
    n_cfg = cfg.B * cfg.n_img * cfg.latent
    stream = torch.cuda.current_stream()

    def one_step(t, s: InputSet):
        kind = step.run(t, s.layer2, s.layer3, s.cache, s.gen, s.exclude)[0]
        if kind == "full":
            mar.mar_cfg_residual(mar.MAR_CFG_UPDATE, s.cond, s.uncond, s.residual)
        else:
            mar.mar_cfg_residual(mar.MAR_CFG_APPLY, s.cond, s.uncond, s.residual)
        return kind

    units = lambda t: cfg.Bp * (cfg.N if is_full_refresh(t) else A)
    clocks = ClockSampler(local)
    clocks.start()

    # warm-up (eager), then one CUDA graph per (input set, step kind)
    W, K = args.warmup, args.steps
    for t in range(W):
        one_step(t, sets[t % N_SETS])
    torch.cuda.synchronize()
    graphs = {}
    side = torch.cuda.Stream()
    for si, s in enumerate(sets):
        for kind_t in (0, 1):        # step 0 -> refresh kind, step 1 -> cached kind
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                one_step(kind_t, s)
            graphs[(si, kind_t)] = g
    # one graph for 10 periods of the schedule (the input sets and the refresh pattern
    # repeat every 3 steps), starting at the phase of the first timed step, so that a
    # graph boundary comes every 30 steps instead of every step
    period = math.lcm(N_SETS, REFRESH_PERIOD) * GRAPH_PERIODS
    period_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(period_graph, stream=side):
        for t in range(W, W + period):
            one_step(t, sets[t % N_SETS])
    torch.cuda.synchronize()

    # timed region: exactly K steps, graph replay
    barrier(ws)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    ev0.record()
    tokens = 0
    t = W
    while t + period <= W + K:
        period_graph.replay()
        tokens += sum(units(u) for u in range(t, t + period))
        t += period
    while t < W + K:  # the steps past the last whole period
        graphs[(t % N_SETS, 0 if is_full_refresh(t) else 1)].replay()
        tokens += units(t)
        t += 1
    ev1.record()
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier(ws)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, ws)
    total_tokens = tokens * ws

    # per-call durations (eager, events around each C-ABI call on the launching stream)
    brk = breakdown(args, cfg, sets, step, mar, W, K, is_full_refresh)

    # end to end through the C ABI from pinned host buffers
    e2e = end_to_end(args, cfg, sets, step, mar, W, K, is_full_refresh, units, dev)
    clocks.stop()

    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    fa = brk["attn_full"]
    roof = {"bound": "hbm", "kernel": "attn_tc5_kernel<64> (full attention, N=320)",
            "achieved": fa["gbs"], "peak": hbm, "unit": "GB/s",
            "frac": fa["gbs"] / hbm if fa["gbs"] else None, "traffic": FULL_ATTN_DRAM_BYTES,
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch "
                              "(profiles/attn_tc5_mar_b.md)",
            "peak_source": "MEASURED_PEAKS.json hbm_gbs" if "hbm_gbs" in peaks else "fallback 6800 GB/s"}
    ca = brk["cache_aware_gather"]
    roof_ca = {"bound": "hbm", "kernel": "attn_tc5_kernel<64> (cache-aware attention of the active rows read "
                                         "in place, fused scatter, A=40)",
               "achieved": ca["gbs"], "peak": hbm, "unit": "GB/s", "frac": ca["gbs"] / hbm if ca["gbs"] else None,
               "traffic": CACHE_AWARE_DRAM_BYTES,
               "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch "
                                 "(profiles/attn_tc5_mar_b.md)"}
    cpu = cpu_baseline(cfg, budget_s=args.cpu_seconds) if (rank == 0 and ws == 1 and not args.no_cpu) else None
    n_launch = sum(launches_per_step(t) for t in range(W, W + K))
    line = {
        "metric": METRIC, "value": total_tokens / (ms_max / 1e3), "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "MAR-B-shaped decode step (batch 32 doubled to 64 for CFG, 12 heads, d=64, "
                               "256+64 tokens, 4 gen + 4 just-decoded + top-32 refresh, full refresh every 3 steps)",
                   "B_rows": cfg.Bp, "heads": cfg.H, "head_dim": cfg.d, "tokens": cfg.N, "active": A,
                   "refresh_period": REFRESH_PERIOD,
                   "steps_full": sum(1 for t in range(W, W + K) if is_full_refresh(t)),
                   "unit_tokens": "B'*A per cached step, B'*N per refresh step",
                   "l2": f"{N_SETS} rotating input sets (~{N_SETS * 8 * bytes_full_attention(cfg) // 4 // 2**20} MB "
                         "total, > L2), no flush", "timing": "CUDA graph replay (one graph per 30 steps = 10 periods of the schedule), "
                             "events on the stream"},
        "roofline": roof,
        "roofline_cache_aware": roof_ca,
        "breakdown": brk,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "cpu_baseline": cpu,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line))


def launches_per_step(t):
    # refresh: attn(L2) + attn with cache refresh (L3) + cfg = 3; cached: attn + score + top-K +
    # cache-aware with the gather and scatter in the launch + cfg = 5
    return 3 if t % REFRESH_PERIOD == 0 else 5


def step_calls(cfg, step, mar):
    """The C-ABI calls of the step (and of the next rows), by name, each a function of one
    input set, with the algorithmic bytes of one call."""
    A = cfg.A
    act = step.active(A)
    oa = step.dense(3, A)
    dev = step.score.device
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
        "topk": lambda s: mar.mar_refresh_topk(step.score, s.exclude, cfg.K, out_idx=step.R, active_out=act),
        "attn_full_select": lambda s: mar.mar_attn_full_select(s.layer2[0], s.layer2[1], s.layer2[2], s.gen, s.exclude,
                                                               cfg.K, step.score, O=step.O2, out_idx=step.R,
                                                               active_out=act, workspace=step.workspace),
        "gather": lambda s: mar.mar_kv_gather(list(s.layer3), act, dsts=[qa, ka, va]),
        "cache_aware": lambda s: mar.mar_attn_cache_aware(qa, ka, va, s.cache[0], s.cache[1], act, O_A=oa,
                                                          fuse_scatter=True),
        "cache_aware_gather": lambda s: mar.mar_attn_cache_aware_gather(s.layer3[0], s.layer3[1], s.layer3[2],
                                                                        s.cache[0], s.cache[1], act, O_A=oa,
                                                                        fuse_scatter=True),
        "attn_full_refresh": lambda s: mar.mar_attn_full_refresh(s.layer3[0], s.layer3[1], s.layer3[2], s.cache[0],
                                                                 s.cache[1], step.O3),
        "cfg": lambda s: mar.mar_cfg_residual(mar.MAR_CFG_APPLY, s.cond, s.uncond, s.residual),
        # next rows, outside the step: KV-drift cosine of the layer-3 cache against the fresh
        # keys, the token cache's recompute set on those similarities, the shared refresh set
        "token_cosine": lambda s: mar.mar_token_cosine(s.cache[0], s.layer3[1], out=cos_buf),
        "select_recompute": lambda s: mar.mar_select_recompute(cos_buf, 0.999, s.exclude, out_idx=sel_idx,
                                                               out_count=sel_cnt),
        "topk_pairs": lambda s: mar.mar_refresh_topk_pairs(step.score, s.exclude, cfg.K, out_idx=step.R,
                                                           active_out=act),
        # context only (not this library): the concatenating alternative of [MARché] Figure 7 --
        # gather the active rows and the cached rows, concatenate, PyTorch's fused attention,
        # then the cache update
        "torch_concat_sdpa (context)": lambda s: torch_concat_sdpa(s, act, cached_idx),
    }
    algo = {"attn_full": bytes_full_attention(cfg),
            "attn_full+score": bytes_full_attention(cfg),
            "topk": cfg.Bp * cfg.N * 4 + cfg.Bp * (cfg.G + cfg.J + cfg.K) * 4,
            "attn_full_select": bytes_full_attention(cfg),
            "gather": 2 * 3 * cfg.Bp * cfg.H * A * cfg.d * 2,
            "cache_aware": bytes_cache_aware(cfg, A) + 2 * cfg.Bp * cfg.H * A * cfg.d * 2,
            "cache_aware_gather": bytes_cache_aware(cfg, A) + 2 * cfg.Bp * cfg.H * A * cfg.d * 2,
            "attn_full_refresh": bytes_full_attention(cfg) + 2 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2,
            "cfg": 3 * cfg.B * cfg.n_img * cfg.latent * 4,
            "token_cosine": 2 * cfg.Bp * cfg.H * cfg.N * cfg.d * 2 + cfg.Bp * cfg.N * 4,
            "select_recompute": cfg.Bp * cfg.N * 4 * 2 + cfg.Bp * (cfg.G + cfg.J) * 4,
            "topk_pairs": cfg.Bp * cfg.N * 4 + cfg.Bp * (cfg.G + cfg.J + cfg.K) * 4,
            "torch_concat_sdpa (context)": bytes_cache_aware(cfg, A) + 2 * cfg.Bp * cfg.H * A * cfg.d * 2}
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


def breakdown(args, cfg, sets, step, mar, W, K, is_full_refresh, reps: int = 24):
    """Device time of each C-ABI call of the step.

    Each call kind is captured into one CUDA graph of ``reps`` back-to-back calls (the
    input sets rotating, so that inputs come from HBM, not L2), replayed after one
    warm-up replay, and timed with CUDA events on the replaying stream; the per-call
    time is the graph's time / reps (host launch overhead excluded, the short gaps
    between kernels of a graph included)."""
    A = cfg.A
    calls, algo = step_calls(cfg, step, mar)
    cached_idx = calls.pop("_cached_idx")

    def set_cached_idx():  # the complement of the current active set, per row (outside the timing)
        torch.cuda.synchronize()
        mask = torch.ones(cfg.Bp, cfg.N, dtype=torch.bool, device=cached_idx.device)
        mask.scatter_(1, step.active(A).long(), False)
        cached_idx.copy_(torch.nonzero(mask)[:, 1].view(cfg.Bp, cfg.N - A))
        torch.cuda.synchronize()
    side = torch.cuda.Stream()
    out = {}
    for name, fn in calls.items():
        if name.startswith("torch_concat_sdpa"):
            set_cached_idx()
        fn(sets[0])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for r in range(reps):
                fn(sets[r % N_SETS])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        out[name] = {"us": us, "calls": reps, "bytes": algo[name], "gbs": algo[name] / (us * 1e-6) / 1e9}
        del g
    out["score (difference)"] = {"us": out["attn_full+score"]["us"] - out["attn_full"]["us"]}
    flops_full = 4 * cfg.Bp * cfg.H * cfg.N * cfg.N * cfg.d
    out["attn_full"]["tflops"] = flops_full / (out["attn_full"]["us"] * 1e-6) / 1e12
    for k in ("cache_aware", "cache_aware_gather"):
        out[k]["tflops"] = 4 * cfg.Bp * cfg.H * A * cfg.N * cfg.d / (out[k]["us"] * 1e-6) / 1e12
    return out


def end_to_end(args, cfg, sets, step, mar, W, K, is_full_refresh, units, dev):
    """Same metric through the public API with host buffers: every step copies its inputs
    from pinned host memory and reads its result back.

    The host-to-device copies of step t + 1 run on a copy stream while step t computes
    (the input sets rotate, and a set is overwritten only after the step that last read it
    has finished); each step's compute waits for its own inputs. The timed region starts
    before the first copy and ends after the last result is back."""
    host = [s.host_copy() for s in sets]
    A = cfg.A
    nstep = min(K, 200)
    res_host = torch.empty(cfg.Bp, cfg.H, A, cfg.d, dtype=torch.bfloat16).pin_memory()
    full_host = torch.empty(cfg.Bp, cfg.H, cfg.N, cfg.d, dtype=torch.bfloat16).pin_memory()
    act_host = torch.empty(cfg.Bp, A, dtype=torch.int32).pin_memory()
    unc_host = torch.empty(cfg.B, cfg.n_img, cfg.latent).pin_memory()
    main = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in range(N_SETS)]    # the set's last step has finished
    ready = [torch.cuda.Event() for _ in range(N_SETS)]   # the set holds the next step's inputs
    h2d = d2h = 0
    tokens = 0

    def copy_inputs(t):
        i = t % N_SETS
        s, h = sets[i], host[i]
        copy_stream.wait_event(done[i])
        with torch.cuda.stream(copy_stream):
            for dst, src in zip(s.layer2 + s.layer3, h["layer2"] + h["layer3"]):
                dst.copy_(src, non_blocking=True)
            s.gen.copy_(h["gen"], non_blocking=True)
            s.exclude.copy_(h["exclude"], non_blocking=True)
            s.cond.copy_(h["cond"], non_blocking=True)
        ready[i].record(copy_stream)
        return sum(x.numel() * x.element_size() for x in h["layer2"] + h["layer3"]) + \
            h["gen"].numel() * 4 + h["exclude"].numel() * 4 + h["cond"].numel() * 4

    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(main)
    copy_stream.wait_event(ev0)
    h2d += copy_inputs(W)
    for t in range(W, W + nstep):
        if t + 1 < W + nstep:
            h2d += copy_inputs(t + 1)
        i = t % N_SETS
        s = sets[i]
        main.wait_event(ready[i])
        kind = step.run(t, s.layer2, s.layer3, s.cache, s.gen, s.exclude)
        if kind[0] == "full":
            mar.mar_cfg_residual(mar.MAR_CFG_UPDATE, s.cond, s.uncond, s.residual)
            full_host.copy_(kind[1], non_blocking=True)
            d2h_step = full_host.numel() * 2
        else:
            mar.mar_cfg_residual(mar.MAR_CFG_APPLY, s.cond, s.uncond, s.residual)
            res_host.copy_(kind[1], non_blocking=True)
            act_host.copy_(kind[2], non_blocking=True)
            unc_host.copy_(s.uncond, non_blocking=True)
            d2h_step = res_host.numel() * 2 + act_host.numel() * 4 + unc_host.numel() * 4
        done[i].record(main)
        d2h += d2h_step
        tokens += units(t)
    ev1.record(main)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d // nstep,
            "d2h_bytes_per_step": d2h // nstep, "steps": nstep,
            "overlap": "next step's host-to-device copies on a second stream during this step's compute"}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# ----------------------------------------------------------------------------- oracle arm
def oracle_pairs_step(t, s_host, pairs, cfg):
    """The oracle's decode step on a sample of (row, head) pairs of one input set.
    Returns the number of active-query tokens processed (fractional per head)."""
    import oracle
    A = cfg.A
    Q2, K2, V2 = s_host["layer2"]
    Q3, K3, V3 = s_host["layer3"]
    Kc, Vc = s_host["cache"]
    gen, excl = s_host["gen"], s_host["exclude"]
    done = 0.0
    by_row = {}
    for b, h in pairs:
        by_row.setdefault(b, []).append(h)
    for b, heads in by_row.items():
        hs = slice(min(heads), max(heads) + 1)
        sl = lambda x: x[b:b + 1, hs]
        if t % REFRESH_PERIOD == 0:
            oracle.full_attn(sl(Q2), sl(K2), sl(V2))
            oracle.full_attn(sl(Q3), sl(K3), sl(V3))
            oracle.scatter(sl(K3), np.arange(cfg.N, dtype=np.int32)[None], sl(Kc))
            done += len(heads) / cfg.H * cfg.N
        else:
            oracle.full_attn(sl(Q2), sl(K2), sl(V2))
            score = oracle.l2_score(sl(Q2), sl(K2), gen[b:b + 1])
            R = oracle.topk(score, excl[b:b + 1], cfg.K)
            act = np.concatenate([excl[b:b + 1].numpy(), R], 1).astype(np.int32)
            qa, ka, va = (torch.from_numpy(oracle.gather(sl(x), act).view(np.int16).copy())
                          .view(torch.bfloat16).reshape(1, len(heads), A, cfg.d) for x in (Q3, K3, V3))
            oracle.cache_aware(qa, ka, va, sl(Kc), sl(Vc), act)
            oracle.scatter(ka, act, sl(Kc))
            done += len(heads) / cfg.H * A
    return done


def host_set(cfg, s):
    ss = workloads.single_step(cfg, device="cpu", seed=cfg.seed * 100 + s)
    sched = host_schedule(cfg, 1, 7000 + 17 * s)
    return {"layer2": (ss.Q2, ss.K2, ss.V2), "layer3": (ss.Q3, ss.K3, ss.V3), "cache": (ss.Kc, ss.Vc),
            "gen": sched[0][0], "exclude": sched[0][1]}


def cpu_baseline(cfg, budget_s: float = 12.0):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    import oracle
    oracle.build()
    s = host_set(cfg.scaled(B=2), 0)         # two images (4 rows) of the same shape
    pairs = [(b, h) for b in range(4) for h in range(cfg.H)]
    t0 = time.time()
    done, t = 0.0, 0
    while time.time() - t0 < budget_s and t < 64:
        done += oracle_pairs_step(t, s, pairs, cfg)
        t += 1
    el = time.time() - t0
    return {"value": done / el, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{t} decode steps (schedule from step 0) of 4 rows x {cfg.H} heads of the same "
                      f"workload, fp64 C oracle, {el:.1f} s"}


def oracle_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (os.cpu_count() or 1)


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = workloads.CONFIGS[CONFIG]
    s = host_set(cfg.scaled(B=1), 0)
    Bp = s["layer2"][0].shape[0]
    all_pairs = [(b, h) for b in range(Bp) for h in range(cfg.H)]
    # size the per-step sample so the whole run stays within ~2 minutes
    t0 = time.time()
    oracle_pairs_step(1, s, all_pairs[:1], cfg)
    per_pair = max(time.time() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_pairs = int(min(len(all_pairs), max(1, budget / per_pair)))
    pairs = all_pairs[:n_pairs]
    for t in range(args.warmup):
        oracle_pairs_step(t, s, pairs, cfg)
    t0 = time.time()
    done = 0.0
    for t in range(args.warmup, args.warmup + args.steps):
        done += oracle_pairs_step(t, s, pairs, cfg)
    el = time.time() - t0
    v = done / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "MAR-B-shaped decode step, oracle on a sample of (row, head) pairs per step",
                       "pairs_per_step": n_pairs},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": f"{n_pairs} (row, head) pairs per step, {args.steps} steps"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", default=None,
                    help="profiling aid: run REPS calls of one C-ABI call kind of the step "
                         "(e.g. attn_full, cache_aware_gather) after one layer-2 select call; no timing")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
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
