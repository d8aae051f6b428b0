"""Seeded synthetic inputs shaped like masked-autoregressive (MAR) image decoding.

This module produces INPUTS only: random Q/K/V tensors, random token orders,
the generating-token schedule and the classifier-free-guidance tensors. It holds
none of the attention, selection, scatter or guidance arithmetic, so that both the
CUDA path and the CPU oracle can consume the same values without sharing code.

Recipe (the pages publish no data for this path, so every workload is synthetic):

* Values: fp32 draws from N(0, 1) (torch generator seeded per tensor), rounded to
  the compute dtype once. Both sides read the rounded tensor.
* Layout: Q/K/V and the KV cache are [B', H, N, d] with B' the batch after CFG
  doubling (rows [0, B) conditional, [B, 2B) unconditional), H heads, N tokens, d
  the head dim. Buffer tokens occupy positions [0, n_buf), image tokens
  [n_buf, N).
* Token order: a seeded random permutation of the image positions; cond and
  uncond rows of one image share it.
* Generating tokens per step: MAR's cosine mask schedule (see `cosine_schedule`).
* Cache drift: a fresh K/V equals its cached value plus 0.05 * N(0, 1), applied in
  fp32 before the single rounding.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

__all__ = [
    "MarConfig", "CONFIGS", "normal", "cosine_schedule", "generation_order",
    "gen_positions", "distinct_positions", "SingleStep", "single_step",
    "DriftStream", "TokenDriftStream",
]


@dataclass(frozen=True)
class MarConfig:
    """Shape of one synthetic MAR workload.

    B images (doubled to 2B rows when ``cfg``), H heads of dim d, N = n_buf + n_img
    tokens; G generating, J just-decoded and K refresh tokens per step; ``steps``
    decoding steps for loop workloads (1 for a single layer-step)."""
    name: str
    B: int
    cfg: bool
    H: int
    d: int
    n_img: int
    n_buf: int
    G: int
    J: int
    K: int
    dtype: str          # "f32" or "bf16"
    seed: int
    steps: int = 1
    drift: float = 0.05
    latent: int = 16    # per-token latent width of the guidance tensors
    sweep_A: tuple = field(default_factory=tuple)  # active-set sizes to sweep

    @property
    def N(self) -> int:
        return self.n_buf + self.n_img

    @property
    def Bp(self) -> int:
        """Rows after classifier-free-guidance doubling."""
        return 2 * self.B if self.cfg else self.B

    @property
    def A(self) -> int:
        return self.G + self.J + self.K

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, **kw) -> "MarConfig":
        return replace(self, **kw)


CONFIGS: dict[str, MarConfig] = {
    # 8x8 grid, no buffer tokens, fp32 path.
    "tiny": MarConfig("tiny", B=1, cfg=False, H=2, d=32, n_img=64, n_buf=0,
                      G=2, J=2, K=4, dtype="f32", seed=0),
    # 16x16 grid + 64 buffer tokens, batch 32 doubled for CFG, one layer-step.
    "mar_b": MarConfig("mar_b", B=32, cfg=True, H=12, d=64, n_img=256, n_buf=64,
                       G=4, J=4, K=32, dtype="bf16", seed=1),
    # 64-step decode loop, batch 128 doubled, top-32 refresh. G/J follow the schedule.
    "mar_l_loop": MarConfig("mar_l_loop", B=128, cfg=True, H=16, d=64, n_img=256,
                            n_buf=64, G=0, J=0, K=32, dtype="bf16", seed=2, steps=64),
    # batch 256 doubled, d=80; active fraction swept 2%..50% of N=320.
    "mar_h": MarConfig("mar_h", B=256, cfg=True, H=16, d=80, n_img=256, n_buf=64,
                       G=4, J=4, K=32, dtype="bf16", seed=3,
                       sweep_A=(6, 16, 32, 64, 96, 160)),
    # 32x32 grid + 64 buffer tokens, batch 64 doubled, top-64 refresh, 64 steps.
    "px512": MarConfig("px512", B=64, cfg=True, H=16, d=80, n_img=1024, n_buf=64,
                       G=0, J=0, K=64, dtype="bf16", seed=4, steps=64),
}


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, dtype=torch.float32, device="cpu", std: float = 1.0,
           base: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 draw from N(0, std^2) (plus ``base`` if given), rounded once to ``dtype``."""
    x = torch.randn(tuple(shape), generator=_generator(seed, device),
                    dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    if base is not None:
        x.add_(base.to(device=device, dtype=torch.float32))
    return x.to(dtype)


def cosine_schedule(n_img: int, steps: int) -> list[int]:
    """Number of tokens generated at each step under MAR's cosine mask schedule.

    MAR keeps ``floor(n_img * cos(pi/2 * (t+1)/steps))`` tokens masked after step t,
    clamped so that every step decodes at least one token and the last step decodes
    all that remain. The pages fix only the 64-step default and the fixed random
    order; the cosine form is the MAR default that the workload names."""
    out, masked = [], n_img
    for t in range(steps):
        if t == steps - 1:
            after = 0
        else:
            after = math.floor(n_img * math.cos(math.pi / 2.0 * (t + 1) / steps))
            after = max(1, min(after, masked - 1))
        out.append(masked - after)
        masked = after
    return out


def generation_order(n_img: int, n_buf: int, seed: int) -> torch.Tensor:
    """Seeded random order over image positions [n_buf, n_buf + n_img) (int64)."""
    perm = torch.randperm(n_img, generator=_generator(seed, "cpu"))
    return perm + n_buf


def gen_positions(order: torch.Tensor, schedule: list[int], t: int) -> torch.Tensor:
    """Positions generated at step t: the next ``schedule[t]`` entries of ``order``."""
    start = sum(schedule[:t])
    return order[start:start + schedule[t]].clone()


def distinct_positions(rows: int, count: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """[rows, count] int32, each row ``count`` distinct positions from [lo, hi)."""
    g = _generator(seed, "cpu")
    out = torch.empty(rows, count, dtype=torch.int32)
    for r in range(rows):
        out[r] = (torch.randperm(hi - lo, generator=g)[:count] + lo).to(torch.int32)
    return out


@dataclass
class SingleStep:
    """Inputs of one cached layer-step.

    Layer 2 (full attention + score): Q2, K2, V2 [B', H, N, d].
    Layer 3 (cache-aware attention): fresh Q3, K3, V3 [B', H, N, d] and the stored
    cache Kc, Vc [B', H, N, d] with K3 = Kc + drift, V3 = Vc + drift.
    gen [B', G], just [B', J] int32 (cond/uncond rows of an image share them).
    Guidance tensors cond, uncond, residual [B, n_img, latent] fp32."""
    cfg: MarConfig
    Q2: torch.Tensor
    K2: torch.Tensor
    V2: torch.Tensor
    Q3: torch.Tensor
    K3: torch.Tensor
    V3: torch.Tensor
    Kc: torch.Tensor
    Vc: torch.Tensor
    gen: torch.Tensor
    just: torch.Tensor
    cond: torch.Tensor
    uncond: torch.Tensor
    residual: torch.Tensor


def single_step(cfg: MarConfig, device="cpu", seed: int | None = None) -> SingleStep:
    """Seeded inputs for one cached layer-step of ``cfg`` on ``device``."""
    s = cfg.seed if seed is None else seed
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    dt = cfg.torch_dtype
    base = 1000 * s
    Kc32 = normal(shape, base + 5, torch.float32, device)
    Vc32 = normal(shape, base + 6, torch.float32, device)
    ss = SingleStep(
        cfg=cfg,
        Q2=normal(shape, base + 1, dt, device),
        K2=normal(shape, base + 2, dt, device),
        V2=normal(shape, base + 3, dt, device),
        Q3=normal(shape, base + 4, dt, device),
        K3=normal(shape, base + 7, dt, device, std=cfg.drift, base=Kc32),
        V3=normal(shape, base + 8, dt, device, std=cfg.drift, base=Vc32),
        Kc=Kc32.to(dt), Vc=Vc32.to(dt),
        gen=None, just=None, cond=None, uncond=None, residual=None)
    del Kc32, Vc32
    pos = distinct_positions(cfg.B, cfg.G + cfg.J, cfg.n_buf, cfg.N, base + 9)
    if cfg.cfg:
        pos = torch.cat([pos, pos], 0)
    ss.gen = pos[:, :cfg.G].contiguous().to(device)
    ss.just = pos[:, cfg.G:].contiguous().to(device)
    gshape = (cfg.B, cfg.n_img, cfg.latent)
    ss.cond = normal(gshape, base + 10, torch.float32, device)
    ss.uncond = normal(gshape, base + 11, torch.float32, device)
    ss.residual = normal(gshape, base + 12, torch.float32, device, std=0.1)
    return ss


class DriftStream:
    """Per-step fresh tensors of a decode loop.

    Keeps fp32 "true" values X and, at each step, adds ``drift * N(0,1)`` drawn
    from the generator seeded with ``seed + step``; the step's tensor is the single
    bf16 (or fp32) rounding of X. Call ``advance()`` once per step."""

    def __init__(self, shape, seed: int, dtype, device, drift: float):
        self.shape, self.seed, self.dtype = tuple(shape), seed, dtype
        self.device, self.drift, self.step = device, drift, -1
        self.x = normal(self.shape, seed, torch.float32, device)

    def advance(self) -> torch.Tensor:
        self.step += 1
        if self.step > 0:
            noise = torch.randn(self.shape, generator=_generator(self.seed + self.step, self.device),
                                dtype=torch.float32, device=self.device)
            self.x.add_(noise, alpha=self.drift)
        return self.x.to(self.dtype)


class TokenDriftStream:
    """Per-step features [B, 1, N, D] of one layer of a token cache.

    Keeps fp32 "true" values X. Each token has its own drift scale s[b, n], drawn once
    from U[lo, hi]; at every step after the first, X[b, :, n] += s[b, n] * N(0, 1) (the
    generator seeded with ``seed + step``), and the positions passed to ``advance`` (the
    tokens decoded at that step) also jump by ``jump`` * N(0, 1). The step's tensor is
    the single rounding of X to ``dtype``. Tokens whose features move little between
    steps are the ones a token cache reuses."""

    def __init__(self, B: int, N: int, D: int, seed: int, dtype, device, lo: float = 0.005,
                 hi: float = 0.3, jump: float = 1.0):
        self.shape, self.seed, self.dtype, self.device = (B, 1, N, D), seed, dtype, device
        self.jump, self.step = jump, -1
        g = _generator(seed + 7_000_000, device)
        self.scale = lo + (hi - lo) * torch.rand(B, 1, N, 1, generator=g, device=device)
        self.x = normal(self.shape, seed, torch.float32, device)

    def advance(self, decoded: torch.Tensor | None = None) -> torch.Tensor:
        """``decoded`` [B, k] int positions that jump at this step (or None)."""
        self.step += 1
        if self.step > 0:
            g = _generator(self.seed + self.step, self.device)
            noise = torch.randn(self.shape, generator=g, dtype=torch.float32, device=self.device)
            self.x.add_(noise * self.scale)
            if decoded is not None and decoded.numel():
                jump = torch.randn(self.shape, generator=g, dtype=torch.float32, device=self.device)
                mask = torch.zeros(self.shape[0], 1, self.shape[2], 1, device=self.device)
                mask.scatter_(2, decoded.to(self.device).long()[:, None, :, None], 1.0)
                self.x.add_(jump * mask * self.jump)
        return self.x.to(self.dtype)
