"""Comparison helpers for the GPU parity tests (no method arithmetic here).

Tolerances: bf16 storage with fp32 accumulation -> max-abs 2e-2 and relative
Frobenius 5e-3; fp32 path -> max-abs 1e-5. Index and byte outputs: bit-exact.
Top-K sets: bit-exact except where the oracle's fp64 scores put a differing position
within 1e-6 (relative) of the K-th candidate score (a near-tie); those are returned so
that the test can log them.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3
F32_MAX_ABS = 1e-5
TIE_REL = 1e-6


def to_np(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().to("cpu")
        if x.dtype == torch.bfloat16:
            x = x.float()
        return x.numpy()
    return np.asarray(x)


def assert_close(got, want, dtype: str, what: str = ""):
    g = to_np(got).astype(np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - w)
    if dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{what}: max-abs {err.max():.3g} > {F32_MAX_ABS}"
    else:
        rel = np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30)
        assert err.max() <= BF16_MAX_ABS, f"{what}: max-abs {err.max():.3g} > {BF16_MAX_ABS}"
        assert rel <= BF16_REL_FRO, f"{what}: rel-Frobenius {rel:.3g} > {BF16_REL_FRO}"
    return float(err.max())


def bits(x) -> np.ndarray:
    """Raw bit patterns of a tensor (int16 for bf16, int32 for fp32/int32)."""
    x = x.detach().to("cpu").contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy()
    if x.dtype in (torch.float32, torch.int32):
        return x.view(torch.int32).numpy()
    return x.numpy()


def topk_mismatches(got: np.ndarray, want: np.ndarray, score64: np.ndarray, exclude: np.ndarray, K: int):
    """Rows where got != want. Raises if a mismatch is not a near-tie; returns the ties."""
    ties = []
    for b in range(got.shape[0]):
        g, w = set(got[b].tolist()), set(want[b].tolist())
        if g == w:
            continue
        cand = np.setdiff1d(np.arange(score64.shape[1]), exclude[b])
        sc = np.sort(score64[b, cand])[::-1]
        thr = sc[K - 1]
        for j in g ^ w:
            gap = abs(score64[b, j] - thr)
            assert gap <= TIE_REL * abs(thr), (
                f"row {b}: position {j} differs and is not a near-tie (gap {gap:.3g}, K-th {thr:.6g})")
            ties.append((b, j, gap / abs(thr)))
    return ties


# Sentinel bit patterns for the guard regions around outputs: a NaN payload no kernel
# writes (bf16, fp32) and an arbitrary word (int32).
_GUARD = {2: 0x7FC1, 4: 0x7FC0A5A5}


def guarded(shape, dtype, device="cuda", guard_bytes: int = 4096, fill=None):
    """A contiguous tensor of ``shape`` carved from a larger buffer whose ``guard_bytes``
    before and after it hold a sentinel bit pattern (the tensor starts 4096 bytes into a
    256-byte aligned allocation, so its own alignment is what a plain allocation gives).
    ``fill``: initial contents (default: the sentinel too, so that unwritten elements can
    be found). Returns (tensor, check); check(what) asserts that both guard regions still
    hold the sentinel."""
    el = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape))
    g = guard_bytes // el
    buf = torch.empty(n + 2 * g, dtype=dtype, device=device)
    raw = buf.view({2: torch.int16, 4: torch.int32}[el])
    pat = _GUARD[el]
    pat = pat - (1 << 32) if el == 4 and pat >= 1 << 31 else pat
    raw.fill_(pat)
    t = buf[g:g + n].view(shape)
    if fill is not None:
        t.copy_(fill)

    def check(what: str = ""):
        torch.cuda.synchronize()
        assert bool((raw[:g] == pat).all()), f"{what}: written before the tensor's first element"
        assert bool((raw[g + n:] == pat).all()), f"{what}: written past the tensor's last element"

    def untouched() -> torch.Tensor:
        """Elements of the tensor that still hold the sentinel (never written)."""
        return raw[g:g + n].view(shape) == pat

    check.untouched = untouched
    return t, check
