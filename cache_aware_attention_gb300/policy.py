"""Host policies around the decode step: the LazyMAR token cache and the KV-drift report.

No arithmetic here: the similarities, selections and attention passes run in the
library's kernels; this module only decides which of them to call at which step.
"""
from __future__ import annotations

import torch

from . import mar_attn_cache_aware, mar_kv_gather, mar_kv_scatter, mar_select_recompute, mar_token_cosine


class TokenCache:
    """LazyMAR token cache for one layer's features ([B, 1, N, D], or [B, H, N, d]).

    LazyMAR notes, Token Cache and the cache-reuse-refresh strategy: the first ``warmup``
    steps compute every token and fill the cache; afterwards the first
    ``shallow_layers`` layers still compute every token, while deeper layers recompute
    only the tokens whose current feature is not close to the cached one (cosine
    similarity above ``tau`` means reuse), plus the tokens forced in (those decoded at
    this step); every ``period`` steps the cache is refreshed by a full computation.
    The pages leave the threshold, the period and the warm-up open; they are parameters."""

    def __init__(self, cached: torch.Tensor, tau: float, warmup: int = 3, period: int = 5,
                 shallow_layers: int = 3):
        if period < 1 or warmup < 0:
            raise ValueError("period >= 1 and warmup >= 0")
        self.cached, self.tau = cached, float(tau)
        self.warmup, self.period, self.shallow_layers = warmup, period, shallow_layers

    def full_compute(self, step: int) -> bool:
        """Warm-up steps and refresh steps compute every token."""
        return step < self.warmup or (step - self.warmup) % self.period == 0

    def reuses(self, step: int, layer: int) -> bool:
        """Whether this layer of this step may reuse cached tokens."""
        return not self.full_compute(step) and layer >= self.shallow_layers

    def recompute_set(self, feat: torch.Tensor, force: torch.Tensor | None = None, stream=None):
        """(idx [B, N] ascending then -1, count [B]): the tokens to recompute."""
        cos = mar_token_cosine(feat, self.cached, stream=stream)
        return mar_select_recompute(cos, self.tau, force, stream=stream)

    def refresh(self, feat: torch.Tensor, stream=None):
        """A full-compute step: the cache takes every token's feature."""
        mar_kv_scatter(feat, None, None, self.cached, None, stream=stream)

    def update(self, feat: torch.Tensor, idx: torch.Tensor, work: torch.Tensor, stream=None):
        """A reuse step: the recomputed tokens' features (rows ``idx`` [B, N] of ``feat``,
        padded with -1 as ``recompute_set`` returns them) replace their cached rows.
        ``work`` is a dense buffer of the cache's shape: the rows are gathered into it and
        scattered from it (two row-copy launches; -1 slots are skipped)."""
        mar_kv_gather([feat], idx, dsts=[work], stream=stream)
        mar_kv_scatter(work, None, idx, self.cached, None, stream=stream)


def kv_drift(K_cache: torch.Tensor, K_fresh: torch.Tensor, V_cache: torch.Tensor, V_fresh: torch.Tensor,
             stream=None):
    """MARché notes, Figure 1 and Figures 10-11: per-token cosine similarity [B, N] between
    the cached and the freshly projected keys, and likewise for the values."""
    return (mar_token_cosine(K_cache, K_fresh, stream=stream),
            mar_token_cosine(V_cache, V_fresh, stream=stream))


def stale_and_current_outputs(Q_A, K_A, V_A, cache, fresh, active, stream=None):
    """The active queries' cache-aware attention over the stale cache and over a current
    one (which, by the MARché Appendix A equivalence, equals full attention over the fresh
    K/V): their difference is what a refresh recovers. ``cache`` and ``fresh`` are (K, V)
    pairs [B, H, N, d]. Returns (O_stale, O_current) [B, H, A, d]; the caller forms
    whatever error measure it reports."""
    o_stale = mar_attn_cache_aware(Q_A, K_A, V_A, cache[0], cache[1], active, stream=stream)
    o_current = mar_attn_cache_aware(Q_A, K_A, V_A, fresh[0], fresh[1], active, stream=stream)
    return o_stale, o_current
