"""Host policies around the decode step: the LazyMAR token cache and the KV-drift report.

No arithmetic here: the similarities, selections and attention passes run in the
library's kernels; this module only decides which of them to call at which step.
"""
from __future__ import annotations

import torch

from . import mar_attn_cache_aware, mar_kv_scatter, mar_select_recompute, mar_token_cosine


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


def kv_drift(K_cache: torch.Tensor, K_fresh: torch.Tensor, V_cache: torch.Tensor, V_fresh: torch.Tensor,
             stream=None):
    """MARché notes, Figure 1 and Figures 10-11: per-token cosine similarity [B, N] between
    the cached and the freshly projected keys, and likewise for the values."""
    return (mar_token_cosine(K_cache, K_fresh, stream=stream),
            mar_token_cosine(V_cache, V_fresh, stream=stream))


def stale_attention_error(Q_A, K_A, V_A, cache, fresh, active, stream=None) -> float:
    """Relative error ||O_stale - O_fresh|| / ||O_fresh|| of the active queries' cache-aware
    attention over the stale cache against the same attention over a current cache (which,
    by the MARché Appendix A equivalence, equals full attention over the fresh K/V): what a
    refresh recovers. ``cache`` and ``fresh`` are (K, V) pairs [B, H, N, d]."""
    o_stale = mar_attn_cache_aware(Q_A, K_A, V_A, cache[0], cache[1], active, stream=stream)
    o_fresh = mar_attn_cache_aware(Q_A, K_A, V_A, fresh[0], fresh[1], active, stream=stream)
    num = (o_stale.float() - o_fresh.float()).norm()
    return float(num / o_fresh.float().norm())
