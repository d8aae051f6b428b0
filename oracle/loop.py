"""Oracle decode loop for sampled batch rows (TEST INFRASTRUCTURE, fp64).

Follows the MARché decode step (paper notes, Overall Architecture and Key Designs 1-3)
for a few batch rows, keeping its own copy of the layer-3 KV cache:

* full-refresh step (step 0 and every step with step mod 3 == 0): layer 3 runs full
  attention over all tokens and its cache becomes the fresh K/V;
* cached step: the layer-2 relevance score of the generating tokens picks the top-K
  refreshing tokens among the tokens that are neither generating nor just decoded;
  the active set is [generating, just-decoded, refreshing]; layer 3 attends from the
  active queries over fresh active K/V and cached K/V, then the fresh active rows are
  written into the cache.

Rows are independent (top-K, cache and attention are all per row), so following a
subset of rows is exact. Each row's cache is kept as raw bytes, so a bit-exact
comparison with the GPU cache is possible after every step.
"""
from __future__ import annotations

import numpy as np

from . import cache_aware, full_attn, gather, l2_score, scatter, select_recompute, token_cosine, topk

REFRESH_EVERY = 3


class OracleRows:
    def __init__(self, rows, K: int):
        self.rows = list(rows)
        self.K = K
        self.Kc = None   # raw bytes [R, H, N, row_bytes]
        self.Vc = None

    def step(self, t: int, layer2, layer3, gen: np.ndarray, exclude: np.ndarray, override_R=None):
        """``layer2``/``layer3``: (Q, K, V) torch tensors of the sampled rows (CPU).
        ``gen`` [R, G], ``exclude`` [R, G+J] for the sampled rows.

        Returns a dict: kind, and for cached steps score, R, active, O; for full steps O.
        ``override_R`` replaces the refresh set (used only to follow a near-tie choice
        made by the other side)."""
        Q2, K2, V2 = layer2
        Q3, K3, V3 = layer3
        dtype = K3.dtype
        if t % REFRESH_EVERY == 0:
            O, _ = full_attn(Q3, K3, V3)
            self.Kc = scatter(K3, np.tile(np.arange(K3.shape[2], dtype=np.int32), (K3.shape[0], 1)),
                              K3)
            self.Vc = scatter(V3, np.tile(np.arange(V3.shape[2], dtype=np.int32), (V3.shape[0], 1)),
                              V3)
            return {"kind": "full", "O": O}
        score = l2_score(Q2, K2, gen)
        R = topk(score, exclude, self.K) if override_R is None else override_R
        active = np.concatenate([exclude, R], axis=1).astype(np.int32)
        q_a, k_a, v_a = (_from_bytes(gather(x, active), dtype) for x in (Q3, K3, V3))
        Kc, Vc = _from_bytes(self.Kc, dtype), _from_bytes(self.Vc, dtype)
        O, _ = cache_aware(q_a, k_a, v_a, Kc, Vc, active)
        self.Kc = scatter(k_a, active, self.Kc)
        self.Vc = scatter(v_a, active, self.Vc)
        return {"kind": "cached", "score": score, "R": R, "active": active, "O": O}


def _from_bytes(raw: np.ndarray, dtype):
    """Raw row bytes [..., row_bytes] -> torch tensor of ``dtype`` (bit copy)."""
    import torch
    item = torch.empty((), dtype=dtype).element_size()
    view = {2: np.int16, 4: np.int32}[item]
    arr = np.ascontiguousarray(raw).view(view)
    t = torch.from_numpy(arr.copy())
    return t.view(dtype)


class OracleTokenCache:
    """LazyMAR token cache of one layer, followed on the host (notes: Token Cache and the
    cache-reuse-refresh strategy). The first ``warmup`` steps and every ``period``-th step
    after them compute every token, and so does every layer below ``shallow_layers``;
    otherwise a token is recomputed when its feature's cosine similarity to its cached
    feature is not above ``tau``, or when it is forced (decoded this step), and keeps its
    cached feature otherwise. The cache is kept as raw bytes [B, 1, N, row_bytes].

    The decision is taken on fp32 similarities (``decide_on``: the values the other side
    computed, so that both sides decide on the same numbers); the fp64 similarities are
    returned for the accuracy check."""

    def __init__(self, tau: float, warmup: int, period: int, shallow_layers: int, layer: int):
        self.tau, self.warmup, self.period = float(tau), warmup, period
        self.shallow, self.layer = shallow_layers, layer
        self.cache = None

    def full_compute(self, step: int) -> bool:
        if self.layer < self.shallow or step < self.warmup:
            return True
        return (step - self.warmup) % self.period == 0

    def step(self, t: int, feat, force: np.ndarray, decide_on=None):
        """``feat`` [B, 1, N, D] torch tensor (CPU); ``force`` [B, F] positions. Returns a
        dict: kind; for reuse steps cos64 [B, N], idx [B, N] (-1 padded), count [B]."""
        if self.cache is None or self.full_compute(t):
            self.cache = _rows(feat).copy()
            return {"kind": "full"}
        cached = _from_bytes(self.cache, feat.dtype)
        cos64 = token_cosine(feat, cached)
        cos32 = cos64.astype(np.float32) if decide_on is None else np.asarray(decide_on, np.float32)
        idx, cnt = select_recompute(cos32, self.tau, force)
        rows = _rows(feat)
        for b in range(idx.shape[0]):
            sel = idx[b, :cnt[b]]
            self.cache[b, :, sel] = rows[b, :, sel]
        return {"kind": "reuse", "cos64": cos64, "idx": idx, "count": cnt}


def _rows(x) -> np.ndarray:
    """A torch tensor [..., D] as raw bytes [..., row_bytes] (bit copy)."""
    import torch
    x = x.detach().to("cpu").contiguous()
    view = {2: torch.int16, 4: torch.int32}[x.element_size()]
    return x.view(view).numpy().view(np.uint8).reshape(*x.shape[:-1], -1)