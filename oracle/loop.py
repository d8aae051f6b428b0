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

from . import cache_aware, full_attn, gather, l2_score, scatter, topk

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
