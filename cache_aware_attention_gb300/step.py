"""One MARché decode step over the two layers the hot path changes.

MARché notes, Overall Architecture and Key Designs 1-3: at every step the first two
layers run full attention and layer 2 yields the head-averaged relevance score of the
generating tokens; the top-K tokens by that score (excluding the generating and
just-decoded tokens) are refreshed; layers from 3 on run cache-aware attention for the
active set (generating + just-decoded + refreshing) and write the refreshed K/V back
into their cache. Key Design 3: step 0 and every step with step % 3 == 0 is a full
refresh: every layer runs full attention and its whole cache is overwritten.

``DecodeStep`` drives that sequence through the C ABI on one stream: layer 2 stands
for the always-full layers, layer 3 for the cache-aware layers. It owns the step's
scratch buffers (allocated once, for the largest active set) and holds no arithmetic:
the schedule decision is the only logic here.
"""
from __future__ import annotations

import torch

from . import (mar_attn_cache_aware, mar_attn_cache_aware_gather, mar_attn_full, mar_attn_full_refresh,
               mar_attn_full_select, mar_attn_full_workspace_bytes, mar_kv_gather, mar_refresh_topk_pairs)

REFRESH_PERIOD = 3


def is_full_refresh(step: int, period: int = REFRESH_PERIOD) -> bool:
    """Key Design 3: the initial step and every step with step mod period == 0."""
    return step % period == 0


class DecodeStep:
    """Buffers and call sequence of one decode step for a batch of B' rows.

    Shapes: fresh Q/K/V of each layer and the layer-3 cache are [B', H, N, d];
    ``exclude`` is the host schedule's [B', G+J] int32 device tensor (generating then
    just-decoded positions). ``K`` refresh tokens per row; ``a_max`` bounds G+J+K.

    ``budget``: the fixed-budget form of the refresh count (MARché Key Design 1 and the
    latency/FID trade-off of Figure 6 speak of a fixed number of active tokens per step):
    K = budget - (G + J) at each step instead of a fixed K. ``shared_pairs``: rows b and
    b + B'/2 (conditional and unconditional halves of a guidance batch) share one refresh
    set, ranked on the sum of their scores. ``fused_gather``: the cache-aware layer reads its
    active rows in place from the fresh tensors (one launch for gather, attention and cache
    update) instead of gathering them into dense blocks first. ``stale_finite``: the V caches
    passed to ``run`` hold finite values (they do once a full-refresh step has written them
    from finite fresh V, and so does any finite initial cache); the cache-aware launch then
    uses the stale rows of the active positions as loaded, their weight being exactly 0,
    instead of zeroing them first (MAR_CA_STALE_FINITE)."""

    def __init__(self, B: int, H: int, N: int, d: int, K: int, a_max: int, dtype=torch.bfloat16,
                 device="cuda", max_gen: int | None = None, budget: int | None = None,
                 shared_pairs: bool = False, fused_gather: bool = True, stale_finite: bool = False):
        if shared_pairs and B % 2:
            raise ValueError("shared_pairs needs an even number of rows")
        self.B, self.H, self.N, self.d, self.K, self.a_max = B, H, N, d, K, a_max
        self.budget, self.shared_pairs, self.fused_gather = budget, shared_pairs, fused_gather
        self.stale_finite = stale_finite
        self.device = torch.device(device)
        dev, f32, i32 = self.device, torch.float32, torch.int32
        self.score = torch.empty(B, N, dtype=f32, device=dev)
        self._R = torch.empty(B * max(K, budget or 0, 1), dtype=i32, device=dev)
        self._active = torch.empty(B * a_max, dtype=i32, device=dev)
        n_dense = 0 if fused_gather else B * H * a_max * d   # dense Q_A/K_A/V_A copies
        self._qkv = [torch.empty(n_dense, dtype=dtype, device=dev) for _ in range(3)]
        self._oa = torch.empty(B * H * a_max * d, dtype=dtype, device=dev)
        self.O2 = torch.empty(B, H, N, d, dtype=dtype, device=dev)
        self.O3 = torch.empty(B, H, N, d, dtype=dtype, device=dev)
        probe = torch.empty(1, 1, 1, d, dtype=dtype, device=dev).expand(B, H, N, d)
        ws = mar_attn_full_workspace_bytes(probe, max_gen or N, True)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def refresh_count(self, n_exclude: int) -> int:
        """K of a cached step: fixed, or budget - (G + J) (at least 0, at most the candidates)."""
        if self.budget is None:
            return self.K
        return max(0, min(self.budget - n_exclude, self.N - n_exclude))

    @property
    def R(self) -> torch.Tensor:
        return self._R[: self.B * self.K].view(self.B, self.K)

    def refresh_set(self, K: int) -> torch.Tensor:
        return self._R[: self.B * K].view(self.B, K)

    def active(self, A: int) -> torch.Tensor:
        return self._active[: self.B * A].view(self.B, A)

    def dense(self, i: int, A: int) -> torch.Tensor:
        buf = self._oa if i == 3 else self._qkv[i]
        return buf[: self.B * self.H * A * self.d].view(self.B, self.H, A, self.d)

    def run(self, step: int, layer2, layer3, cache, gen: torch.Tensor, exclude: torch.Tensor,
            stream=None, events=None):
        """Run one step. ``layer2``/``layer3`` are (Q, K, V); ``cache`` is (K_cache, V_cache).
        ``events``: optional (start, end) CUDA events recorded on the stream around the
        layer-3 call (the cache-aware launch, or the full attention with the cache refresh).

        Returns ("full", O3 [B',H,N,d]) on a full-refresh step, else
        ("cached", O_A [B',H,A,d], active [B',A])."""
        Q2, K2, V2 = layer2
        Q3, K3, V3 = layer3
        Kc, Vc = cache
        if is_full_refresh(step):
            mar_attn_full(Q2, K2, V2, self.O2, status=self.status, stream=stream)
            # layer 3: full attention and the whole-cache overwrite in one call
            _record(events, 0, stream)
            mar_attn_full_refresh(Q3, K3, V3, Kc, Vc, self.O3, status=self.status, stream=stream)
            _record(events, 1, stream)
            return ("full", self.O3)
        K = self.refresh_count(exclude.shape[1])
        A = exclude.shape[1] + K
        if A > self.a_max:
            raise ValueError(f"active set of {A} exceeds a_max = {self.a_max}")
        act = self.active(A)
        if self.shared_pairs:
            mar_attn_full(Q2, K2, V2, self.O2, gen_idx=gen, score_out=self.score, workspace=self.workspace,
                          status=self.status, stream=stream)
            mar_refresh_topk_pairs(self.score, exclude, K, out_idx=self.refresh_set(K), active_out=act,
                                   status=self.status, stream=stream)
        else:
            # layer 2: attention, score, refresh set and active set
            mar_attn_full_select(Q2, K2, V2, gen, exclude, K, self.score, O=self.O2, out_idx=self.refresh_set(K),
                                 active_out=act, workspace=self.workspace, status=self.status, stream=stream)
        return self.cached_layer(A, layer3, cache, stream=stream, events=events)

    def cached_layer(self, A: int, layer3, cache, stream=None, events=None):
        """Cache-aware attention of layer 3's active rows with the fused cache scatter, using
        the active set already in ``active(A)``: in one launch reading the rows in place, or
        as a gather into dense blocks followed by the attention."""
        Q3, K3, V3 = layer3
        Kc, Vc = cache
        act = self.active(A)
        oa = self.dense(3, A)
        if self.fused_gather:
            _record(events, 0, stream)
            mar_attn_cache_aware_gather(Q3, K3, V3, Kc, Vc, act, O_A=oa, fuse_scatter=True, status=self.status,
                                        stream=stream, stale_finite=self.stale_finite)
            _record(events, 1, stream)
            return ("cached", oa, act)
        qa, ka, va = (self.dense(i, A) for i in range(3))
        _record(events, 0, stream)
        mar_kv_gather([Q3, K3, V3], act, dsts=[qa, ka, va], status=self.status, stream=stream)
        mar_attn_cache_aware(qa, ka, va, Kc, Vc, act, O_A=oa, fuse_scatter=True, status=self.status,
                             stream=stream, stale_finite=self.stale_finite)
        _record(events, 1, stream)
        return ("cached", oa, act)


def _record(events, i: int, stream):
    if events is not None:
        events[i].record(stream if stream is not None else torch.cuda.current_stream())
