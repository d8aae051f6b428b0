"""Host logic of the step policies (CPU only): the refresh count under a fixed budget and
the LazyMAR token cache's schedule."""
import pytest
import torch

from cache_aware_attention_gb300.policy import TokenCache
from cache_aware_attention_gb300.step import DecodeStep, is_full_refresh


def test_refresh_schedule():
    assert [s for s in range(10) if is_full_refresh(s)] == [0, 3, 6, 9]


def test_refresh_count_fixed_and_budget():
    st = DecodeStep(4, 2, 320, 64, 32, 64, device="cpu")
    assert st.refresh_count(8) == 32                    # fixed K
    bud = DecodeStep(4, 2, 320, 64, 0, 64, device="cpu", budget=64)
    assert bud.refresh_count(8) == 56                   # 64 - (G + J)
    assert bud.refresh_count(64) == 0
    assert bud.refresh_count(70) == 0                   # never negative
    small = DecodeStep(2, 1, 40, 64, 0, 64, device="cpu", budget=64)
    assert small.refresh_count(10) == 30                # at most the candidates


def test_shared_pairs_need_even_rows():
    with pytest.raises(ValueError):
        DecodeStep(3, 2, 64, 64, 4, 16, device="cpu", shared_pairs=True)


def test_token_cache_schedule():
    tc = TokenCache(torch.empty(1), tau=0.95, warmup=2, period=4, shallow_layers=3)
    full = [s for s in range(12) if tc.full_compute(s)]
    assert full == [0, 1, 2, 6, 10]                     # warm-up, then every 4th step
    assert not tc.reuses(3, 2) and tc.reuses(3, 3)      # shallow layers always compute
    assert not tc.reuses(6, 5)                          # refresh step
    with pytest.raises(ValueError):
        TokenCache(torch.empty(1), 0.9, period=0)
