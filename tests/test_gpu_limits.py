"""GPU parity at the size limits the C header declares, against the fp64 oracle.

Cache-aware attention takes up to 16384 tokens per row (the limit of its cached list): both
forms run there with the fused cache update, at active counts that select each Q-buffer
height (64, 96 and 128 rows) and two query tiles (A > 128); every output, the LSE and the
whole updated cache are compared. Full attention runs on rows of 16384 tokens and is
compared on sampled query rows (the oracle takes them one by one). The top-K runs at its
limit of 4096 candidates, with K up to every candidate that is not excluded, bit-exact.
"""
import numpy as np
import pytest
import torch

import _parity as P
import cache_aware_attention_gb300 as mar
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
N_MAX = 16384   # cached-list limit of the cache-aware calls
N_TOPK = 4096   # candidate limit of the top-K


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from cache_aware_attention_gb300 import _build
    _build.build()
    mar.load()
    oracle.build()


def _gather_host(x, idx):
    x = x.detach().cpu()
    idx = idx.detach().cpu().long()
    return torch.stack([x[b][:, idx[b]] for b in range(x.shape[0])])


@pytest.mark.parametrize("form", ["gather", "dense"])
@pytest.mark.parametrize("d,A", [(80, 1), (80, 90), (80, 100), (64, 70), (64, 200)])
def test_cache_aware_at_the_token_limit(form, d, A):
    B, H, N = 1, 2, N_MAX
    shape = (B, H, N, d)
    Q, K, V, K0, V0 = (workloads.normal(shape, 900 + 10 * A + i, torch.bfloat16, DEV) for i in range(5))
    idx = workloads.distinct_positions(B, A, 0, N, 950 + A).to(DEV)
    QA, KA, VA = (_gather_host(x, idx) for x in (Q, K, V))
    Kc, Vc = K0.clone(), V0.clone()
    lse = torch.empty(B, H, A, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if form == "gather":
        O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, lse_out=lse, fuse_scatter=True, status=st)
    else:
        O = mar.mar_attn_cache_aware(QA.to(DEV), KA.to(DEV), VA.to(DEV), Kc, Vc, idx, lse_out=lse,
                                     fuse_scatter=True, status=st)
    assert mar.mar_status_read(st) == 0
    O_ref, L_ref = oracle.cache_aware(QA, KA, VA, K0.cpu(), V0.cpu(), idx.cpu())
    P.assert_close(O, O_ref, "bf16", f"O_A {form} d={d} A={A}")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=2e-4, rtol=0)
    want_K = np.asarray(oracle.scatter(KA, idx.cpu(), K0.cpu())).view(np.int16).reshape(P.bits(Kc).shape)
    want_V = np.asarray(oracle.scatter(VA, idx.cpu(), V0.cpu())).view(np.int16).reshape(P.bits(Vc).shape)
    assert np.array_equal(P.bits(Kc), want_K) and np.array_equal(P.bits(Vc), want_V), "fused scatter"


@pytest.mark.parametrize("d", [64, 80])
def test_full_attention_long_rows_sampled(d):
    B, H, N = 1, 2, N_MAX
    Q, K, V = (workloads.normal((B, H, N, d), 970 + i, torch.bfloat16, DEV) for i in range(3))
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    O = mar.mar_attn_full(Q, K, V, lse_out=lse)
    torch.cuda.synchronize()
    rows = sorted({0, 1, 127, 128, N // 2 - 1, N - 129, N - 1} |
                  set(np.random.default_rng(d).choice(N, 9, replace=False).tolist()))
    O_ref, L_ref = oracle.full_attn(Q[:, :, rows].cpu(), K.cpu(), V.cpu())
    P.assert_close(O[:, :, rows], O_ref, "bf16", f"O full d={d}")
    np.testing.assert_allclose(lse[:, :, rows].cpu().numpy(), L_ref, atol=2e-4, rtol=0)


@pytest.mark.parametrize("E,K,levels", [(0, N_TOPK, 0), (16, 64, 7), (100, N_TOPK - 100, 3), (8, 1000, 0)])
def test_topk_at_the_candidate_limit(E, K, levels):
    B, N = 3, N_TOPK
    g = np.random.default_rng(E + K)
    sc = g.random((B, N)).astype(np.float32)
    if levels:
        sc = (np.floor(sc * levels) / levels).astype(np.float32)      # many exact ties
    excl = np.stack([g.permutation(N)[:E] for _ in range(B)]).astype(np.int32).reshape(B, E)
    score = torch.from_numpy(sc).to(DEV)
    ex = torch.from_numpy(excl).to(DEV) if E else None
    out = torch.empty(B, K, dtype=torch.int32, device=DEV)
    mar.mar_refresh_topk(score, ex, K, out_idx=out)
    assert np.array_equal(out.cpu().numpy(), oracle.topk(sc.astype(np.float64), excl, K))
