"""GPU parity over a seeded sweep of small shapes: cache-aware and full attention against
the fp64 oracle.

The shapes come from a fixed seed (the same list every run) and spread over the places
where the tensor-core kernel changes its tiling: the Q-buffer height switches at 64 and 96
queries, query tiles of 128 rows, ragged key blocks (N not a multiple of 64), A = 1, A = N
(no cache block) and A just below N. These shapes are small, so their fused scatter is
written by the index warp; the path where softmax warps without a live row write it needs
at least four tiles per CTA and runs in the full-size MAR-H and MAR-L tests and loops. Both head dims of the tensor-core kernel (64, 80) and both
forms of the cache-aware call (active rows dense, or read in place from the fresh
tensors) run, with and without the fused cache update; every output is compared with the
oracle (MARche notes, Key Designs 2: the two partial softmax sums merged by the running
max and sum) at the bf16 tolerance, the LSE within 2e-4, and the updated cache rows bit
for bit.
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


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        d = int(rng.choice([64, 80]))
        N = int(rng.choice([33, 64, 96, 130, 200, 257, 320, 400, 513]))
        # A spread over 1..N with the tiling switches weighted in
        A = int(rng.choice([1, 7, 40, 63, 64, 65, 95, 96, 97, 128, 129, N - 1, N]))
        A = max(1, min(A, N))
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 5))
        out.append((B, H, N, A, d, int(rng.integers(0, 1 << 30))))
    return out


CASES = _cases(24, 20261202)


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


@pytest.mark.parametrize("fuse", [0, 1])
@pytest.mark.parametrize("form", ["dense", "gather"])
@pytest.mark.parametrize("B,H,N,A,d,seed", CASES)
def test_cache_aware_sweep(B, H, N, A, d, seed, form, fuse):
    t = torch.bfloat16
    Q, K, V, K0, V0 = (workloads.normal((B, H, N, d), seed + i, t, DEV) for i in range(5))
    idx = workloads.distinct_positions(B, A, 0, N, seed + 9).to(DEV)
    QA, KA, VA = (_gather_host(x, idx) for x in (Q, K, V))
    Kc, Vc = K0.clone(), V0.clone()
    lse = torch.empty(B, H, A, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if form == "dense":
        O = mar.mar_attn_cache_aware(QA.to(DEV), KA.to(DEV), VA.to(DEV), Kc, Vc, idx, lse_out=lse,
                                     fuse_scatter=bool(fuse), status=st)
    else:
        O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, lse_out=lse, fuse_scatter=bool(fuse), status=st)
    assert mar.mar_status_read(st) == 0
    O_ref, L_ref = oracle.cache_aware(QA, KA, VA, K0.cpu(), V0.cpu(), idx.cpu())
    P.assert_close(O, O_ref, "bf16", f"O_A {form}")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=2e-4, rtol=0)
    want_K = oracle.scatter(KA, idx.cpu(), K0.cpu()) if fuse else P.bits(K0)
    want_V = oracle.scatter(VA, idx.cpu(), V0.cpu()) if fuse else P.bits(V0)
    assert np.array_equal(P.bits(Kc), np.asarray(want_K).view(np.int16).reshape(P.bits(Kc).shape))
    assert np.array_equal(P.bits(Vc), np.asarray(want_V).view(np.int16).reshape(P.bits(Vc).shape))


@pytest.mark.parametrize("B,H,N,A,d,seed", CASES[:12])
def test_full_attention_sweep(B, H, N, A, d, seed):
    Q, K, V = (workloads.normal((B, H, N, d), seed + 20 + i, torch.bfloat16, DEV) for i in range(3))
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    O = mar.mar_attn_full(Q, K, V, lse_out=lse)
    O_ref, L_ref = oracle.full_attn(Q.cpu(), K.cpu(), V.cpu())
    P.assert_close(O, O_ref, "bf16", "O full")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=2e-4, rtol=0)


@pytest.mark.parametrize("form", ["dense", "gather"])
@pytest.mark.parametrize("B,H,N,A,d,seed", CASES[::3])
def test_cache_aware_stale_finite_is_bit_identical(B, H, N, A, d, seed, form):
    # With the caller's guarantee of finite V cache rows at the active positions the kernel
    # uses those rows as loaded (their weight is exactly 0) instead of zeroing them: every
    # output and the updated cache are the same bits as without it, and match the oracle
    t = torch.bfloat16
    Q, K, V, K0, V0 = (workloads.normal((B, H, N, d), seed + 40 + i, t, DEV) for i in range(5))
    idx = workloads.distinct_positions(B, A, 0, N, seed + 49).to(DEV)
    QA, KA, VA = (_gather_host(x, idx) for x in (Q, K, V))
    res = []
    for finite in (False, True):
        Kc, Vc = K0.clone(), V0.clone()
        lse = torch.empty(B, H, A, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        if form == "dense":
            O = mar.mar_attn_cache_aware(QA.to(DEV), KA.to(DEV), VA.to(DEV), Kc, Vc, idx, lse_out=lse,
                                         fuse_scatter=True, status=st, stale_finite=finite)
        else:
            O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, lse_out=lse, fuse_scatter=True, status=st,
                                                stale_finite=finite)
        assert mar.mar_status_read(st) == 0
        res.append((P.bits(O), lse.cpu().numpy().view(np.int32), P.bits(Kc), P.bits(Vc)))
    for a, b in zip(*res):
        assert np.array_equal(a, b)
    O_ref, L_ref = oracle.cache_aware(QA, KA, VA, K0.cpu(), V0.cpu(), idx.cpu())
    P.assert_close(O, O_ref, "bf16", f"O_A {form} finite stale rows")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=2e-4, rtol=0)
