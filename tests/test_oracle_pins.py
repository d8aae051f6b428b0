"""Pins for the CPU oracle (CPU only).

The oracle is the yardstick for the CUDA path, so it is itself checked against
things other than its own formulas: library routines (torch fp64 SDPA, numpy
sorting and fancy indexing), hand-derived closed forms in ``tests/golden``, the
exact equivalence the MARche paper proves (split attention over a current cache
equals full attention over all tokens), reductions to plain attention, and brute
force on tiny inputs. Each test is built so that a plausible slip in the oracle
(dropped term, wrong sign or index, transposed operand, double-counted row)
fails it.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


@pytest.fixture(scope="module")
def hand():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale)


def _positions(B, A, N, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(N, generator=g)[:A] for _ in range(B)]).to(torch.int32)


# --------------------------------------------------------------------------- full attention
@pytest.mark.parametrize("B,H,Nq,Nk,d", [(1, 1, 1, 1, 8), (2, 3, 5, 7, 16), (1, 2, 64, 64, 32),
                                         (2, 2, 40, 320, 64), (1, 1, 9, 33, 80)])
def test_full_attn_matches_torch_sdpa(oracle_lib, B, H, Nq, Nk, d):
    q, k, v = _rand((B, H, Nq, d), 1), _rand((B, H, Nk, d), 2), _rand((B, H, Nk, d), 3)
    O, L = oracle.full_attn(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double())
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)
    lse = torch.logsumexp(q.double() @ k.double().transpose(-1, -2) / math.sqrt(d), dim=-1)
    np.testing.assert_allclose(L, lse.numpy(), rtol=0, atol=1e-12)


def test_full_attn_explicit_scale_matches_sdpa(oracle_lib):
    q, k, v = _rand((1, 2, 6, 8), 4), _rand((1, 2, 9, 8), 5), _rand((1, 2, 9, 8), 6)
    O, _ = oracle.full_attn(q, k, v, scale=0.37)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double(), scale=0.37)
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)


def test_full_attn_hand_odds(oracle_lib, hand):
    c = hand["attention_odds_1_to_3"]
    i = c["inputs"]
    O, L = oracle.full_attn(np.array(i["q"]), np.array(i["k"]), np.array(i["v"]), scale=i["scale"])
    np.testing.assert_allclose(O, np.array(c["expect_o"]), rtol=c["rtol"])
    np.testing.assert_allclose(L, [math.log(x) for x in c["expect_lse_log_of"]], rtol=c["rtol"])


def test_full_attn_hand_equal_keys(oracle_lib, hand):
    c = hand["attention_equal_keys"]
    i = c["inputs"]
    O, L = oracle.full_attn(np.array(i["q"]), np.array(i["k"]), np.array(i["v"], np.float32),
                            scale=i["scale"])
    np.testing.assert_allclose(O, np.array(c["expect_o"]), rtol=c["rtol"])
    (a, n), = c["expect_lse_plus_log"]
    np.testing.assert_allclose(L, [a + math.log(n)], rtol=c["rtol"])


def test_full_attn_dominant_key(oracle_lib):
    # One key aligned with the query and 100x larger: its weight is ~1, so o ~ its V row.
    d, N = 16, 12
    q = np.zeros((1, d), np.float32); q[0, 3] = 1.0
    k = _rand((N, d), 7, 0.1).numpy(); k[5] = 0; k[5, 3] = 100.0 * math.sqrt(d)
    v = _rand((N, d), 8).numpy()
    O, _ = oracle.full_attn(q, k, v)
    np.testing.assert_allclose(O[0], v[5], atol=1e-12)


def test_full_attn_rows_are_convex_combinations(oracle_lib):
    # With V = identity columns (one-hot per key), o_i is exactly the weight row: sums to 1, >= 0.
    N, d = 10, 10
    q, k = _rand((1, 3, d), 9), _rand((1, N, d), 10)
    v = np.eye(N, d, dtype=np.float32)[None]
    O, L = oracle.full_attn(q, k, v)
    assert np.all(O >= 0)
    np.testing.assert_allclose(O.sum(-1), 1.0, atol=1e-14)
    # and the weights are exp(s - lse)
    s = (q.double() @ k.double().transpose(-1, -2)).numpy() / math.sqrt(d)
    np.testing.assert_allclose(O, np.exp(s - L[..., None]), atol=1e-14)


# --------------------------------------------------------------------------- cache-aware attention
def _gather_np(x, idx):
    # numpy fancy indexing: x [B,H,N,d], idx [B,A] -> [B,H,A,d]
    x = np.asarray(x)
    idx = np.asarray(idx, np.int64)
    return np.stack([x[b][:, idx[b], :] for b in range(x.shape[0])])


@pytest.mark.parametrize("method", ["concat", "split"])
@pytest.mark.parametrize("B,H,N,A,d", [(1, 2, 64, 8, 32), (2, 3, 40, 13, 16), (2, 2, 320, 40, 64),
                                        (1, 1, 17, 1, 8), (1, 2, 33, 32, 8)])
def test_cache_aware_equals_full_when_cache_current(oracle_lib, method, B, H, N, A, d):
    """MARche's Appendix A (via the review's 'Assumptions'): with every cached K/V current,
    the split attention equals standard full attention over all N tokens."""
    K, V = _rand((B, H, N, d), 11), _rand((B, H, N, d), 12)
    idx = _positions(B, A, N, 13)
    Q_A = _rand((B, H, A, d), 14)
    K_A, V_A = _gather_np(K.numpy(), idx), _gather_np(V.numpy(), idx)
    O, L = oracle.cache_aware(Q_A, K_A, V_A, K, V, idx, method=method)
    Of, Lf = oracle.full_attn(Q_A, K, V)
    np.testing.assert_allclose(O, Of, atol=1e-12)
    np.testing.assert_allclose(L, Lf, atol=1e-12)


@pytest.mark.parametrize("method", ["concat", "split"])
def test_cache_aware_ignores_stale_rows_of_active_positions(oracle_lib, method):
    B, H, N, A, d = 2, 2, 48, 10, 16
    K, V = _rand((B, H, N, d), 21), _rand((B, H, N, d), 22)
    idx = _positions(B, A, N, 23)
    Q_A = _rand((B, H, A, d), 24)
    K_A, V_A = _gather_np(K.numpy(), idx), _gather_np(V.numpy(), idx)
    Kst, Vst = K.clone(), V.clone()
    for b in range(B):
        Kst[b][:, idx[b].long(), :] = 50.0      # stale rows must not be read
        Vst[b][:, idx[b].long(), :] = 1.0e6
    O, _ = oracle.cache_aware(Q_A, K_A, V_A, Kst, Vst, idx, method=method)
    Of, _ = oracle.full_attn(Q_A, K, V)
    np.testing.assert_allclose(O, Of, atol=1e-12)


@pytest.mark.parametrize("method", ["concat", "split"])
def test_cache_aware_with_no_cached_tokens_is_plain_attention(oracle_lib, method):
    # A = N: every position is active, the cached set is empty.
    B, H, N, d = 2, 2, 24, 8
    idx = _positions(B, N, N, 31)
    Q_A, K_A, V_A = _rand((B, H, N, d), 32), _rand((B, H, N, d), 33), _rand((B, H, N, d), 34)
    Kc, Vc = _rand((B, H, N, d), 35), _rand((B, H, N, d), 36)
    O, L = oracle.cache_aware(Q_A, K_A, V_A, Kc, Vc, idx, method=method)
    ref = torch.nn.functional.scaled_dot_product_attention(Q_A.double(), K_A.double(), V_A.double())
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)


def test_cache_aware_split_equals_concat_on_stale_cache(oracle_lib):
    B, H, N, A, d = 3, 2, 100, 21, 32
    idx = _positions(B, A, N, 41)
    Q_A, K_A, V_A = _rand((B, H, A, d), 42), _rand((B, H, A, d), 43), _rand((B, H, A, d), 44)
    Kc, Vc = _rand((B, H, N, d), 45, 2.0), _rand((B, H, N, d), 46)
    O1, L1 = oracle.cache_aware(Q_A, K_A, V_A, Kc, Vc, idx, method="concat")
    O2, L2 = oracle.cache_aware(Q_A, K_A, V_A, Kc, Vc, idx, method="split")
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def test_cache_aware_permutation_equivariance(oracle_lib):
    B, H, N, A, d = 2, 2, 40, 9, 16
    idx = _positions(B, A, N, 51)
    Q_A, K_A, V_A = _rand((B, H, A, d), 52), _rand((B, H, A, d), 53), _rand((B, H, A, d), 54)
    Kc, Vc = _rand((B, H, N, d), 55), _rand((B, H, N, d), 56)
    O, L = oracle.cache_aware(Q_A, K_A, V_A, Kc, Vc, idx)
    perm = torch.randperm(A, generator=torch.Generator().manual_seed(57))
    Op, Lp = oracle.cache_aware(Q_A[:, :, perm], K_A[:, :, perm], V_A[:, :, perm], Kc, Vc,
                                idx[:, perm])
    np.testing.assert_allclose(Op, O[:, :, perm.numpy()], atol=1e-12)
    np.testing.assert_allclose(Lp, L[:, :, perm.numpy()], atol=1e-12)


def test_cache_aware_hand_case(oracle_lib, hand):
    c = hand["cache_aware_two_paths"]
    i = c["inputs"]
    e = math.e
    f = lambda a, b, cc, ff: (a + b * e) / (cc + ff * e)
    want = np.array([[f(*x) for x in row] for row in c["expect_o"]])
    want_lse = np.array([math.log(a + b * e) for a, b in c["expect_lse_log_of_coeffs"]])
    t = lambda x: np.array(x, np.float32)[None, None]
    for method in ("concat", "split"):
        O, L = oracle.cache_aware(t(i["q_a"]), t(i["k_a"]), t(i["v_a"]), t(i["k_cache"]),
                                  t(i["v_cache"]), np.array([i["idx"]], np.int32),
                                  scale=i["scale"], method=method)
        np.testing.assert_allclose(O[0, 0], want, rtol=c["rtol"])
        np.testing.assert_allclose(L[0, 0], want_lse, rtol=c["rtol"])


def test_cache_aware_rejects_bad_index(oracle_lib):
    q = _rand((1, 1, 2, 4), 60)
    kc = _rand((1, 1, 5, 4), 61)
    with pytest.raises(ValueError):
        oracle.cache_aware(q, q, q, kc, kc, np.array([[1, 1]], np.int32))
    with pytest.raises(ValueError):
        oracle.cache_aware(q, q, q, kc, kc, np.array([[0, 5]], np.int32))


# --------------------------------------------------------------------------- scatter / gather
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_scatter_gather_match_fancy_indexing(oracle_lib, dtype):
    B, H, N, A, d = 3, 2, 30, 7, 16
    cache = _rand((B, H, N, d), 71).to(dtype)
    src = _rand((B, H, A, d), 72).to(dtype)
    idx = _positions(B, A, N, 73)
    got = oracle.scatter(src, idx, cache)
    want = cache.clone()
    for b in range(B):
        want[b][:, idx[b].long(), :] = src[b]
    tint = torch.int16 if dtype == torch.bfloat16 else torch.int32
    want_b = want.view(tint).numpy()
    assert np.array_equal(got.view(want_b.dtype).reshape(want_b.shape), want_b)
    # untouched rows are bit-identical to the input cache
    mask = np.ones((B, N), bool)
    for b in range(B):
        mask[b, idx[b].numpy()] = False
    cb = cache.view(tint).numpy()
    g = got.view(want_b.dtype).reshape(want_b.shape)
    for b in range(B):
        assert np.array_equal(g[b][:, mask[b]], cb[b][:, mask[b]])
    # gather reads back exactly what was scattered
    back = oracle.gather(want, idx)
    assert np.array_equal(back.view(want_b.dtype).reshape(src.shape),
                          src.view(tint).numpy())


# --------------------------------------------------------------------------- layer-2 score
def test_l2_score_rows_sum_to_one(oracle_lib):
    B, H, N, d, G = 3, 4, 50, 16, 5
    Q, K = _rand((B, H, N, d), 81), _rand((B, H, N, d), 82)
    gen = _positions(B, G, N, 83)
    s = oracle.l2_score(Q, K, gen)
    assert np.all(s >= 0)
    np.testing.assert_allclose(s.sum(-1), 1.0, atol=1e-13)


def test_l2_score_single_query_is_its_softmax_row(oracle_lib):
    B, H, N, d = 2, 1, 30, 8
    Q, K = _rand((B, H, N, d), 91), _rand((B, H, N, d), 92)
    gen = torch.tensor([[7], [0]], dtype=torch.int32)
    s = oracle.l2_score(Q, K, gen)
    for b in range(B):
        row = torch.softmax(Q[b, 0, gen[b, 0]].double() @ K[b, 0].double().T / math.sqrt(d), -1)
        np.testing.assert_allclose(s[b], row.numpy(), atol=1e-14)


def test_l2_score_equals_full_attention_weights(oracle_lib):
    # Average of the full-attention weight rows (read out with one-hot V, so d = N) of the
    # generating queries.
    B, H, N, d, G = 2, 3, 20, 20, 4
    Q, K = _rand((B, H, N, d), 93), _rand((B, H, N, d), 94)
    gen = _positions(B, G, N, 95)
    eye = torch.eye(N, dtype=torch.float32).expand(B, H, N, N).contiguous()
    Q_g = torch.stack([Q[b][:, gen[b].long()] for b in range(B)])
    W, _ = oracle.full_attn(Q_g, K, eye)            # W[b,h,g,j] = softmax weight
    np.testing.assert_allclose(oracle.l2_score(Q, K, gen), W.mean(axis=(1, 2)), atol=1e-14)


def test_l2_score_head_linearity(oracle_lib):
    B, H, N, d, G = 2, 4, 25, 8, 3
    Q, K = _rand((B, H, N, d), 101), _rand((B, H, N, d), 102)
    gen = _positions(B, G, N, 103)
    full = oracle.l2_score(Q, K, gen)
    per_head = [oracle.l2_score(Q[:, h:h + 1].contiguous(), K[:, h:h + 1].contiguous(), gen)
                for h in range(H)]
    np.testing.assert_allclose(full, np.mean(per_head, axis=0), atol=1e-14)


# --------------------------------------------------------------------------- top-K
def _lexsort_topk(score, exclude, K):
    B, N = score.shape
    out = np.zeros((B, K), np.int32)
    for b in range(B):
        cand = np.setdiff1d(np.arange(N), exclude[b])
        order = np.lexsort((cand, -score[b, cand]))   # primary: -score, secondary: position
        out[b] = np.sort(cand[order[:K]])
    return out


@pytest.mark.parametrize("B,N,E,K,levels", [(4, 320, 8, 32, 0), (4, 320, 8, 32, 7), (3, 64, 4, 4, 3),
                                             (2, 1088, 50, 64, 0), (2, 1088, 50, 64, 11),
                                             (2, 10, 0, 10, 2), (1, 16, 3, 0, 0)])
def test_topk_matches_lexsort(oracle_lib, B, N, E, K, levels):
    g = np.random.default_rng(111)
    score = g.random((B, N))
    if levels:                           # quantise to force many ties
        score = np.floor(score * levels) / levels
    exclude = np.stack([g.permutation(N)[:E] for _ in range(B)]).astype(np.int32).reshape(B, E)
    got = oracle.topk(score, exclude, K)
    np.testing.assert_array_equal(got, _lexsort_topk(score, exclude, K))


def test_topk_brute_force_subsets(oracle_lib):
    # The chosen set maximises the score sum; among maximisers it takes the lowest positions.
    g = np.random.default_rng(121)
    for trial in range(60):
        N = int(g.integers(2, 11))
        E = int(g.integers(0, N - 1))
        K = int(g.integers(0, N - E + 1))
        score = g.integers(0, 4, size=(1, N)).astype(np.float64)   # integer scores: exact sums, ties
        exclude = g.permutation(N)[:E].astype(np.int32).reshape(1, E)
        cand = [j for j in range(N) if j not in set(exclude[0].tolist())]
        best = max(itertools.combinations(cand, K),
                   key=lambda S: (sum(score[0, j] for j in S), -sum(S)))
        np.testing.assert_array_equal(oracle.topk(score, exclude, K)[0], sorted(best))


def test_topk_hand_ties(oracle_lib, hand):
    c = hand["topk_ties"]
    sc = np.array([c["inputs"]["score"]])
    ex = np.array([c["inputs"]["exclude"]], np.int32)
    for k, want in c["expect"].items():
        np.testing.assert_array_equal(oracle.topk(sc, ex, int(k))[0], want)


def test_topk_rejects_too_few_candidates(oracle_lib):
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 5)), np.array([[0, 1]], np.int32), 4)


# --------------------------------------------------------------------------- condition cache
def test_cfg_hand(oracle_lib, hand):
    c = hand["cfg_condition_cache"]
    i = c["inputs"]
    u, _, gd = oracle.cfg(oracle.CFG_APPLY, np.array(i["cond"]), residual=np.array(i["residual"]),
                          w=i["w"])
    np.testing.assert_array_equal(u, c["expect_apply_uncond"])
    np.testing.assert_array_equal(gd, c["expect_apply_guided"])
    _, r, gd = oracle.cfg(oracle.CFG_UPDATE, np.array(i["cond"]), uncond=np.array(i["uncond_in"]),
                          w=i["w"])
    np.testing.assert_array_equal(r, c["expect_update_residual"])
    np.testing.assert_array_equal(gd, c["expect_update_guided"])


def test_cfg_apply_is_exact_fp32_subtraction_and_round_trips(oracle_lib):
    g = np.random.default_rng(131)
    cond = (g.standard_normal(4096) * 3).astype(np.float32)
    res = (g.standard_normal(4096) * 0.1).astype(np.float32)
    u, _, _ = oracle.cfg(oracle.CFG_APPLY, cond, residual=res)
    # fp64 difference of two fp32 values rounds to the IEEE fp32 difference (p' >= 2p+2)
    np.testing.assert_array_equal(u.astype(np.float32), cond - res)
    # update with that uncond recovers the residual up to the fp32 rounding of uncond
    _, r, _ = oracle.cfg(oracle.CFG_UPDATE, cond, uncond=u.astype(np.float32))
    np.testing.assert_allclose(r, res, atol=4e-7 * 3 * 4)
    # guidance weight 1 returns cond, weight 0 returns uncond
    _, _, g1 = oracle.cfg(oracle.CFG_APPLY, cond, residual=res, w=1.0)
    np.testing.assert_allclose(g1, cond, atol=1e-12)
    _, _, g0 = oracle.cfg(oracle.CFG_APPLY, cond, residual=res, w=0.0)
    np.testing.assert_array_equal(g0, u)


# ------------------------------------------------------------------------------ token similarity
def test_token_cosine_matches_scipy_on_the_concatenated_heads(oracle_lib):
    from scipy.spatial import distance
    B, H, N, d = 2, 3, 7, 8
    X, Y = _rand((B, H, N, d), 901).numpy(), _rand((B, H, N, d), 902).numpy()
    got = oracle.token_cosine(X, Y)
    for b in range(B):
        for n in range(N):
            x = X[b, :, n, :].astype(np.float64).reshape(-1)      # the token's H*d features
            y = Y[b, :, n, :].astype(np.float64).reshape(-1)
            assert got[b, n] == pytest.approx(1.0 - distance.cosine(x, y), abs=1e-12)


def test_token_cosine_closed_forms(oracle_lib):
    X = _rand((1, 2, 4, 16), 903).numpy()
    np.testing.assert_allclose(oracle.token_cosine(X, X), 1.0, atol=1e-12)
    np.testing.assert_allclose(oracle.token_cosine(X, -X), -1.0, atol=1e-12)
    np.testing.assert_allclose(oracle.token_cosine(X, 2.5 * X), 1.0, atol=1e-12)   # scale invariant
    # orthogonal: x in the first head only, y in the second head only
    x = np.zeros((1, 2, 1, 4), np.float32)
    y = np.zeros((1, 2, 1, 4), np.float32)
    x[0, 0, 0, :] = [1, 2, 3, 4]
    y[0, 1, 0, :] = [4, 3, 2, 1]
    assert oracle.token_cosine(x, y)[0, 0] == 0.0
    # hand-derived: x = (1, 0 | 0, 0), y = (1, 1 | 0, 0) -> 1 / sqrt(2)
    x = np.zeros((1, 2, 1, 2), np.float32)
    y = np.zeros((1, 2, 1, 2), np.float32)
    x[0, 0, 0] = [1, 0]
    y[0, 0, 0] = [1, 1]
    assert oracle.token_cosine(x, y)[0, 0] == pytest.approx(1 / math.sqrt(2), abs=1e-15)
    # a component in the second head counts: x = (1, 0 | 1, 0), y = (1, 0 | 0, 0) -> 1/sqrt(2)
    x[0, 1, 0] = [1, 0]
    y[0, 0, 0] = [1, 0]
    assert oracle.token_cosine(x, y)[0, 0] == pytest.approx(1 / math.sqrt(2), abs=1e-15)


def test_token_cosine_zero_vectors(oracle_lib):
    z = np.zeros((1, 1, 2, 4), np.float32)
    x = np.ones((1, 1, 2, 4), np.float32)
    np.testing.assert_array_equal(oracle.token_cosine(z, z), 1.0)
    np.testing.assert_array_equal(oracle.token_cosine(z, x), 0.0)
    np.testing.assert_array_equal(oracle.token_cosine(x, z), 0.0)


def test_select_recompute_threshold_edges(oracle_lib):
    cos = np.array([[0.5, 0.99, 0.9, np.nan, 0.95, -1.0],
                    [1.0, 1.0, 1.0, 1.0, 1.0, 1.0]], np.float32)
    idx, cnt = oracle.select_recompute(cos, 0.9)
    assert cnt.tolist() == [4, 0]
    assert idx[0].tolist() == [0, 2, 3, 5, -1, -1]      # equal to tau and NaN are recomputed
    assert idx[1].tolist() == [-1] * 6
    idx, cnt = oracle.select_recompute(cos, 0.9, force=np.array([[1, 4], [5, 0]], np.int32))
    assert idx[0].tolist() == [0, 1, 2, 3, 4, 5] and cnt[0] == 6
    assert idx[1].tolist() == [0, 5, -1, -1, -1, -1] and cnt[1] == 2   # ascending, whatever the force order
    with pytest.raises(ValueError):
        oracle.select_recompute(cos, 0.9, force=np.array([[7], [0]], np.int32))


def test_topk_pairs_symmetry_and_lexsort(oracle_lib):
    g = np.random.default_rng(905)
    Bp, N, E, K = 3, 40, 5, 7
    sc = g.random((2 * Bp, N)).astype(np.float32)
    sc[:, 3] = sc[:, 4]                                  # exact ties inside a pair's sum
    ex = np.stack([g.permutation(N)[:E] for _ in range(Bp)]).astype(np.int32)
    ex = np.concatenate([ex, ex], 0)
    R = oracle.topk_pairs(sc, ex, K)
    np.testing.assert_array_equal(R[:Bp], R[Bp:])
    swapped = np.concatenate([sc[Bp:], sc[:Bp]], 0)       # cond and uncond exchanged
    np.testing.assert_array_equal(oracle.topk_pairs(swapped, ex, K), R)
    for b in range(Bp):
        comb = (sc[b] + sc[b + Bp]).astype(np.float32).astype(np.float64)
        cand = np.setdiff1d(np.arange(N), ex[b])
        order = np.lexsort((cand, -comb[cand]))         # score descending, position ascending
        np.testing.assert_array_equal(R[b], np.sort(cand[order[:K]]))


# ------------------------------------------------------------------------------ stale-cache error
def test_stale_attention_error_is_zero_on_a_current_cache(oracle_lib):
    # Appendix A equivalence: a current cache makes the cached path full attention
    g = np.random.default_rng(40)
    B, H, N, A, d = 2, 3, 40, 9, 16
    K, V = g.standard_normal((B, H, N, d)), g.standard_normal((B, H, N, d))
    idx = np.stack([g.permutation(N)[:A] for _ in range(B)]).astype(np.int32)
    QA = g.standard_normal((B, H, A, d))
    KA = np.stack([K[b][:, idx[b]] for b in range(B)])
    VA = np.stack([V[b][:, idx[b]] for b in range(B)])
    assert oracle_lib.stale_attention_error(QA, KA, VA, K, V, K, V, idx) < 1e-12
    # every position active: no cached token, whatever the cache holds
    idx_all = np.stack([g.permutation(N) for _ in range(B)]).astype(np.int32)
    KA = np.stack([K[b][:, idx_all[b]] for b in range(B)])
    VA = np.stack([V[b][:, idx_all[b]] for b in range(B)])
    QA = g.standard_normal((B, H, N, d))
    junk = g.standard_normal((B, H, N, d)) * 10
    assert oracle_lib.stale_attention_error(QA, KA, VA, junk, junk, K, V, idx_all) < 1e-12


def test_stale_attention_error_grows_with_the_drift(oracle_lib):
    g = np.random.default_rng(41)
    B, H, N, A, d = 2, 4, 64, 8, 16
    Kc, Vc = g.standard_normal((B, H, N, d)), g.standard_normal((B, H, N, d))
    idx = np.stack([g.permutation(N)[:A] for _ in range(B)]).astype(np.int32)
    QA = g.standard_normal((B, H, A, d))
    nK, nV = g.standard_normal((B, H, N, d)), g.standard_normal((B, H, N, d))
    errs = []
    for drift in (0.01, 0.05, 0.2):
        K, V = Kc + drift * nK, Vc + drift * nV
        KA = np.stack([K[b][:, idx[b]] for b in range(B)])
        VA = np.stack([V[b][:, idx[b]] for b in range(B)])
        errs.append(oracle_lib.stale_attention_error(QA, KA, VA, Kc, Vc, K, V, idx))
    assert 0 < errs[0] < errs[1] < errs[2]
    # first order in the drift: the error scales about linearly at small drift
    assert errs[1] / errs[0] == pytest.approx(5.0, rel=0.1)


# ------------------------------------------------------------------------------ token-cache loop
def test_oracle_token_cache_extremes(oracle_lib):
    # LazyMAR token cache: a threshold no similarity exceeds (tau = 1) recomputes every token,
    # one every similarity exceeds except exact opposites (tau = -1) recomputes only the forced
    # tokens; warm-up and refresh steps take every token
    import torch
    from oracle.loop import OracleTokenCache
    B, N, D = 2, 12, 8
    g = np.random.default_rng(42)
    feats = [torch.from_numpy(g.standard_normal((B, 1, N, D)).astype(np.float32)) for _ in range(6)]
    force = np.array([[3], [7]], np.int32)
    every = OracleTokenCache(1.0, warmup=1, period=3, shallow_layers=2, layer=4)
    only_forced = OracleTokenCache(-1.0, warmup=1, period=3, shallow_layers=2, layer=4)
    shallow = OracleTokenCache(-1.0, warmup=1, period=3, shallow_layers=2, layer=1)
    raw = lambda x: x.numpy().view(np.uint8).reshape(B, 1, N, -1)
    for t, f in enumerate(feats):
        r1 = every.step(t, f, force)
        r2 = only_forced.step(t, f, force)
        shallow.step(t, f, force)
        assert np.array_equal(every.cache, raw(f)) and np.array_equal(shallow.cache, raw(f))
        if t in (0, 1, 4):                       # warm-up and the refresh step
            assert r1["kind"] == r2["kind"] == "full" and np.array_equal(only_forced.cache, raw(f))
        else:
            assert r2["kind"] == "reuse" and list(r2["count"]) == [1, 1]
            last = raw(feats[1] if t < 4 else feats[4])
            for b in range(B):
                for n in range(N):
                    want = raw(f)[b, 0, n] if n == force[b, 0] else None
                    if want is not None:
                        assert np.array_equal(only_forced.cache[b, 0, n], want)
            # the untouched tokens keep their bytes from the last full step or earlier forcing
            assert np.array_equal(only_forced.cache[0, 0, 0], last[0, 0, 0])
