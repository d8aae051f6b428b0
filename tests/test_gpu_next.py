"""GPU parity of the next rows: token similarity (KV drift, LazyMAR token cache), the
token cache's recompute set, and the shared refresh set of guidance pairs.

Inputs come from the seeded generators in ``workloads``; expected values only from
``oracle``. Where a float decides an index (a threshold, a ranking) the oracle takes the
decision on the same fp32 values the GPU produced, and the fp32 values themselves are
checked against the fp64 oracle separately.
"""
import numpy as np
import pytest
import torch

import cache_aware_attention_gb300 as mar
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from cache_aware_attention_gb300 import _build
    _build.build()
    mar.load()
    oracle.build()


def _rand(shape, seed, dtype, std=1.0):
    return workloads.normal(shape, seed, dtype, DEV, std=std)


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ------------------------------------------------------------------------------ token cosine
@pytest.mark.parametrize("B,H,N,d,dtype,drift", [
    (4, 12, 320, 64, torch.bfloat16, 0.05),    # MAR-B key projections, one step of drift
    (3, 1, 50, 768, torch.bfloat16, 0.2),      # a [B, N, D] hidden state (LazyMAR token cache)
    (2, 4, 77, 32, torch.float32, 0.5),
    (2, 3, 65, 8, torch.bfloat16, 1.0),        # one 16-byte chunk per head row
    (1, 16, 1088, 80, torch.bfloat16, 0.05),   # 512 px shape
])
def test_token_cosine(B, H, N, d, dtype, drift):
    X = _rand((B, H, N, d), 700, torch.float32)
    Y = (X + drift * _rand((B, H, N, d), 701, torch.float32)).to(dtype)
    X = X.to(dtype)
    if N > 10:                                   # some tokens: zero in one or both tensors
        X[0, :, 3] = 0
        Y[0, :, 3] = 0
        X[-1, :, 7] = 0
        Y[0, :, 9] = 0
    got = mar.mar_token_cosine(X.contiguous(), Y.contiguous())
    ref = oracle.token_cosine(X, Y)
    err = np.abs(got.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= 1e-6, f"max |cos - ref| = {err.max():.3g}"


def test_token_cosine_is_deterministic():
    X = _rand((2, 12, 320, 64), 702, torch.bfloat16)
    Y = _rand((2, 12, 320, 64), 703, torch.bfloat16)
    a = mar.mar_token_cosine(X, Y)
    b = mar.mar_token_cosine(X, Y)
    assert torch.equal(a, b)


# ------------------------------------------------------------------------------ recompute set
@pytest.mark.parametrize("B,N,F,tau", [(4, 320, 4, 0.99), (3, 1088, 0, 0.95), (2, 16384, 30, 0.5),
                                        (5, 64, 64, 0.0), (2, 1, 0, 0.3)])
def test_select_recompute_bit_exact(B, N, F, tau):
    g = np.random.default_rng(N + F)
    cos = (1.0 - g.random((B, N)) ** 3 * 0.2).astype(np.float32)   # mostly close to 1
    cos[0, : min(N, 5)] = np.float32(tau)                         # equal to the threshold
    if N > 8:
        cos[-1, 6] = np.nan
    force = np.stack([g.permutation(N)[:F] for _ in range(B)]).astype(np.int32) if F else None
    c = torch.from_numpy(cos).to(DEV)
    f = torch.from_numpy(force).to(DEV) if F else None
    st = _status()
    idx, cnt = mar.mar_select_recompute(c, tau, f, status=st)
    assert mar.mar_status_read(st) == 0
    ref_idx, ref_cnt = oracle.select_recompute(cos, tau, force)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)


def test_select_recompute_on_gpu_similarities():
    # the token-cache flow: similarity of this step's features to the cached ones, then the
    # recompute set with the tokens decoded this step forced in
    B, N, D = 4, 320, 768
    cached = _rand((B, 1, N, D), 710, torch.float32)
    moved = torch.zeros(B, N, dtype=torch.bool)
    moved[:, 64:80] = True                                        # the just-decoded tokens move
    cur = cached + 0.02 * _rand((B, 1, N, D), 711, torch.float32)
    cur[:, :, 64:80] += 1.0 * _rand((B, 1, 16, D), 712, torch.float32)
    cached, cur = cached.to(torch.bfloat16), cur.to(torch.bfloat16)
    cos = mar.mar_token_cosine(cur, cached)
    force = workloads.distinct_positions(B, 4, 100, N, 713).to(DEV)
    idx, cnt = mar.mar_select_recompute(cos, 0.99, force)
    ref_idx, ref_cnt = oracle.select_recompute(cos.cpu().numpy(), 0.99, force.cpu().numpy())
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    sel = [set(r[:c].tolist()) for r, c in zip(idx.cpu().numpy(), cnt.cpu().numpy())]
    for b in range(B):
        assert set(range(64, 80)) <= sel[b]                       # every moved token recomputed
        assert set(force[b].tolist()) <= sel[b]


def test_select_recompute_reports_bad_force():
    cos = torch.ones(2, 10, device=DEV)
    st = _status()
    idx, cnt = mar.mar_select_recompute(cos, 0.5, torch.tensor([[3], [12]], dtype=torch.int32, device=DEV), status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_RANGE
    assert cnt.cpu().tolist() == [1, 0]


# ------------------------------------------------------------------------------ shared refresh set
@pytest.mark.parametrize("Bp,N,E,K,levels", [(32, 320, 8, 32, 0), (32, 320, 8, 32, 4), (4, 1088, 50, 64, 0),
                                              (3, 4096, 10, 500, 0), (2, 20, 3, 0, 0)])
def test_refresh_topk_pairs_bit_exact(Bp, N, E, K, levels):
    g = np.random.default_rng(N + E + K)
    sc = g.random((2 * Bp, N)).astype(np.float32)
    if levels:
        sc = (np.floor(sc * levels) / levels).astype(np.float32)  # many exact ties
    ex = np.stack([g.permutation(N)[:E] for _ in range(Bp)]).astype(np.int32).reshape(Bp, E)
    ex = np.concatenate([ex, ex], 0)
    score = torch.from_numpy(sc).to(DEV)
    exd = torch.from_numpy(ex).to(DEV) if E else None
    active = torch.empty(2 * Bp, E + K, dtype=torch.int32, device=DEV)
    R = mar.mar_refresh_topk_pairs(score, exd, K, active_out=active)
    if K == 0:
        return
    ref = oracle.topk_pairs(sc, ex, K)
    np.testing.assert_array_equal(R.cpu().numpy(), ref)
    np.testing.assert_array_equal(active.cpu().numpy(), np.concatenate([ex, ref], 1))


# ------------------------------------------------------------------------------ step policies
def test_decode_step_budget_and_shared_pairs():
    from cache_aware_attention_gb300.step import DecodeStep
    cfg = workloads.CONFIGS["mar_b"]
    Bp, H, N, d = 8, cfg.H, cfg.N, cfg.d                 # 4 guidance pairs
    ss = workloads.single_step(cfg.scaled(B=Bp // 2), device=DEV, seed=720)
    G, J, budget = 4, 4, 64
    pos = workloads.distinct_positions(Bp // 2, G + J, cfg.n_buf, N, 721)
    pos = torch.cat([pos, pos], 0).to(DEV)
    gen, excl = pos[:, :G].contiguous(), pos.contiguous()
    step = DecodeStep(Bp, H, N, d, 0, budget, device=DEV, max_gen=G, budget=budget, shared_pairs=True)
    Kc0, Vc0 = ss.Kc.clone(), ss.Vc.clone()
    kind, oa, act = step.run(1, (ss.Q2, ss.K2, ss.V2), (ss.Q3, ss.K3, ss.V3), (ss.Kc, ss.Vc), gen, excl)
    torch.cuda.synchronize()
    assert kind == "cached" and act.shape == (Bp, budget)
    R = act[:, G + J:].cpu().numpy()
    np.testing.assert_array_equal(R[: Bp // 2], R[Bp // 2:])          # pairs share the set
    np.testing.assert_array_equal(R, oracle.topk_pairs(step.score.cpu().numpy(), excl.cpu().numpy(),
                                                       budget - G - J))
    # the cache-aware output of a sampled row against the oracle, on the pre-step cache
    b = 5
    a = act[b:b + 1].cpu()
    qa, ka, va = (torch.stack([x[b][:, a[0].long()].cpu()]) for x in (ss.Q3, ss.K3, ss.V3))
    O_ref, _ = oracle.cache_aware(qa, ka, va, Kc0[b:b + 1].cpu(), Vc0[b:b + 1].cpu(), a)
    got = oa[b:b + 1].float().cpu().numpy()
    assert np.abs(got - O_ref).max() < 2e-2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_drift_and_stale_attention_error_over_steps(dtype):
    # MARche notes, Figure 1 / Figures 10-11 and Key Design 3: the keys drift from step to
    # step; between refreshes the cache goes stale and the cached path's error grows; a
    # refresh brings it back to zero. The per-token cosines and both attention outputs are
    # compared with the oracle; the error is formed on the host from the GPU outputs and
    # compared with the oracle's fp64 error within the bound the outputs' own tolerances
    # give: two outputs each within relative Frobenius eps of exact move the ratio by at
    # most 2 eps (1 + e) (bf16: eps = 5e-3; fp32: eps from the 1e-5 max-abs bound).
    import _parity as P
    from cache_aware_attention_gb300.policy import kv_drift, stale_and_current_outputs
    t_ = torch.bfloat16 if dtype == "bf16" else torch.float32
    B, H, N, d, A = 4, 12, 320, 64, 40
    K = _rand((B, H, N, d), 730, torch.float32)
    V = _rand((B, H, N, d), 731, torch.float32)
    Kc, Vc = K.to(t_), V.to(t_)
    errs, coss = [], []
    for t in range(1, 7):
        K = K + 0.05 * _rand((B, H, N, d), 740 + t, torch.float32)
        V = V + 0.05 * _rand((B, H, N, d), 760 + t, torch.float32)
        Kf, Vf = K.to(t_), V.to(t_)
        if t % 3 == 0:
            Kc, Vc = Kf.clone(), Vf.clone()              # full refresh
        ck, cv = kv_drift(Kc, Kf, Vc, Vf)
        for got, x, y in ((ck, Kc, Kf), (cv, Vc, Vf)):
            ref = oracle.token_cosine(x, y)
            assert np.abs(got.cpu().numpy().astype(np.float64) - ref).max() <= 1e-6
        coss.append(float(ck.double().mean()))
        idx = workloads.distinct_positions(B, A, 0, N, 780 + t).to(DEV)
        QA = _rand((B, H, A, d), 790 + t, t_)
        KA, VA = mar.mar_kv_gather([Kf, Vf], idx)
        o_stale, o_cur = stale_and_current_outputs(QA, KA, VA, (Kc, Vc), (Kf, Vf), idx)
        ref_stale, _ = oracle.cache_aware(QA, KA, VA, Kc, Vc, idx)
        ref_full, _ = oracle.full_attn(QA, Kf, Vf)
        P.assert_close(o_stale, ref_stale, dtype, f"step {t} stale")
        P.assert_close(o_cur, ref_full, dtype, f"step {t} current")
        g_s, g_c = (P.to_np(x).astype(np.float64) for x in (o_stale, o_cur))
        e_gpu = np.linalg.norm(g_s - g_c) / np.linalg.norm(g_c)
        e_ref = oracle.stale_attention_error(QA, KA, VA, Kc, Vc, Kf, Vf, idx)
        eps = P.BF16_REL_FRO if dtype == "bf16" else P.F32_MAX_ABS * np.sqrt(ref_full.size) / np.linalg.norm(ref_full)
        assert abs(e_gpu - e_ref) <= 2 * eps * (1 + e_ref), (t, e_gpu, e_ref)
        errs.append(e_ref)
    assert errs[2] < 1e-12 and errs[5] < 1e-12           # refreshed at t = 3 and 6: current cache
    assert 0 < errs[0] < errs[1] and 0 < errs[3] < errs[4]
    assert coss[2] == pytest.approx(1.0, abs=1e-6) and coss[0] > coss[1] and coss[3] > coss[4]


# ------------------------------------------------------------------------------ LazyMAR token cache
def test_token_cache_loop_against_the_oracle():
    # LazyMAR notes, Token Cache and the cache-reuse-refresh strategy, over 16 steps of one
    # shallow and one deep layer's feature cache [B, 1, N, D]: warm-up steps and every 5th
    # step after them compute every token; the shallow layer always does; the deep layer
    # otherwise recomputes the tokens whose cosine similarity to their cached feature is not
    # above tau, and the tokens decoded at the step, and reuses the rest. Per step: the
    # similarities within 1e-6 of fp64, the recompute sets equal to the oracle's decided on
    # the GPU's fp32 similarities (checked separately against fp64: a decision that differs
    # from the fp64 one must be a near-tie within 1e-6 of tau), and both caches bit-identical
    # to the oracle's.
    from cache_aware_attention_gb300.policy import TokenCache
    from oracle.loop import OracleTokenCache
    B, N, D, T, tau = 4, 320, 256, 16, 0.995
    warmup, period, shallow = 3, 5, 3
    stream = workloads.TokenDriftStream(B, N, D, seed=990, dtype=torch.bfloat16, device=DEV)
    caches = {layer: torch.zeros(B, 1, N, D, dtype=torch.bfloat16, device=DEV) for layer in (1, 4)}
    policies = {layer: TokenCache(caches[layer], tau, warmup=warmup, period=period, shallow_layers=shallow)
                for layer in (1, 4)}
    oracles = {layer: OracleTokenCache(tau, warmup, period, shallow, layer) for layer in (1, 4)}
    work = torch.empty(B, 1, N, D, dtype=torch.bfloat16, device=DEV)
    st = _status()
    recomputed, reused_steps, near = [], 0, []
    for t in range(T):
        decoded = workloads.distinct_positions(B, 4, 64, N, 1000 + t)
        feat = stream.advance(decoded)
        for layer in (1, 4):
            pol, orc = policies[layer], oracles[layer]
            if not pol.reuses(t, layer):
                pol.refresh(feat)
                assert orc.step(t, feat.cpu(), decoded.numpy())["kind"] == "full"
            else:
                idx, cnt = pol.recompute_set(feat, force=decoded.to(DEV))
                cos32 = mar.mar_token_cosine(feat, pol.cached).cpu().numpy()
                ref = orc.step(t, feat.cpu(), decoded.numpy(), decide_on=cos32)
                assert np.abs(cos32.astype(np.float64) - ref["cos64"]).max() <= 1e-6
                np.testing.assert_array_equal(cnt.cpu().numpy(), ref["count"])
                np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
                flip = (ref["cos64"] > tau) != (cos32 > np.float32(tau))
                for b, n in zip(*np.nonzero(flip)):
                    assert abs(ref["cos64"][b, n] - tau) <= 1e-6 * tau
                    near.append((t, int(b), int(n)))
                pol.update(feat, idx, work)
                recomputed.append(float(cnt.double().mean()) / N)
                reused_steps += 1
            torch.cuda.synchronize()
            assert np.array_equal(oracle._rows_as_bytes(pol.cached.cpu()), orc.cache), f"step {t} layer {layer}"
    assert mar.mar_status_read(st) == 0
    assert reused_steps == 10                         # layer 4: steps 0-2 warm up, 3, 8 and 13 refresh
    assert 0.02 < min(recomputed) and max(recomputed) < 0.9, recomputed   # the cache is really used
    if near:
        print(f"near-ties at tau: {near}")
