"""Guard regions around every output: no entry point writes outside its tensors.

Each output (and each cache a call writes into) is carved from a larger buffer whose
4 KB before and after it hold a sentinel bit pattern; after the call the guards must be
intact, and every element the call must produce must have been written (outputs start
as the sentinel). Shapes are ragged on purpose: query tiles clipped at nq (A = 130: two
tiles of 128 rows, the second with 2), key blocks clipped at N (N = 200, 257, 333), the
tail columns of d = 80, the mma.sync (d = 128) and fp32 kernels, the index-driven
scatter and the two score forms. Values are checked elsewhere against the oracle; here a
few are spot-checked so that the guarded buffers are known to be the ones written.
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
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from cache_aware_attention_gb300 import _build
    _build.build()
    mar.load()
    oracle.build()


def _rand(shape, seed, dtype):
    return workloads.normal(shape, seed, dtype, DEV)


def _all_written(check, what):
    assert not bool(check.untouched().any()), f"{what}: elements left unwritten"


@pytest.mark.parametrize("dtype,B,H,N,d", [("bf16", 2, 3, 200, 64), ("bf16", 1, 2, 333, 80), ("bf16", 2, 2, 77, 128),
                                           ("f32", 2, 2, 130, 32), ("bf16", 1, 2, 1088, 80)])
def test_full_attention_and_refresh_stay_inside(dtype, B, H, N, d):
    t = DT[dtype]
    Q, K, V = (_rand((B, H, N, d), 1100 + i, t) for i in range(3))
    O, cO = P.guarded((B, H, N, d), t)
    lse, cL = P.guarded((B, H, N), torch.float32)
    mar.mar_attn_full(Q, K, V, O, lse_out=lse)
    cO("O"), cL("lse")
    _all_written(cO, "O"), _all_written(cL, "lse")
    Kc, cK = P.guarded((B, H, N, d), t)
    Vc, cV = P.guarded((B, H, N, d), t)
    O2, cO2 = P.guarded((B, H, N, d), t)
    mar.mar_attn_full_refresh(Q, K, V, Kc, Vc, O2)
    for c, w in ((cK, "K cache"), (cV, "V cache"), (cO2, "O (refresh)")):
        c(w)
        _all_written(c, w)
    assert torch.equal(O, O2) and np.array_equal(P.bits(Kc), P.bits(K))
    O_ref, _ = oracle.full_attn(Q[:1, :1], K[:1, :1], V[:1, :1])
    P.assert_close(O[:1, :1], O_ref, dtype, "O spot check")


@pytest.mark.parametrize("form", ["dense", "gather"])
@pytest.mark.parametrize("dtype,B,H,N,A,d", [("bf16", 3, 2, 257, 130, 64), ("bf16", 2, 3, 320, 40, 80),
                                             ("bf16", 2, 2, 200, 37, 128), ("f32", 2, 2, 130, 20, 64),
                                             ("bf16", 2, 2, 64, 64, 80)])
def test_cache_aware_stays_inside(form, dtype, B, H, N, A, d):
    t = DT[dtype]
    idx = workloads.distinct_positions(B, A, 0, N, 1200 + A).to(DEV)
    Q, K, V = (_rand((B, H, N, d), 1201 + i, t) for i in range(3))
    K0, V0 = _rand((B, H, N, d), 1205, t), _rand((B, H, N, d), 1206, t)
    Kc, cK = P.guarded((B, H, N, d), t, fill=K0)
    Vc, cV = P.guarded((B, H, N, d), t, fill=V0)
    O, cO = P.guarded((B, H, A, d), t)
    lse, cL = P.guarded((B, H, A), torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    QA, KA, VA = (torch.stack([x[b][:, idx[b].long()] for b in range(B)]).contiguous() for x in (Q, K, V))
    if form == "dense":
        mar.mar_attn_cache_aware(QA, KA, VA, Kc, Vc, idx, O_A=O, lse_out=lse, fuse_scatter=True, status=st)
    else:
        mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, O_A=O, lse_out=lse, fuse_scatter=True, status=st)
    assert mar.mar_status_read(st) == 0
    for c, w in ((cK, "K cache"), (cV, "V cache"), (cO, "O_A"), (cL, "lse")):
        c(w)
    _all_written(cO, "O_A"), _all_written(cL, "lse")
    want = K0.clone()
    for b in range(B):
        want[b][:, idx[b].long()] = KA[b]
    assert np.array_equal(P.bits(Kc), P.bits(want)), "scatter"
    O_ref, _ = oracle.cache_aware(QA[:1].cpu(), KA[:1].cpu(), VA[:1].cpu(), K0[:1].cpu(), V0[:1].cpu(), idx[:1].cpu())
    P.assert_close(O[:1], O_ref, dtype, "O_A spot check")


@pytest.mark.parametrize("B,H,N,d,G,E,K", [(3, 12, 320, 80, 4, 8, 32), (3, 12, 333, 64, 7, 14, 40),
                                           (2, 20, 130, 64, 3, 6, 10)])
@pytest.mark.parametrize("form", ["raw_rows", "separate"])
def test_score_and_selection_stay_inside(B, H, N, d, G, E, K, form):
    Q, Kt, V = (_rand((B, H, N, d), 1300 + i, torch.bfloat16) for i in range(3))
    pos = workloads.distinct_positions(B, G + E, 0, N, 1303).to(DEV)
    gen, excl = pos[:, :G].contiguous(), pos[:, G:].contiguous()
    s = mar.MarShape(B, H, N, d, mar.MAR_BF16)
    nbytes = (mar.load().mar_attn_full_workspace_bytes if form == "raw_rows"
              else mar.load().mar_attn_full_min_workspace_bytes)(s, G, 1)
    ws, cW = P.guarded((max(nbytes, 256) // 4,), torch.float32)
    score, cS = P.guarded((B, N), torch.float32)
    R, cR = P.guarded((B, K), torch.int32)
    act, cA = P.guarded((B, E + K), torch.int32)
    O, cO = P.guarded((B, H, N, d), torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mar.mar_attn_full_select(Q, Kt, V, gen, excl, K, score, O=O, out_idx=R, active_out=act,
                             workspace=ws if nbytes else None, status=st)
    assert mar.mar_status_read(st) == 0
    for c, w in ((cW, "workspace"), (cS, "score"), (cR, "refresh set"), (cA, "active set"), (cO, "O")):
        c(w)
    for c, w in ((cS, "score"), (cR, "refresh set"), (cA, "active set"), (cO, "O")):
        _all_written(c, w)
    np.testing.assert_array_equal(R.cpu().numpy(), oracle.topk(score.cpu().double().numpy(), excl.cpu().numpy(), K))


@pytest.mark.parametrize("dtype,d", [("bf16", 80), ("f32", 32), ("bf16", 768)])
def test_row_copies_stay_inside(dtype, d):
    t = DT[dtype]
    B, H, N, A = 3, 2 if d < 512 else 1, 129, 37
    idx = workloads.distinct_positions(B, A, 0, N, 1400).to(DEV)
    X = _rand((B, H, N, d), 1401, t)
    dst, cD = P.guarded((B, H, A, d), t)
    mar.mar_kv_gather([X], idx, dsts=[dst])
    cD("gather")
    _all_written(cD, "gather")
    C0 = _rand((B, H, N, d), 1402, t)
    C, cC = P.guarded((B, H, N, d), t, fill=C0)
    mar.mar_kv_scatter(dst, None, idx, C, None)
    cC("scatter")
    assert np.array_equal(P.bits(C), oracle.scatter(dst.cpu(), idx.cpu(), C0.cpu()).view(
        np.int16 if t == torch.bfloat16 else np.int32).reshape(P.bits(C).shape))


@pytest.mark.parametrize("n", [1001, 4096 * 16])
def test_condition_cache_stays_inside(n):
    cond = _rand((n,), 1500, torch.float32)
    res = _rand((n,), 1501, torch.float32)
    unc, cU = P.guarded((n,), torch.float32)
    gd, cG = P.guarded((n,), torch.float32)
    mar.mar_cfg_residual(mar.MAR_CFG_APPLY, cond, unc, res, w=3.0, guided=gd)
    res2, cR = P.guarded((n,), torch.float32)
    mar.mar_cfg_residual(mar.MAR_CFG_UPDATE, cond, unc, res2)
    for c, w in ((cU, "uncond"), (cG, "guided"), (cR, "residual")):
        c(w)
        _all_written(c, w)


def test_token_cache_calls_stay_inside():
    B, N, D = 3, 333, 256
    X, Y = _rand((B, 1, N, D), 1600, torch.bfloat16), _rand((B, 1, N, D), 1601, torch.bfloat16)
    cos, cC = P.guarded((B, N), torch.float32)
    mar.mar_token_cosine(X, Y, out=cos)
    cC("cosine")
    _all_written(cC, "cosine")
    idx, cI = P.guarded((B, N), torch.int32)
    cnt, cN = P.guarded((B,), torch.int32)
    mar.mar_select_recompute(cos, 0.0, None, out_idx=idx, out_count=cnt)
    cI("recompute set"), cN("count")
    _all_written(cI, "recompute set"), _all_written(cN, "count")


def test_noalloc_stays_inside():
    B, H, N, d, G = 4, 12, 320, 64, 4
    Q, K, V = (_rand((B, H, N, d), 1700 + i, torch.bfloat16) for i in range(3))
    gen = workloads.distinct_positions(B, G, 0, N, 1703).to(DEV)
    O, cO = P.guarded((B, H, N, d), torch.bfloat16)
    score, cS = P.guarded((B, N), torch.float32)
    mar.mar_attn_full_noalloc(Q, K, V, O, gen_idx=gen, score_out=score)
    cO("O"), cS("score")
    _all_written(cO, "O"), _all_written(cS, "score")
