"""GPU parity: every entry point of the C-ABI library against the CPU oracle.

Inputs come from the seeded generators in ``workloads``; expected values come only
from ``oracle``. Small cases span several tiles and ragged tails; the configs'
full-size cases run the GPU on the whole batch and compare sampled batch rows.
"""
import numpy as np
import pytest
import torch

import cache_aware_attention_gb300 as mar
import oracle
import workloads
import _parity as P

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


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _rand(shape, seed, dtype, device=DEV, std=1.0):
    return workloads.normal(shape, seed, dtype, device, std=std)


def _active(B, A, N, seed, lo=0):
    return workloads.distinct_positions(B, A, lo, N, seed).to(DEV)


def _gather_host(x, idx):
    x = x.detach().cpu()
    idx = idx.detach().cpu().long()
    return torch.stack([x[b][:, idx[b]] for b in range(x.shape[0])])


DT = {"bf16": torch.bfloat16, "f32": torch.float32}


# ------------------------------------------------------------------------------ full attention
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,H,N,d", [(1, 2, 64, 32), (2, 3, 200, 64), (1, 2, 129, 80), (2, 1, 77, 128),
                                     (1, 1, 1, 64), (2, 2, 320, 64)])
def test_full_attention(dtype, B, H, N, d):
    t = DT[dtype]
    Q, K, V = (_rand((B, H, N, d), 10 + i, t) for i in range(3))
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    O = mar.mar_attn_full(Q, K, V, lse_out=lse)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.full_attn(Q, K, V)
    P.assert_close(O, O_ref, dtype, "O")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=1e-5 if dtype == "f32" else 2e-4, rtol=0)


def test_full_attention_explicit_scale():
    Q, K, V = (_rand((1, 2, 96, 64), 20 + i, torch.bfloat16) for i in range(3))
    O = mar.mar_attn_full(Q, K, V, scale=0.3)
    O_ref, _ = oracle.full_attn(Q, K, V, scale=0.3)
    P.assert_close(O, O_ref, "bf16", "O")


@pytest.mark.parametrize("name", ["mar_b", "mar_h", "px512"])
def test_full_attention_config_sampled_rows(name):
    cfg = workloads.CONFIGS[name]
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    Q, K, V = (_rand(shape, cfg.seed * 100 + i, torch.bfloat16) for i in range(3))
    O = mar.mar_attn_full(Q, K, V)
    torch.cuda.synchronize()
    rows = [0, cfg.Bp - 1] if name != "mar_b" else [0, 17, cfg.Bp - 1]
    for b in rows:
        O_ref, _ = oracle.full_attn(Q[b:b + 1], K[b:b + 1], V[b:b + 1])
        P.assert_close(O[b:b + 1], O_ref, "bf16", f"{name} row {b}")


# ------------------------------------------------------------------------------ full attention + cache refresh
@pytest.mark.parametrize("dtype,B,H,N,d", [
    ("bf16", 4, 12, 320, 64),     # MAR-B head shape, one launch
    ("bf16", 2, 16, 320, 80),     # d = 80: tail tiles stored too
    ("bf16", 3, 2, 200, 64),      # ragged last key block: the store is clipped at N
    ("bf16", 2, 3, 50, 64),       # fewer keys than one block
    ("bf16", 1, 4, 1088, 80),     # several query tiles per (b, h): only tile 0 stores
    ("bf16", 2, 2, 77, 128),      # two-launch path (mma.sync kernel + row copy)
    ("f32", 2, 2, 130, 32),       # two-launch path (fp32 kernel + row copy)
])
def test_full_attention_refresh(dtype, B, H, N, d):
    t = DT[dtype]
    Q, K, V = (_rand((B, H, N, d), 40 + i, t) for i in range(3))
    Kc = torch.full((B, H, N, d), float("nan"), dtype=t, device=DEV)
    Vc = torch.full((B, H, N, d), float("nan"), dtype=t, device=DEV)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    st = _status()
    O = mar.mar_attn_full_refresh(Q, K, V, Kc, Vc, lse_out=lse, status=st)
    torch.cuda.synchronize()
    assert mar.mar_status_read(st) == 0
    assert np.array_equal(P.bits(Kc), P.bits(K)) and np.array_equal(P.bits(Vc), P.bits(V))
    rows = range(B) if B * H * N <= 20000 else [0, B - 1]
    for b in rows:
        O_ref, L_ref = oracle.full_attn(Q[b:b + 1], K[b:b + 1], V[b:b + 1])
        P.assert_close(O[b:b + 1], O_ref, dtype, f"O row {b}")
        np.testing.assert_allclose(lse[b:b + 1].cpu().numpy(), L_ref, atol=1e-5 if dtype == "f32" else 2e-4, rtol=0)


def test_full_attention_refresh_rejects_aliasing():
    Q, K, V = (_rand((1, 2, 64, 64), 50 + i, torch.bfloat16) for i in range(3))
    with pytest.raises(mar.MarError) as e:
        mar.mar_attn_full_refresh(Q, K, V, K, torch.empty_like(V))
    assert e.value.code == -1  # MAR_ERR_ARG


# ------------------------------------------------------------------------------ cache-aware attention
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,H,N,A,d", [(1, 2, 64, 8, 32), (2, 3, 300, 70, 64), (2, 2, 320, 40, 80),
                                        (1, 2, 100, 100, 64), (2, 2, 50, 1, 128), (1, 1, 1088, 114, 80),
                                        (3, 2, 257, 130, 64)])
def test_cache_aware_small(dtype, B, H, N, A, d):
    t = DT[dtype]
    idx = _active(B, A, N, 30 + A)
    Q_A, K_A, V_A = (_rand((B, H, A, d), 31 + i, t) for i in range(3))
    Kc, Vc = _rand((B, H, N, d), 35, t), _rand((B, H, N, d), 36, t)
    lse = torch.empty(B, H, A, dtype=torch.float32, device=DEV)
    st = _status()
    O = mar.mar_attn_cache_aware(Q_A, K_A, V_A, Kc, Vc, idx, lse_out=lse, status=st)
    assert mar.mar_status_read(st) == 0
    O_ref, L_ref = oracle.cache_aware(Q_A, K_A, V_A, Kc, Vc, idx)
    P.assert_close(O, O_ref, dtype, "O_A")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=1e-5 if dtype == "f32" else 2e-4, rtol=0)


def test_cache_aware_tiny_config_fp32():
    cfg = workloads.CONFIGS["tiny"]
    ss = workloads.single_step(cfg, device="cpu")
    idx = workloads.distinct_positions(1, cfg.A, 0, cfg.N, 77)
    QA, KA, VA = _gather_host(ss.Q3, idx), _gather_host(ss.K3, idx), _gather_host(ss.V3, idx)
    d = lambda x: x.to(DEV).contiguous()
    O = mar.mar_attn_cache_aware(d(QA), d(KA), d(VA), d(ss.Kc), d(ss.Vc), d(idx))
    O_ref, _ = oracle.cache_aware(QA, KA, VA, ss.Kc, ss.Vc, idx)
    P.assert_close(O, O_ref, "f32", "tiny O_A")


def test_cache_aware_equals_full_attention_when_cache_current():
    # The Appendix A equivalence, on the GPU path: current cache -> full attention result.
    B, H, N, A, d = 2, 4, 320, 40, 64
    K, V = _rand((B, H, N, d), 41, torch.bfloat16), _rand((B, H, N, d), 42, torch.bfloat16)
    idx = _active(B, A, N, 43)
    Q_A = _rand((B, H, A, d), 44, torch.bfloat16)
    K_A, V_A = (_gather_host(x, idx).to(DEV).contiguous() for x in (K, V))   # host gathers
    O = mar.mar_attn_cache_aware(Q_A, K_A, V_A, K, V, idx)
    O_ref, _ = oracle.full_attn(Q_A, K, V)
    P.assert_close(O, O_ref, "bf16", "O_A vs full")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cache_aware_fused_scatter_is_bit_exact(dtype):
    t = DT[dtype]
    B, H, N, A, d = 3, 2, 200, 37, 64
    idx = _active(B, A, N, 51)
    Q_A, K_A, V_A = (_rand((B, H, A, d), 52 + i, t) for i in range(3))
    Kc, Vc = _rand((B, H, N, d), 55, t), _rand((B, H, N, d), 56, t)
    Kc0, Vc0 = Kc.clone(), Vc.clone()
    O = mar.mar_attn_cache_aware(Q_A, K_A, V_A, Kc, Vc, idx, fuse_scatter=True)
    torch.cuda.synchronize()
    O_ref, _ = oracle.cache_aware(Q_A, K_A, V_A, Kc0, Vc0, idx)   # reads the pre-scatter cache
    P.assert_close(O, O_ref, dtype, "O_A")
    assert np.array_equal(oracle._rows_as_bytes(Kc.cpu()), oracle.scatter(K_A.cpu(), idx.cpu(), Kc0.cpu()))
    assert np.array_equal(oracle._rows_as_bytes(Vc.cpu()), oracle.scatter(V_A.cpu(), idx.cpu(), Vc0.cpu()))


def test_cache_aware_mar_b_full_size():
    cfg = workloads.CONFIGS["mar_b"]
    ss = workloads.single_step(cfg, device=DEV)
    idx = torch.cat([ss.gen, ss.just, _active(cfg.Bp, cfg.K, cfg.N, 61)], 1)
    # refresh positions drawn apart from gen/just: rebuild rows that collide
    idx = _distinct_rows(idx, cfg.N, 62)
    QA, KA, VA = (_gather_host(x, idx) for x in (ss.Q3, ss.K3, ss.V3))   # host gathers
    d_ = lambda x: x.to(DEV).contiguous()
    st = _status()
    O = mar.mar_attn_cache_aware(d_(QA), d_(KA), d_(VA), ss.Kc, ss.Vc, idx, status=st)
    assert mar.mar_status_read(st) == 0
    O_ref, _ = oracle.cache_aware(QA, KA, VA, ss.Kc, ss.Vc, idx)
    P.assert_close(O, O_ref, "bf16", "MAR-B O_A")


def _distinct_rows(idx, N, seed):
    """Replace repeated positions within a row by unused ones (keeps the first occurrence)."""
    g = np.random.default_rng(seed)
    a = idx.cpu().numpy().copy()
    for b in range(a.shape[0]):
        seen, free = set(), [p for p in g.permutation(N) if p not in set(a[b].tolist())]
        for i in range(a.shape[1]):
            if a[b, i] in seen:
                a[b, i] = free.pop()
            seen.add(a[b, i])
    return torch.from_numpy(a).to(DEV)


@pytest.mark.parametrize("A", [6, 16, 32, 64, 96, 160])
def test_cache_aware_mar_h_sweep_sampled_rows(A):
    cfg = workloads.CONFIGS["mar_h"]
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    Kc, Vc = _rand(shape, 301, torch.bfloat16), _rand(shape, 302, torch.bfloat16)
    ashape = (cfg.Bp, cfg.H, A, cfg.d)
    Q_A, K_A, V_A = (_rand(ashape, 303 + i, torch.bfloat16) for i in range(3))
    idx = _active(cfg.Bp, A, cfg.N, 310 + A)
    O = mar.mar_attn_cache_aware(Q_A, K_A, V_A, Kc, Vc, idx)
    torch.cuda.synchronize()
    for b in (0, cfg.Bp // 2, cfg.Bp - 1):
        sl = slice(b, b + 1)
        O_ref, _ = oracle.cache_aware(Q_A[sl], K_A[sl], V_A[sl], Kc[sl], Vc[sl], idx[sl])
        P.assert_close(O[sl], O_ref, "bf16", f"MAR-H A={A} row {b}")


def test_cache_aware_px512_sampled_rows():
    cfg = workloads.CONFIGS["px512"]
    A = 25 + 25 + cfg.K
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    Kc, Vc = _rand(shape, 401, torch.bfloat16), _rand(shape, 402, torch.bfloat16)
    Q_A, K_A, V_A = (_rand((cfg.Bp, cfg.H, A, cfg.d), 403 + i, torch.bfloat16) for i in range(3))
    idx = _active(cfg.Bp, A, cfg.N, 410)
    O = mar.mar_attn_cache_aware(Q_A, K_A, V_A, Kc, Vc, idx)
    torch.cuda.synchronize()
    for b in (3, cfg.Bp - 1):
        sl = slice(b, b + 1)
        O_ref, _ = oracle.cache_aware(Q_A[sl], K_A[sl], V_A[sl], Kc[sl], Vc[sl], idx[sl])
        P.assert_close(O[sl], O_ref, "bf16", f"512px row {b}")


@pytest.mark.parametrize("d", [64, 80])
def test_cache_aware_stale_rows_never_contribute(d):
    # Cache rows at active positions are stale; whatever they hold (here NaN and huge
    # values) must not reach the output.
    B, H, N, A = 3, 4, 320, 40
    idx = _active(B, A, N, 81 + d)
    Q_A, K_A, V_A = (_rand((B, H, A, d), 82 + i, torch.bfloat16) for i in range(3))
    Kc, Vc = _rand((B, H, N, d), 86, torch.bfloat16), _rand((B, H, N, d), 87, torch.bfloat16)
    Kp, Vp = Kc.clone(), Vc.clone()
    for b in range(B):
        Kp[b][:, idx[b].long()] = float("nan")
        Vp[b][:, idx[b].long()] = float("nan")
        Kp[b][:, idx[b][:5].long()] = 3.0e4
    O = mar.mar_attn_cache_aware(Q_A, K_A, V_A, Kp, Vp, idx)
    O_ref, _ = oracle.cache_aware(Q_A, K_A, V_A, Kc, Vc, idx)
    P.assert_close(O, O_ref, "bf16", "O_A with poisoned stale rows")


def test_cache_aware_reports_bad_indices():
    B, H, N, A, d = 2, 2, 64, 4, 32
    Q_A = _rand((B, H, A, d), 71, torch.float32)
    Kc = _rand((B, H, N, d), 72, torch.float32)
    dup = torch.tensor([[1, 2, 2, 3], [0, 1, 2, 3]], dtype=torch.int32, device=DEV)
    st = _status()
    mar.mar_attn_cache_aware(Q_A, Q_A, Q_A, Kc, Kc, dup, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_DUP
    bad = torch.tensor([[1, 2, 64, 3], [0, -1, 2, 3]], dtype=torch.int32, device=DEV)
    st = _status()
    mar.mar_attn_cache_aware(Q_A, Q_A, Q_A, Kc, Kc, bad, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_RANGE


# ------------------------------------------------------------------------------ gather + cache-aware in one call
GATHER_CASES = [(1, 2, 64, 8, 32), (2, 3, 300, 70, 64), (2, 2, 320, 40, 80), (1, 2, 100, 100, 64),
                (2, 2, 50, 1, 128), (1, 1, 1088, 114, 80), (3, 2, 257, 130, 64), (2, 3, 320, 3, 64),
                (1, 2, 640, 301, 80),
                # the Q buffer height switches at 64 queries (64-row buffers and, at d = 80, a
                # fourth K/V stage at or below it): A = 64 and 65 on both sides, at both head
                # dims; A == N has no cache block
                (1, 3, 200, 20, 64), (3, 1, 130, 64, 80), (2, 2, 200, 65, 80), (2, 1, 130, 64, 64),
                (1, 2, 48, 48, 64), (5, 1, 96, 33, 64)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,H,N,A,d", GATHER_CASES)
def test_cache_aware_gather_small(dtype, B, H, N, A, d):
    # the active rows read in place from the fresh tensors: the oracle gathers on the host
    t = DT[dtype]
    idx = _active(B, A, N, 90 + A)
    Q, K, V = (_rand((B, H, N, d), 91 + i, t) for i in range(3))
    Kc, Vc = _rand((B, H, N, d), 95, t), _rand((B, H, N, d), 96, t)
    lse = torch.empty(B, H, A, dtype=torch.float32, device=DEV)
    st = _status()
    O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, lse_out=lse, status=st)
    assert mar.mar_status_read(st) == 0
    QA, KA, VA = (_gather_host(x, idx) for x in (Q, K, V))
    O_ref, L_ref = oracle.cache_aware(QA, KA, VA, Kc, Vc, idx)
    P.assert_close(O, O_ref, dtype, "O_A (gathered in the launch)")
    np.testing.assert_allclose(lse.cpu().numpy(), L_ref, atol=1e-5 if dtype == "f32" else 2e-4, rtol=0)
    # the same kernels over dense copies of the same rows: identical bits
    d_ = lambda x: x.to(DEV).contiguous()
    O2 = mar.mar_attn_cache_aware(d_(QA), d_(KA), d_(VA), Kc, Vc, idx)
    assert torch.equal(O, O2)


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 80), ("f32", 64), ("bf16", 32)])
def test_cache_aware_gather_fused_scatter_is_bit_exact(dtype, d):
    t = DT[dtype]
    B, H, N, A = 3, 2, 200, 37
    idx = _active(B, A, N, 151)
    Q, K, V = (_rand((B, H, N, d), 152 + i, t) for i in range(3))
    Kc, Vc = _rand((B, H, N, d), 155, t), _rand((B, H, N, d), 156, t)
    Kc0, Vc0 = Kc.clone(), Vc.clone()
    st = _status()
    O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, fuse_scatter=True, status=st)
    assert mar.mar_status_read(st) == 0
    QA, KA, VA = (_gather_host(x, idx) for x in (Q, K, V))
    O_ref, _ = oracle.cache_aware(QA, KA, VA, Kc0, Vc0, idx)   # reads the pre-scatter cache
    P.assert_close(O, O_ref, dtype, "O_A")
    assert np.array_equal(oracle._rows_as_bytes(Kc.cpu()), oracle.scatter(KA, idx.cpu(), Kc0.cpu()))
    assert np.array_equal(oracle._rows_as_bytes(Vc.cpu()), oracle.scatter(VA, idx.cpu(), Vc0.cpu()))


def test_cache_aware_gather_mar_b_full_size():
    cfg = workloads.CONFIGS["mar_b"]
    ss = workloads.single_step(cfg, device=DEV)
    idx = _distinct_rows(torch.cat([ss.gen, ss.just, _active(cfg.Bp, cfg.K, cfg.N, 161)], 1), cfg.N, 162)
    Kc0, Vc0 = ss.Kc.clone(), ss.Vc.clone()
    st = _status()
    O = mar.mar_attn_cache_aware_gather(ss.Q3, ss.K3, ss.V3, ss.Kc, ss.Vc, idx, fuse_scatter=True, status=st)
    assert mar.mar_status_read(st) == 0
    QA, KA, VA = (_gather_host(x, idx) for x in (ss.Q3, ss.K3, ss.V3))
    O_ref, _ = oracle.cache_aware(QA, KA, VA, Kc0, Vc0, idx)
    P.assert_close(O, O_ref, "bf16", "MAR-B O_A (gathered in the launch)")
    assert np.array_equal(oracle._rows_as_bytes(ss.Kc.cpu()), oracle.scatter(KA, idx.cpu(), Kc0.cpu()))


@pytest.mark.parametrize("name,A", [("mar_h", 160), ("mar_h", 6), ("px512", 114)])
def test_cache_aware_gather_config_sampled_rows(name, A):
    cfg = workloads.CONFIGS[name]
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    Q, K, V = (_rand(shape, 501 + i, torch.bfloat16) for i in range(3))
    Kc, Vc = _rand(shape, 505, torch.bfloat16), _rand(shape, 506, torch.bfloat16)
    idx = _active(cfg.Bp, A, cfg.N, 510 + A)
    O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx)
    torch.cuda.synchronize()
    for b in (0, cfg.Bp // 2 + 1, cfg.Bp - 1):
        sl = slice(b, b + 1)
        QA, KA, VA = (_gather_host(x[sl], idx[sl]) for x in (Q, K, V))
        O_ref, _ = oracle.cache_aware(QA, KA, VA, Kc[sl], Vc[sl], idx[sl])
        P.assert_close(O[sl], O_ref, "bf16", f"{name} A={A} row {b}")


@pytest.mark.parametrize("d", [64, 80])
def test_cache_aware_gather_stale_rows_never_contribute(d):
    B, H, N, A = 3, 4, 320, 40
    idx = _active(B, A, N, 181 + d)
    Q, K, V = (_rand((B, H, N, d), 182 + i, torch.bfloat16) for i in range(3))
    Kc, Vc = _rand((B, H, N, d), 186, torch.bfloat16), _rand((B, H, N, d), 187, torch.bfloat16)
    Kp, Vp = Kc.clone(), Vc.clone()
    for b in range(B):
        Kp[b][:, idx[b].long()] = float("nan")
        Vp[b][:, idx[b].long()] = float("nan")
    O = mar.mar_attn_cache_aware_gather(Q, K, V, Kp, Vp, idx)
    QA, KA, VA = (_gather_host(x, idx) for x in (Q, K, V))
    O_ref, _ = oracle.cache_aware(QA, KA, VA, Kc, Vc, idx)
    P.assert_close(O, O_ref, "bf16", "O_A with poisoned stale rows")


@pytest.mark.parametrize("dtype,d,N,A", [("bf16", 64, 64, 4), ("f32", 32, 64, 4), ("bf16", 64, 8, 8),
                                         ("bf16", 80, 64, 4)])
def test_cache_aware_gather_reports_bad_indices(dtype, d, N, A):
    t = DT[dtype]
    B, H = 2, 2
    Q = _rand((B, H, N, d), 171, t)
    Kc, Vc = _rand((B, H, N, d), 172, t), _rand((B, H, N, d), 173, t)
    dup = torch.arange(A, dtype=torch.int32, device=DEV).repeat(B, 1)
    dup[0, 2] = dup[0, 1]
    st = _status()
    mar.mar_attn_cache_aware_gather(Q, Q, Q, Kc, Vc, dup, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_DUP
    bad = torch.arange(A, dtype=torch.int32, device=DEV).repeat(B, 1)
    bad[0, 2], bad[1, 1] = N, -1
    st = _status()
    mar.mar_attn_cache_aware_gather(Q, Q, Q, Kc, Vc, bad, fuse_scatter=True, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_RANGE


# ------------------------------------------------------------------------------ gather / scatter
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gather_and_scatter_bit_exact(dtype):
    t = DT[dtype]
    B, H, N, A, d = 4, 3, 321, 45, 80
    idx = _active(B, A, N, 81)
    X, Y, Z = (_rand((B, H, N, d), 82 + i, t) for i in range(3))
    gx, gy, gz = mar.mar_kv_gather([X, Y, Z], idx)
    for g, full in ((gx, X), (gy, Y), (gz, Z)):
        assert np.array_equal(oracle._rows_as_bytes(g.cpu()), oracle.gather(full.cpu(), idx.cpu()))
    Kc, Vc = _rand((B, H, N, d), 90, t), _rand((B, H, N, d), 91, t)
    K0, V0 = Kc.clone().cpu(), Vc.clone().cpu()
    KA, VA = _rand((B, H, A, d), 92, t), _rand((B, H, A, d), 93, t)
    mar.mar_kv_scatter(KA, VA, idx, Kc, Vc)
    assert np.array_equal(oracle._rows_as_bytes(Kc.cpu()), oracle.scatter(KA.cpu(), idx.cpu(), K0))
    assert np.array_equal(oracle._rows_as_bytes(Vc.cpu()), oracle.scatter(VA.cpu(), idx.cpu(), V0))


def test_full_refresh_overwrite():
    B, H, N, d = 2, 2, 100, 64
    K, V = _rand((B, H, N, d), 95, torch.bfloat16), _rand((B, H, N, d), 96, torch.bfloat16)
    Kc, Vc = torch.zeros_like(K), torch.zeros_like(V)
    mar.mar_kv_scatter(K, V, None, Kc, Vc)
    assert np.array_equal(P.bits(Kc), P.bits(K)) and np.array_equal(P.bits(Vc), P.bits(V))


def test_scatter_reports_out_of_range():
    B, H, N, A, d = 1, 1, 16, 2, 32
    X = _rand((B, H, A, d), 97, torch.float32)
    C0 = _rand((B, H, N, d), 98, torch.float32)
    C = C0.clone()
    st = _status()
    mar.mar_kv_scatter(X, X, torch.tensor([[3, 99]], dtype=torch.int32, device=DEV), C, C, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_RANGE
    assert torch.equal(C[0, 0, 3], X[0, 0, 0])          # the valid row still lands
    assert torch.equal(C[0, 0, 4:], C0[0, 0, 4:])


# ------------------------------------------------------------------------------ score + top-K
@pytest.mark.parametrize("name,G,K", [("tiny", 2, 4), ("mar_b", 4, 32), ("mar_h", 4, 16), ("mar_h", 4, 64),
                                      ("px512", 25, 64)])
def test_score_and_topk(name, G, K):
    cfg = workloads.CONFIGS[name]
    rows = cfg.Bp if cfg.Bp <= 64 else 8
    shape = (rows, cfg.H, cfg.N, cfg.d)
    Q, Kt, V = (_rand(shape, 500 + i, cfg.torch_dtype) for i in range(3))
    pos = workloads.distinct_positions(rows, 2 * G, cfg.n_buf, cfg.N, 510).to(DEV)
    gen, just = pos[:, :G].contiguous(), pos[:, G:].contiguous()
    score = torch.empty(rows, cfg.N, dtype=torch.float32, device=DEV)
    st = _status()
    mar.mar_attn_full(Q, Kt, V, gen_idx=gen, score_out=score, status=st)
    assert mar.mar_status_read(st) == 0
    ref = oracle.l2_score(Q, Kt, gen)
    got = score.cpu().numpy().astype(np.float64)
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1e-6, f"score relative error {rel.max():.3g}"
    excl = torch.cat([gen, just], 1).contiguous()
    active = torch.empty(rows, 2 * G + K, dtype=torch.int32, device=DEV)
    R = mar.mar_refresh_topk(score, excl, K, active_out=active)
    R_np = R.cpu().numpy()
    # selection logic: bit-exact against the oracle's sort of the SAME fp32 scores
    assert np.array_equal(R_np, oracle.topk(got, excl.cpu(), K))
    # end to end against the fp64 scores: exact except near-ties (logged)
    ties = P.topk_mismatches(R_np, oracle.topk(ref, excl.cpu(), K), ref, excl.cpu().numpy(), K)
    if ties:
        print(f"near-ties within {P.TIE_REL:g}: {ties}")
    assert np.array_equal(active.cpu().numpy(), np.concatenate([excl.cpu().numpy(), R_np], 1))


@pytest.mark.parametrize("B,H,N,d,dtype,G", [
    (3, 1, 200, 64, torch.bfloat16, 3),      # cluster of one CTA
    (2, 5, 333, 128, torch.bfloat16, 11),    # odd head count, two passes over the queries
    (2, 3, 97, 80, torch.float32, 2),        # fp32 rows of 20 chunks (sequential chunk sum)
    (2, 7, 77, 32, torch.float32, 9),
    (2, 20, 130, 64, torch.bfloat16, 5),     # more heads than one cluster holds: two-kernel path
    (2, 3, 333, 64, torch.bfloat16, 4),      # ragged N
    (1, 2, 64, 64, torch.bfloat16, 1),
    (2, 12, 640, 64, torch.bfloat16, 4),
])
def test_score_shapes(B, H, N, d, dtype, G):
    Q, Kt, V = (_rand((B, H, N, d), 520 + i, dtype) for i in range(3))
    gen = workloads.distinct_positions(B, G, 0, N, 530).to(DEV)
    score = torch.empty(B, N, dtype=torch.float32, device=DEV)
    st = _status()
    mar.mar_attn_full(Q, Kt, V, gen_idx=gen, score_out=score, status=st)
    assert mar.mar_status_read(st) == 0
    ref = oracle.l2_score(Q, Kt, gen)
    rel = np.abs(score.cpu().numpy().astype(np.float64) - ref) / ref
    assert rel.max() < 1e-6, f"score relative error {rel.max():.3g}"


# N % 8 == 0 takes 32-byte raw-score stores, N % 8 == 4 16-byte ones, N % 4 != 0 the separate kernel
@pytest.mark.parametrize("d,N,G", [(64, 320, 4), (80, 320, 4), (64, 333, 7), (80, 1088, 25), (64, 200, 32),
                                   (64, 200, 33), (64, 300, 4), (80, 212, 6)])
def test_score_raw_rows_and_partials_agree(d, N, G):
    # bf16 with d = 64/80: a workspace of the full size takes the raw-score rows the
    # attention launch leaves; one of the minimum size takes the separate score launch
    B, H = 3, 12
    Q, Kt, V = (_rand((B, H, N, d), 540 + i, torch.bfloat16) for i in range(3))
    gen = workloads.distinct_positions(B, G, 0, N, 550).to(DEV)
    ref = oracle.l2_score(Q, Kt, gen)
    s = mar.MarShape(B, H, N, d, mar.MAR_BF16)
    full = mar.load().mar_attn_full_workspace_bytes(s, G, 1)
    least = mar.load().mar_attn_full_min_workspace_bytes(s, G, 1)
    up = lambda n: n + (-n) % 256
    assert least == 0                     # 12 heads: the separate launch sums in a cluster, no scratch
    raw = N % 4 == 0 and G <= 32          # the raw-row form: N % 4 == 0, at most 32 generating queries
    assert full == (up(4 * B * H * G * N) + up(8 * B * H * G) if raw else 0)
    errs = []
    for nbytes in (full, least):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV) if nbytes else None
        score = torch.empty(B, N, dtype=torch.float32, device=DEV)
        st = _status()
        mar.mar_attn_full(Q, Kt, V, gen_idx=gen, score_out=score, workspace=ws, status=st)
        assert mar.mar_status_read(st) == 0
        rel = np.abs(score.cpu().numpy().astype(np.float64) - ref) / ref
        errs.append(rel.max())
    print(f"score relative error: raw rows {errs[0]:.3g}, partials {errs[1]:.3g}")
    assert max(errs) < 1e-6, errs


def test_score_raw_rows_repeated_generating_position():
    # a position listed twice counts twice in the average, as in the oracle
    B, H, N, d = 2, 4, 256, 64
    Q, Kt, V = (_rand((B, H, N, d), 560 + i, torch.bfloat16) for i in range(3))
    gen = torch.tensor([[5, 77, 5], [200, 3, 3]], dtype=torch.int32, device=DEV)
    score = torch.empty(B, N, dtype=torch.float32, device=DEV)
    st = _status()
    mar.mar_attn_full(Q, Kt, V, gen_idx=gen, score_out=score, status=st)
    assert mar.mar_status_read(st) == 0
    ref = oracle.l2_score(Q, Kt, gen)
    assert (np.abs(score.cpu().numpy().astype(np.float64) - ref) / ref).max() < 1e-6


@pytest.mark.parametrize("B,H,N,d,G,E,K", [
    (8, 12, 320, 64, 4, 8, 32),       # MAR-B head shape
    (2, 16, 1088, 80, 6, 12, 64),     # 512 px shape
    (2, 20, 130, 64, 3, 6, 10),       # more heads than a cluster: two-kernel score
    (3, 4, 200, 64, 2, 0, 7),         # no exclusions
    (2, 2, 64, 32, 1, 2, 0),          # K = 0: only the exclusions are copied
])
def test_attn_full_select_equals_full_then_topk(B, H, N, d, G, E, K):
    t = torch.bfloat16 if d != 32 else torch.float32
    Q, Kt, V = (_rand((B, H, N, d), 560 + i, t) for i in range(3))
    pos = workloads.distinct_positions(B, G + E, 0, N, 563).to(DEV)
    gen = pos[:, :G].contiguous()
    excl = pos[:, G:G + E].contiguous() if E else None
    score = torch.empty(B, N, dtype=torch.float32, device=DEV)
    R = torch.empty(B, K, dtype=torch.int32, device=DEV)
    act = torch.empty(B, E + K, dtype=torch.int32, device=DEV)
    st = _status()
    O = mar.mar_attn_full_select(Q, Kt, V, gen, excl, K, score, out_idx=R, active_out=act, status=st)
    assert mar.mar_status_read(st) == 0
    # the same call pair, separately
    O2 = mar.mar_attn_full(Q, Kt, V, gen_idx=gen, score_out=(score2 := torch.empty_like(score)))
    assert torch.equal(O, O2) and torch.equal(score, score2)
    ex_np = excl.cpu().numpy() if E else np.zeros((B, 0), np.int32)
    ref = oracle.topk(score.cpu().numpy().astype(np.float64), ex_np, K)
    if K:
        np.testing.assert_array_equal(R.cpu().numpy(), ref)
    np.testing.assert_array_equal(act.cpu().numpy(), np.concatenate([ex_np, ref], 1))


def test_attn_full_select_reports_bad_exclusion():
    B, H, N, d = 2, 12, 320, 64
    Q, Kt, V = (_rand((B, H, N, d), 570 + i, torch.bfloat16) for i in range(3))
    gen = workloads.distinct_positions(B, 4, 0, N, 571).to(DEV)
    excl = gen.clone()
    excl[1, 0] = -3
    score = torch.empty(B, N, dtype=torch.float32, device=DEV)
    R = torch.empty(B, 8, dtype=torch.int32, device=DEV)
    st = _status()
    mar.mar_attn_full_select(Q, Kt, V, gen, excl, 8, score, out_idx=R, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_RANGE
    np.testing.assert_array_equal(R[:1].cpu().numpy(),
                                  oracle.topk(score[:1].cpu().numpy().astype(np.float64), gen[:1].cpu().numpy(), 8))


@pytest.mark.parametrize("G,d", [(3, 64), (3, 80)])
def test_score_reports_bad_generating_position(G, d):
    # an out-of-range generating position is reported and left out of the score
    B, H, N = 2, 4, 150
    Q, Kt, V = (_rand((B, H, N, d), 540 + i, torch.bfloat16) for i in range(3))
    gen = workloads.distinct_positions(B, G, 0, N, 541).to(DEV)
    gen[1, 2] = N + 5
    score = torch.empty(B, N, dtype=torch.float32, device=DEV)
    st = _status()
    mar.mar_attn_full(Q, Kt, V, gen_idx=gen, score_out=score, status=st)
    assert mar.mar_status_read(st) & mar.MAR_STATUS_INDEX_RANGE
    ref0 = oracle.l2_score(Q[:1], Kt[:1], gen[:1])
    rel = np.abs(score[:1].cpu().numpy().astype(np.float64) - ref0) / ref0
    assert rel.max() < 1e-6
    # row 1: the valid generating queries only, averaged over H * G (the invalid one adds 0)
    ref1 = oracle.l2_score(Q[1:], Kt[1:], gen[1:, :2]) * (2.0 / G)
    rel1 = np.abs(score[1:].cpu().numpy().astype(np.float64) - ref1) / ref1
    assert rel1.max() < 1e-6


@pytest.mark.parametrize("N,E,K,levels", [(320, 8, 32, 0), (320, 8, 32, 5), (1088, 50, 64, 3), (64, 4, 4, 0),
                                          (300, 0, 300, 2), (4000, 10, 700, 0), (20, 3, 0, 0)])
def test_topk_selection_bit_exact(N, E, K, levels):
    g = np.random.default_rng(N + K)
    B = 6
    sc = g.random((B, N)).astype(np.float32)
    if levels:
        sc = (np.floor(sc * levels) / levels).astype(np.float32)      # many exact ties
    sc[0, :5] = [0.0, -0.0, np.inf, 1e-30, 3.0]
    excl = np.stack([g.permutation(N)[:E] for _ in range(B)]).astype(np.int32).reshape(B, E)
    score = torch.from_numpy(sc).to(DEV)
    ex = torch.from_numpy(excl).to(DEV) if E else None
    out = torch.empty(B, K, dtype=torch.int32, device=DEV)
    mar.mar_refresh_topk(score, ex, K, out_idx=out)
    if K:
        assert np.array_equal(out.cpu().numpy(), oracle.topk(sc.astype(np.float64), excl, K))


# ------------------------------------------------------------------------------ condition cache
@pytest.mark.parametrize("n", [4096 * 16, 1024 * 16 * 64, 1001])
def test_cfg_residual(n):
    cond = _rand((n,), 601, torch.float32) * 3
    res = _rand((n,), 602, torch.float32, std=0.1)
    unc = torch.empty_like(cond)
    guided = torch.empty_like(cond)
    mar.mar_cfg_residual(mar.MAR_CFG_APPLY, cond, unc, res, w=4.0, guided=guided)
    u_ref, _, g_ref = oracle.cfg(oracle.CFG_APPLY, cond, residual=res, w=4.0)
    assert np.array_equal(unc.cpu().numpy(), u_ref.astype(np.float32))      # one IEEE subtraction
    np.testing.assert_allclose(guided.cpu().numpy(), g_ref, rtol=1e-6, atol=1e-6)
    res2 = torch.empty_like(cond)
    mar.mar_cfg_residual(mar.MAR_CFG_UPDATE, cond, unc, res2)
    _, r_ref, _ = oracle.cfg(oracle.CFG_UPDATE, cond, uncond=unc)
    assert np.array_equal(res2.cpu().numpy(), r_ref.astype(np.float32))


@pytest.mark.parametrize("stale_finite", [False, True])
@pytest.mark.parametrize("A", [40, 96])
@pytest.mark.parametrize("form", ["gather", "dense"])
def test_cache_aware_fused_scatter_mar_h_full_size(form, A, stale_finite):
    # MAR-H shape (8192 short tiles, many per CTA): at A = 40 the fused scatter is written by
    # the softmax warps without a live row, at A = 96 (a single such warp, whose share would
    # be 30 16-byte chunks per lane) by the index warp; the whole cache is bit-exact and
    # sampled rows of the output match the oracle on the pre-scatter cache; with stale_finite
    # the (finite) stale V rows are used as loaded instead of zeroed
    cfg = workloads.CONFIGS["mar_h"]
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    Q, K, V = (_rand(shape, 601 + i, torch.bfloat16) for i in range(3))
    Kc, Vc = _rand(shape, 605, torch.bfloat16), _rand(shape, 606, torch.bfloat16)
    Kc0, Vc0 = Kc.clone(), Vc.clone()
    idx = _active(cfg.Bp, A, cfg.N, 607)
    st = _status()
    if form == "gather":
        O = mar.mar_attn_cache_aware_gather(Q, K, V, Kc, Vc, idx, fuse_scatter=True, status=st,
                                            stale_finite=stale_finite)
    else:
        QA, KA, VA = (torch.stack([x[b][:, idx[b].long()] for b in range(cfg.Bp)]).contiguous() for x in (Q, K, V))
        O = mar.mar_attn_cache_aware(QA, KA, VA, Kc, Vc, idx, fuse_scatter=True, status=st,
                                     stale_finite=stale_finite)
    assert mar.mar_status_read(st) == 0
    rows = [0, 129, cfg.Bp - 1]
    for b in rows:
        sl = slice(b, b + 1)
        QA_, KA_, VA_ = (_gather_host(x[sl], idx[sl]) for x in (Q, K, V))
        O_ref, _ = oracle.cache_aware(QA_, KA_, VA_, Kc0[sl], Vc0[sl], idx[sl])
        P.assert_close(O[sl], O_ref, "bf16", f"MAR-H row {b}")
    want_k, want_v = Kc0, Vc0
    for b in range(cfg.Bp):
        want_k[b][:, idx[b].long()] = K[b][:, idx[b].long()]
        want_v[b][:, idx[b].long()] = V[b][:, idx[b].long()]
    assert torch.equal(Kc, want_k) and torch.equal(Vc, want_v), "fused scatter"
