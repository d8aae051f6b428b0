"""mar_attn_full_noalloc: the allocation-free variant of mar_attn_full (GPU).

Some callers of this library cannot allocate device memory -- for instance a plugin
inside a host framework whose allocator owns the whole device pool, or a decode loop
that must not risk an allocation stalling or failing mid-step. For them the layer-2
score's scratch lives in a fixed buffer compiled into the library. This file checks,
through the C ABI that two calls in a row give the same output as mar_attn_full with a
caller workspace (within the bf16 / fp32 tolerances used by the other parity tests), that
at a shape whose score takes the separate launch it matches the fp64 oracle directly, and
that a shape beyond the buffer is rejected with its own error code.

It lives in a file of its own, named to be collected last, so that a failure here does
not stop a -x run before the other tests; it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import _parity as P
import cache_aware_attention_gb300 as mar
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from cache_aware_attention_gb300 import _build
    _build.build()
    return mar.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, Q, K, V, gen, score, lse, status):
    s = mar.MarShape(*Q.shape, mar.MAR_BF16 if Q.dtype == torch.bfloat16 else mar.MAR_F32)
    O = torch.empty_like(Q)
    rc = lib.mar_attn_full_noalloc(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), ctypes.c_float(0.0),
                                   _ptr(gen), gen.shape[1], _ptr(score), _ptr(lse), _ptr(status),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, O


@pytest.mark.parametrize("name,dtype", [("mar_b", torch.bfloat16), ("mar_b", torch.float32)])
def test_noalloc_matches_workspace_call_twice(lib, name, dtype):
    cfg = workloads.CONFIGS[name]
    dt = "bf16" if dtype == torch.bfloat16 else "f32"
    for call, seed in enumerate((901, 902)):           # two calls in a row, different inputs
        shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
        Q, K, V = (workloads.normal(shape, seed * 10 + i, dtype, "cuda") for i in range(3))
        gen = workloads.distinct_positions(cfg.Bp, cfg.G, cfg.n_buf, cfg.N, seed).cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        score_a = torch.empty(cfg.Bp, cfg.N, dtype=torch.float32, device="cuda")
        lse_a = torch.empty(cfg.Bp, cfg.H, cfg.N, dtype=torch.float32, device="cuda")
        rc, O_a = _noalloc(lib, Q, K, V, gen, score_a, lse_a, st)
        assert rc == 0, mar.mar_error_string(rc)
        score_b = torch.empty_like(score_a)
        lse_b = torch.empty_like(lse_a)
        O_b = mar.mar_attn_full(Q, K, V, gen_idx=gen, score_out=score_b, lse_out=lse_b, status=st)
        torch.cuda.synchronize()
        assert mar.mar_status_read(st) == 0
        P.assert_close(O_a, P.to_np(O_b).astype(np.float64), dt, f"call {call} O")
        s_a, s_b = score_a.cpu().numpy().astype(np.float64), score_b.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(s_a - s_b) / s_b) < 1e-6, f"call {call} score"
        np.testing.assert_allclose(lse_a.cpu().numpy(), lse_b.cpu().numpy(), atol=1e-5, rtol=0)


def test_noalloc_matches_the_oracle_where_the_score_takes_the_separate_launch(lib):
    # MAR-H shape: the raw-score rows (4*B*H*G*N = 42 MB) do not fit the 24 MiB buffer, so the
    # call computes the score in the separate launch, which needs no scratch at 16 heads
    cfg = workloads.CONFIGS["mar_h"]
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    s = mar.MarShape(*shape, mar.MAR_BF16)
    assert lib.mar_attn_full_workspace_bytes(ctypes.byref(s), cfg.G, 1) > lib.mar_noalloc_scratch_bytes()
    Q, K, V = (workloads.normal(shape, 930 + i, torch.bfloat16, "cuda") for i in range(3))
    gen = workloads.distinct_positions(cfg.Bp, cfg.G, cfg.n_buf, cfg.N, 931).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        score = torch.full((cfg.Bp, cfg.N), float("nan"), dtype=torch.float32, device="cuda")
        rc, O = _noalloc(lib, Q, K, V, gen, score, None, st)
        assert rc == 0, mar.mar_error_string(rc)
        torch.cuda.synchronize()
        assert mar.mar_status_read(st) == 0
        for b in (0, cfg.Bp - 1):
            sl = slice(b, b + 1)
            O_ref, _ = oracle.full_attn(Q[sl], K[sl], V[sl])
            P.assert_close(O[sl], O_ref, "bf16", f"call {call} row {b} O")
            ref = oracle.l2_score(Q[sl], K[sl], gen[sl])
            assert np.max(np.abs(score[sl].cpu().numpy() - ref) / ref) < 1e-6, f"call {call} row {b} score"


def test_noalloc_rejects_shapes_beyond_its_buffer(lib):
    limit = lib.mar_noalloc_scratch_bytes()
    assert limit == 24 << 20
    # 20 heads: the separate score launch keeps fp64 partials, 8*B*H*N = 26.2 MB, and the
    # raw-score rows (52 MB) do not fit either: rejected on the host before any launch
    s = mar.MarShape(512, 20, 320, 64, mar.MAR_BF16)
    assert lib.mar_attn_full_min_workspace_bytes(ctypes.byref(s), 4, 1) > limit
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.mar_attn_full_noalloc(ctypes.byref(s), fake, fake, fake, fake, ctypes.c_float(0.0), fake, 4,
                                   fake, None, None, None)
    assert rc == -8 and "no-allocation" in mar.mar_error_string(rc)
