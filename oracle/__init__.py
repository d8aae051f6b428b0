"""CPU oracle for cache-aware attention in MAR decoding (fp64, plain loops).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library never does,
and the two share no code. The arithmetic lives in ``mar_oracle.c`` (plain C,
double precision, compiled with gcc); this module only converts arrays and calls
it through ctypes. Each function names the passage it follows in its C comment.

Parity status of each function (pins live in ``tests/test_oracle_pins.py``):
  full_attn          pinned: torch fp64 SDPA, hand-derived fixtures, closed forms
  cache_aware        pinned: equals full attention over the concatenated current
                     K/V (paper's Appendix A), C=0 reduction, split == concat,
                     permutation invariance
  scatter / gather   pinned: numpy fancy indexing, untouched rows unchanged
  l2_score           pinned: row sums = 1, head linearity, single-query softmax
  topk               pinned: numpy lexsort, brute-force subset search, ties
  cfg                pinned: closed-form identities, exact fp32 subtraction
  token_cosine       pinned: scipy's cosine distance, closed forms (x vs x, -x, 2x,
                     orthogonal), a hand-derived case, zero-vector conventions
  select_recompute   pinned: threshold edge cases (equal to tau, NaN), forced tokens
  topk_pairs         pinned: pair symmetry, numpy lexsort of the fp32 summed scores
  stale_attention_error
                     pinned: zero on a current cache (the Appendix A equivalence) and
                     with every position active, positive and growing with the drift
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mar_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

CFG_APPLY, CFG_UPDATE = 0, 1


def build(force: bool = False) -> str:
    """Compile ``mar_oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
            lib.oracle_full_attn.argtypes = [I, I, I, I, P, P, P, D, P, P]
            lib.oracle_full_attn.restype = None
            for f in (lib.oracle_cache_aware_concat, lib.oracle_cache_aware_split):
                f.argtypes = [I, I, I, I, I, P, P, P, P, P, P, D, P, P]
                f.restype = ctypes.c_int
            for f in (lib.oracle_scatter_rows, lib.oracle_gather_rows):
                f.argtypes = [I, I, I, I, I, P, P, P]
                f.restype = None
            lib.oracle_l2_score.argtypes = [I, I, I, I, I, P, P, P, D, P]
            lib.oracle_l2_score.restype = None
            lib.oracle_topk.argtypes = [I, I, P, I, P, I, P]
            lib.oracle_topk.restype = ctypes.c_int
            lib.oracle_cfg.argtypes = [ctypes.c_int, I, P, P, P, D, P, P, P]
            lib.oracle_token_cosine.argtypes = [I, I, I, I, P, P, P]
            lib.oracle_token_cosine.restype = None
            lib.oracle_select_recompute.argtypes = [I, I, P, ctypes.c_float, P, I, P, P]
            lib.oracle_select_recompute.restype = ctypes.c_int
            lib.oracle_cfg.restype = None
            _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    """Exact float32 copy of a bf16/fp32 tensor or array (bf16 -> fp32 is exact)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu")
        if x.dtype != torch.float32:
            x = x.to(torch.float32)
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_scale(d: int) -> float:
    """1/sqrt(d): the standard transformer softmax scale (not printed on the pages)."""
    return 1.0 / math.sqrt(d)


def full_attn(Q, K, V, scale: float | None = None):
    """Full bidirectional attention. Q [..., Nq, d], K/V [..., Nk, d] -> (O, LSE) fp64."""
    q, k, v = _f32(Q), _f32(K), _f32(V)
    *lead, Nq, d = q.shape
    Nk = k.shape[-2]
    BH = int(np.prod(lead)) if lead else 1
    O = np.empty((BH, Nq, d), np.float64)
    L = np.empty((BH, Nq), np.float64)
    _load().oracle_full_attn(BH, Nq, Nk, d, _ptr(q), _ptr(k), _ptr(v),
                             default_scale(d) if scale is None else scale, _ptr(O), _ptr(L))
    return O.reshape(*lead, Nq, d), L.reshape(*lead, Nq)


def cache_aware(Q_A, K_A, V_A, Kc, Vc, idx, scale: float | None = None,
                method: str = "concat"):
    """Cache-aware attention of active queries.

    Q_A/K_A/V_A [B, H, A, d]; Kc/Vc [B, H, N, d]; idx [B, A] -> (O [B,H,A,d], LSE
    [B,H,A]) fp64. ``method`` "concat" builds the concatenated key list, "split"
    runs the two partial softmax paths and merges them."""
    q, ka, va, kc, vc, ix = _f32(Q_A), _f32(K_A), _f32(V_A), _f32(Kc), _f32(Vc), _i32(idx)
    B, H, A, d = q.shape
    N = kc.shape[2]
    O = np.empty((B, H, A, d), np.float64)
    L = np.empty((B, H, A), np.float64)
    fn = {"concat": _load().oracle_cache_aware_concat,
          "split": _load().oracle_cache_aware_split}[method]
    rc = fn(B, H, N, A, d, _ptr(q), _ptr(ka), _ptr(va), _ptr(kc), _ptr(vc), _ptr(ix),
            default_scale(d) if scale is None else scale, _ptr(O), _ptr(L))
    if rc != 0:
        raise ValueError("active index rows must hold distinct positions in [0, N)")
    return O, L


def _rows_as_bytes(x):
    """View a tensor/array as raw bytes with its last axis flattened to bytes."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").contiguous()
        x = x.view(torch.uint8) if x.dtype.itemsize == 1 else x.view(
            {2: torch.int16, 4: torch.int32, 8: torch.int64}[x.dtype.itemsize])
        x = x.numpy()
    x = np.ascontiguousarray(x)
    return x.view(np.uint8).reshape(*x.shape[:-1], x.shape[-1] * x.itemsize)


def scatter(src, idx, cache) -> np.ndarray:
    """Return a copy of ``cache`` [B,H,N,row] with rows idx[b,a] := src[b,h,a] (bytes)."""
    s, c = _rows_as_bytes(src), _rows_as_bytes(cache).copy()
    ix = _i32(idx)
    B, H, N, rb = c.shape
    A = ix.shape[1]
    _load().oracle_scatter_rows(B, H, N, A, rb, _ptr(s), _ptr(ix), _ptr(c))
    return c


def gather(full, idx) -> np.ndarray:
    """dst[b,h,a] = full[b,h,idx[b,a]] as raw bytes [B,H,A,row_bytes]."""
    f = _rows_as_bytes(full)
    ix = _i32(idx)
    B, H, N, rb = f.shape
    A = ix.shape[1]
    dst = np.empty((B, H, A, rb), np.uint8)
    _load().oracle_gather_rows(B, H, N, A, rb, _ptr(f), _ptr(ix), _ptr(dst))
    return dst


def l2_score(Q, K, gen, scale: float | None = None) -> np.ndarray:
    """Head-averaged layer-2 relevance score [B, N] (fp64)."""
    q, k, g = _f32(Q), _f32(K), _i32(gen)
    B, H, N, d = q.shape
    G = g.shape[1]
    out = np.empty((B, N), np.float64)
    _load().oracle_l2_score(B, H, N, d, G, _ptr(q), _ptr(k), _ptr(g),
                            default_scale(d) if scale is None else scale, _ptr(out))
    return out


def topk(score, exclude, K: int) -> np.ndarray:
    """Refresh set [B, K] int32: top-K of score over non-excluded positions, ascending."""
    if hasattr(score, "detach"):
        score = score.detach().to("cpu").double().numpy()
    sc = np.ascontiguousarray(score, dtype=np.float64)
    B, N = sc.shape
    ex = _i32(exclude).reshape(B, -1)
    E = ex.shape[1]
    out = np.zeros((B, K), np.int32)
    if K > 0 and _load().oracle_topk(B, N, _ptr(sc), E, _ptr(ex), K, _ptr(out)) != 0:
        raise ValueError("fewer than K candidates, or exclude out of range")
    return out


def cfg(mode: int, cond, uncond=None, residual=None, w: float | None = None):
    """LazyMAR condition cache. Returns (uncond_out, residual_out, guided) fp64;
    entries not produced by ``mode`` are None."""
    c = _f32(cond)
    n = c.size
    u = _f32(uncond) if uncond is not None else np.zeros(1, np.float32)
    r = _f32(residual) if residual is not None else np.zeros(1, np.float32)
    uo = np.empty(c.shape, np.float64) if mode == CFG_APPLY else None
    ro = np.empty(c.shape, np.float64) if mode == CFG_UPDATE else None
    go = np.empty(c.shape, np.float64) if w is not None else None
    _load().oracle_cfg(mode, n, _ptr(c), _ptr(u), _ptr(r), 0.0 if w is None else float(w),
                       _ptr(uo) if uo is not None else None,
                       _ptr(ro) if ro is not None else None,
                       _ptr(go) if go is not None else None)
    return uo, ro, go


def token_cosine(X, Y) -> np.ndarray:
    """Per-token cosine similarity [B, N] (fp64) of two [B, H, N, d] feature tensors,
    a token's feature being its values over all heads."""
    x, y = _f32(X), _f32(Y)
    B, H, N, d = x.shape
    out = np.empty((B, N), np.float64)
    _load().oracle_token_cosine(B, H, N, d, _ptr(x), _ptr(y), _ptr(out))
    return out


def select_recompute(cos, tau: float, force=None):
    """Token-cache recompute set from fp32 similarities [B, N]: positions with not
    (cos > tau), or forced; returns (idx [B, N] ascending then -1, count [B])."""
    c = _f32(cos)
    B, N = c.shape
    f = _i32(force).reshape(B, -1) if force is not None else np.zeros((B, 0), np.int32)
    F = f.shape[1]
    idx = np.empty((B, N), np.int32)
    cnt = np.empty(B, np.int32)
    if _load().oracle_select_recompute(B, N, _ptr(c), np.float32(tau), _ptr(f) if F else None, F,
                                       _ptr(idx), _ptr(cnt)) != 0:
        raise ValueError("forced position out of range")
    return idx, cnt


def topk_pairs(score, exclude, K: int) -> np.ndarray:
    """Shared refresh set of classifier-free-guidance pairs: rows b and b + B/2 take the
    top-K of the fp32 sum of their scores (an IEEE single addition, as on the GPU), with
    row b's exclusions; returns [B, K] with both rows of a pair equal."""
    sc = _f32(score)
    B2, N = sc.shape
    Bp = B2 // 2
    comb = (sc[:Bp] + sc[Bp:]).astype(np.float32)      # float32 + float32 in float32
    ex = _i32(exclude).reshape(B2, -1)
    R = topk(comb.astype(np.float64), ex[:Bp], K)
    return np.concatenate([R, R], 0)


def stale_attention_error(Q_A, K_A, V_A, Kc, Vc, K_fresh, V_fresh, idx) -> float:
    """MARché notes, Background & Motivation and Key Design 3: between full refreshes the
    cached K/V go stale. The error this leaves in a cached step's output is the relative
    Frobenius distance between the cache-aware attention of the active queries over the
    stale cache and full attention of the same queries over the fresh K/V (which is what
    cache-aware attention over a current cache computes, by the Appendix A equivalence):
        ||O_stale - O_full||_F / ||O_full||_F    (fp64)."""
    O_stale, _ = cache_aware(Q_A, K_A, V_A, Kc, Vc, idx)
    O_full, _ = full_attn(Q_A, K_fresh, V_fresh)
    return float(np.linalg.norm(O_stale - O_full) / np.linalg.norm(O_full))
