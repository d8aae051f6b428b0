"""Cache-aware attention for masked-autoregressive (MAR) decoding on GB300.

Thin ctypes binding over the C ABI of ``libmarattn.so`` (declared in
``include/marattn.h``). Each function here has the name of the C entry point it
calls and only marshals arguments: it checks tensor dtype/shape/contiguity, passes
data pointers and the current CUDA stream, and raises ``MarError`` on a non-zero
return code. All computation runs in the library's CUDA kernels; there is no other
implementation to fall back to, so importing without the built library, or calling
with CPU tensors, fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "MarError", "MarShape", "load", "library_path", "mar_attn_full", "mar_attn_full_workspace_bytes",
    "mar_attn_full_noalloc", "mar_attn_full_refresh", "mar_attn_full_select",
    "mar_attn_cache_aware", "mar_attn_cache_aware_gather", "mar_kv_scatter", "mar_kv_gather",
    "mar_refresh_topk", "mar_refresh_topk_pairs", "mar_token_cosine", "mar_select_recompute",
    "mar_cfg_residual", "mar_status_read", "mar_error_string", "mar_version", "mar_selftest_wait_timeout",
    "MAR_F32", "MAR_BF16", "MAR_CFG_APPLY", "MAR_CFG_UPDATE",
    "MAR_STATUS_INDEX_RANGE", "MAR_STATUS_INDEX_DUP", "MAR_STATUS_TIMEOUT",
]

MAR_F32, MAR_BF16 = 0, 1
MAR_CFG_APPLY, MAR_CFG_UPDATE = 0, 1
MAR_STATUS_INDEX_RANGE, MAR_STATUS_INDEX_DUP, MAR_STATUS_TIMEOUT = 0x1, 0x2, 0x4

_lib = None


class MarError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = mar_error_string(code) if _lib is not None else str(code)
        if code == -6 and _lib is not None:
            msg += f" (cudaError {_lib.mar_last_cuda_error()})"
        super().__init__(f"{fn} failed: {code} {msg}")
        self.code = code


class MarShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
                ("d", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load ``libmarattn.so`` (built in-tree by ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with cache_aware_attention_gb300._build.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    SP = ctypes.POINTER(MarShape)
    sig = {
        "mar_error_string": ([ctypes.c_int], ctypes.c_char_p),
        "mar_last_cuda_error": ([], ctypes.c_int),
        "mar_version": ([], ctypes.c_int),
        "mar_attn_full_workspace_bytes": ([SP, I32, ctypes.c_int], SZ),
        "mar_attn_full_min_workspace_bytes": ([SP, I32, ctypes.c_int], SZ),
        "mar_attn_full": ([SP, P, P, P, P, F, P, I32, P, P, P, SZ, P, P], ctypes.c_int),
        "mar_attn_full_refresh": ([SP, P, P, P, P, P, P, F, P, P, P], ctypes.c_int),
        "mar_attn_full_select": ([SP, P, P, P, P, F, P, I32, P, I32, I32, P, P, P, P, P, SZ, P, P], ctypes.c_int),
        "mar_attn_cache_aware_workspace_bytes": ([SP, I32], SZ),
        "mar_attn_cache_aware": ([SP, I32, P, P, P, P, P, P, P, F, P, I32, P, SZ, P, P], ctypes.c_int),
        "mar_attn_cache_aware_gather": ([SP, I32, P, P, P, P, P, P, P, F, P, I32, P, P], ctypes.c_int),
        "mar_kv_scatter": ([SP, I32, P, P, P, P, P, P, P], ctypes.c_int),
        "mar_kv_gather": ([SP, I32, I32, P, P, P, P, P], ctypes.c_int),
        "mar_refresh_topk": ([I32, I32, P, P, I32, I32, P, P, P, P], ctypes.c_int),
        "mar_refresh_topk_pairs": ([I32, I32, P, P, I32, I32, P, P, P, P], ctypes.c_int),
        "mar_token_cosine": ([SP, P, P, P, P], ctypes.c_int),
        "mar_select_recompute": ([I32, I32, P, F, P, I32, P, P, P, P], ctypes.c_int),
        "mar_cfg_residual": ([I32, I64, P, P, P, F, P, P], ctypes.c_int),
        "mar_status_read": ([P, P, P], ctypes.c_int),
        "mar_noalloc_scratch_bytes": ([], SZ),
        "mar_attn_full_noalloc": ([SP, P, P, P, P, F, P, I32, P, P, P, P], ctypes.c_int),
        "mar_selftest_wait_timeout": ([ctypes.c_uint32, P, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes, f.restype = args, res
    _lib = lib
    return lib


# ----------------------------------------------------------------------------- helpers
def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MAR_BF16
    if t.dtype == torch.float32:
        return MAR_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _shape(x: torch.Tensor, N: int | None = None) -> MarShape:
    B, H, n, d = x.shape
    return MarShape(B, H, n if N is None else N, d, _dtype_code(x))


def _check(fn: str, rc: int):
    if rc != 0:
        raise MarError(fn, rc)


def mar_error_string(code: int) -> str:
    return load().mar_error_string(code).decode()


def mar_version() -> int:
    return load().mar_version()


# ----------------------------------------------------------------------------- entry points
def mar_attn_full_workspace_bytes(Q: torch.Tensor, G: int, want_score: bool) -> int:
    s = _shape(Q)
    return load().mar_attn_full_workspace_bytes(ctypes.byref(s), int(G), int(bool(want_score)))


def mar_attn_full(Q, K, V, O=None, scale: float = 0.0, gen_idx=None, score_out=None, lse_out=None,
                  workspace=None, status=None, stream=None):
    """Full bidirectional attention [B,H,N,d]; optional layer-2 score [B,N] and LSE [B,H,N].

    Returns O (allocated when not given). ``workspace`` is allocated when needed and not
    given."""
    lib = load()
    s = _shape(Q)
    if O is None:
        O = torch.empty_like(Q)
    G = 0 if gen_idx is None else int(gen_idx.shape[1])
    need = lib.mar_attn_full_workspace_bytes(ctypes.byref(s), G, int(score_out is not None))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mar_attn_full(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), float(scale),
                           _ptr(gen_idx), G, _ptr(score_out), _ptr(lse_out), _ptr(workspace), wb,
                           _ptr(status), _stream(stream))
    _check("mar_attn_full", rc)
    return O


def mar_attn_full_select(Q, K, V, gen_idx, exclude_idx, Ksel: int, score_out, O=None, out_idx=None,
                         active_out=None, scale: float = 0.0, lse_out=None, workspace=None, status=None,
                         stream=None):
    """Layer-2 call of a cached step: full attention, the score [B,N] and the refresh set
    out_idx [B,Ksel] / active set active_out [B,E+Ksel] on it (mar_attn_full followed by
    mar_refresh_topk, as one call). Returns O."""
    lib = load()
    s = _shape(Q)
    if O is None:
        O = torch.empty_like(Q)
    G = int(gen_idx.shape[1])
    E = 0 if exclude_idx is None else int(exclude_idx.shape[1])
    need = lib.mar_attn_full_workspace_bytes(ctypes.byref(s), G, 1)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mar_attn_full_select(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), float(scale),
                                  _ptr(gen_idx), G, _ptr(exclude_idx), E, int(Ksel), _ptr(score_out),
                                  _ptr(out_idx), _ptr(active_out), _ptr(lse_out), _ptr(workspace), wb,
                                  _ptr(status), _stream(stream))
    _check("mar_attn_full_select", rc)
    return O


def mar_attn_full_refresh(Q, K, V, K_cache, V_cache, O=None, scale: float = 0.0, lse_out=None, status=None,
                          stream=None):
    """Full attention of a full-refresh step plus the full cache overwrite
    (K_cache := K, V_cache := V); one launch for bf16 with d = 64 or 80. Returns O."""
    lib = load()
    s = _shape(Q)
    if O is None:
        O = torch.empty_like(Q)
    rc = lib.mar_attn_full_refresh(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(K_cache),
                                   _ptr(V_cache), float(scale), _ptr(lse_out), _ptr(status), _stream(stream))
    _check("mar_attn_full_refresh", rc)
    return O


def mar_attn_full_noalloc(Q, K, V, O=None, scale: float = 0.0, gen_idx=None, score_out=None,
                          lse_out=None, status=None, stream=None):
    """mar_attn_full without a workspace argument: the score's scratch is the library's
    built-in buffer, so the call allocates no device memory of its own (for callers that
    must not allocate). Overlapping calls on one device race on that buffer."""
    lib = load()
    s = _shape(Q)
    if O is None:
        O = torch.empty_like(Q)
    G = 0 if gen_idx is None else int(gen_idx.shape[1])
    rc = lib.mar_attn_full_noalloc(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), float(scale),
                                   _ptr(gen_idx), G, _ptr(score_out), _ptr(lse_out), _ptr(status),
                                   _stream(stream))
    _check("mar_attn_full_noalloc", rc)
    return O


MAR_CA_FUSE_SCATTER = 0x1
MAR_CA_STALE_FINITE = 0x2


def _ca_flags(fuse_scatter: bool, stale_finite: bool) -> int:
    return (MAR_CA_FUSE_SCATTER if fuse_scatter else 0) | (MAR_CA_STALE_FINITE if stale_finite else 0)


def mar_attn_cache_aware(Q_A, K_A, V_A, K_cache, V_cache, active_idx, O_A=None, scale: float = 0.0,
                         lse_out=None, fuse_scatter: bool = False, workspace=None, status=None,
                         stream=None, stale_finite: bool = False):
    """Split active/cached attention of the A active queries; returns O_A [B,H,A,d].
    stale_finite: the caller guarantees finite V_cache rows at the active positions
    (MAR_CA_STALE_FINITE)."""
    lib = load()
    A = int(Q_A.shape[2])
    s = _shape(Q_A, N=int(K_cache.shape[2]))
    if O_A is None:
        O_A = torch.empty_like(Q_A)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mar_attn_cache_aware(ctypes.byref(s), A, _ptr(Q_A), _ptr(K_A), _ptr(V_A), _ptr(K_cache),
                                  _ptr(V_cache), _ptr(active_idx), _ptr(O_A), float(scale),
                                  _ptr(lse_out), _ca_flags(fuse_scatter, stale_finite), _ptr(workspace), wb,
                                  _ptr(status), _stream(stream))
    _check("mar_attn_cache_aware", rc)
    return O_A


def mar_attn_cache_aware_gather(Q, K, V, K_cache, V_cache, active_idx, O_A=None, scale: float = 0.0,
                                lse_out=None, fuse_scatter: bool = False, status=None, stream=None,
                                stale_finite: bool = False):
    """Cache-aware attention of the active rows of the fresh Q/K/V [B,H,N,d], read in place
    through active_idx [B,A] (gather, attention and optional cache update in one launch);
    returns O_A [B,H,A,d]. stale_finite as for mar_attn_cache_aware."""
    lib = load()
    A = int(active_idx.shape[1])
    s = _shape(Q)
    if O_A is None:
        O_A = torch.empty(Q.shape[0], Q.shape[1], A, Q.shape[3], dtype=Q.dtype, device=Q.device)
    rc = lib.mar_attn_cache_aware_gather(ctypes.byref(s), A, _ptr(Q), _ptr(K), _ptr(V), _ptr(K_cache),
                                         _ptr(V_cache), _ptr(active_idx), _ptr(O_A), float(scale),
                                         _ptr(lse_out), _ca_flags(fuse_scatter, stale_finite), _ptr(status),
                                         _stream(stream))
    _check("mar_attn_cache_aware_gather", rc)
    return O_A


def mar_kv_scatter(K_A, V_A, active_idx, K_cache, V_cache, status=None, stream=None):
    """cache[b,h,idx[b,a]] = K_A/V_A[b,h,a] (active_idx None: full overwrite, A == N)."""
    ref = K_A if K_A is not None else V_A
    cache = K_cache if K_cache is not None else V_cache
    s = _shape(ref, N=int(cache.shape[2]))
    A = int(ref.shape[2])
    rc = load().mar_kv_scatter(ctypes.byref(s), A, _ptr(K_A), _ptr(V_A), _ptr(active_idx),
                               _ptr(K_cache), _ptr(V_cache), _ptr(status), _stream(stream))
    _check("mar_kv_scatter", rc)


def mar_kv_gather(srcs, active_idx, dsts=None, status=None, stream=None):
    """dst[t][b,h,a] = src[t][b,h,idx[b,a]] for up to 3 tensors; returns the dst list."""
    srcs = list(srcs)
    A = int(active_idx.shape[1])
    if dsts is None:
        dsts = [torch.empty(s.shape[0], s.shape[1], A, s.shape[3], dtype=s.dtype, device=s.device)
                for s in srcs]
    s = _shape(srcs[0])
    n = len(srcs)
    src_arr = (ctypes.c_void_p * n)(*[_ptr(x) for x in srcs])
    dst_arr = (ctypes.c_void_p * n)(*[_ptr(x) for x in dsts])
    rc = load().mar_kv_gather(ctypes.byref(s), A, n, src_arr, dst_arr, _ptr(active_idx), _ptr(status),
                              _stream(stream))
    _check("mar_kv_gather", rc)
    return dsts


def mar_refresh_topk(score, exclude_idx, K: int, out_idx=None, active_out=None, status=None, stream=None):
    """Top-K refresh positions [B,K] (ascending) and optional active set [B,E+K]."""
    B, N = score.shape
    E = 0 if exclude_idx is None else int(exclude_idx.shape[1])
    if out_idx is None:
        out_idx = torch.empty(B, K, dtype=torch.int32, device=score.device)
    rc = load().mar_refresh_topk(B, N, _ptr(score), _ptr(exclude_idx), E, int(K), _ptr(out_idx),
                                 _ptr(active_out), _ptr(status), _stream(stream))
    _check("mar_refresh_topk", rc)
    return out_idx



def mar_refresh_topk_pairs(score, exclude_idx, K: int, out_idx=None, active_out=None, status=None, stream=None):
    """Shared refresh set of guidance pairs: rows b and b + B/2 of score [B, N] take the top-K of
    their fp32 summed scores. Returns out_idx [B, K] (both rows of a pair equal)."""
    B2, N = score.shape
    if B2 % 2:
        raise ValueError("score needs an even number of rows (conditional, then unconditional)")
    E = 0 if exclude_idx is None else int(exclude_idx.shape[1])
    if out_idx is None:
        out_idx = torch.empty(B2, K, dtype=torch.int32, device=score.device)
    rc = load().mar_refresh_topk_pairs(B2 // 2, N, _ptr(score), _ptr(exclude_idx), E, int(K), _ptr(out_idx),
                                       _ptr(active_out), _ptr(status), _stream(stream))
    _check("mar_refresh_topk_pairs", rc)
    return out_idx


def mar_token_cosine(X, Y, out=None, stream=None):
    """Per-token cosine similarity [B, N] of two [B, H, N, d] tensors (a token's values over all
    heads); a [B, N, D] hidden state is passed as [B, 1, N, D]."""
    lib = load()
    if X.shape != Y.shape or X.dtype != Y.dtype:
        raise ValueError("X and Y need the same shape and dtype")
    s = _shape(X)
    if out is None:
        out = torch.empty(X.shape[0], X.shape[2], dtype=torch.float32, device=X.device)
    rc = lib.mar_token_cosine(ctypes.byref(s), _ptr(X), _ptr(Y), _ptr(out), _stream(stream))
    _check("mar_token_cosine", rc)
    return out


def mar_select_recompute(cos, tau: float, force_idx=None, out_idx=None, out_count=None, status=None, stream=None):
    """Token-cache recompute set: (idx [B, N] ascending then -1, count [B]) of the positions with
    not (cos > tau), or in force_idx [B, F]."""
    B, N = cos.shape
    F = 0 if force_idx is None else int(force_idx.shape[1])
    if out_idx is None:
        out_idx = torch.empty(B, N, dtype=torch.int32, device=cos.device)
    if out_count is None:
        out_count = torch.empty(B, dtype=torch.int32, device=cos.device)
    rc = load().mar_select_recompute(B, N, _ptr(cos), float(tau), _ptr(force_idx), F, _ptr(out_idx),
                                     _ptr(out_count), _ptr(status), _stream(stream))
    _check("mar_select_recompute", rc)
    return out_idx, out_count

def mar_cfg_residual(mode: int, cond, uncond, residual, w: float | None = None, guided=None, stream=None):
    """LazyMAR condition cache: APPLY writes uncond, UPDATE writes residual."""
    if w is None:
        w, guided = 0.0, None
    rc = load().mar_cfg_residual(int(mode), cond.numel(), _ptr(cond), _ptr(uncond), _ptr(residual),
                                 float(w), _ptr(guided), _stream(stream))
    _check("mar_cfg_residual", rc)


def mar_status_read(status, stream=None) -> int:
    out = ctypes.c_uint32(0)
    rc = load().mar_status_read(_ptr(status), ctypes.byref(out), _stream(stream))
    _check("mar_status_read", rc)
    return int(out.value)


def mar_selftest_wait_timeout(spin_limit: int, status, stream=None):
    """Diagnostic: a kernel waits on a barrier that never completes, with the bounded wait of
    the tensor-core kernels limited to ``spin_limit`` polls; it sets MAR_STATUS_TIMEOUT in
    ``status`` and returns."""
    rc = load().mar_selftest_wait_timeout(int(spin_limit), _ptr(status), _stream(stream))
    _check("mar_selftest_wait_timeout", rc)
