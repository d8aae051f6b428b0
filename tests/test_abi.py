"""The C-ABI library loads and exports every entry point its header declares (CPU only).

Also checks host-side argument validation, which returns before any CUDA work, so
no GPU is needed: the pointers passed are never dereferenced on those paths.
"""
import ctypes
import glob
import os
import re

import pytest

import cache_aware_attention_gb300 as mar
from cache_aware_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(mar_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mar.load()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ["mar_attn_full", "mar_attn_cache_aware", "mar_attn_cache_aware_gather", "mar_kv_scatter", "mar_kv_gather",
              "mar_refresh_topk", "mar_cfg_residual", "mar_status_read"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_build.LIB)
    missing = [n for n in _declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_error_strings(lib):
    assert mar.mar_version() >= 10000
    for code in range(0, -9, -1):
        assert mar.mar_error_string(code)
    assert mar.MAR_STATUS_TIMEOUT == 0x4


def test_status_bits_match_the_header():
    text = open(os.path.join(ROOT, "include", "marattn.h")).read()
    bits = dict(re.findall(r"#define (MAR_STATUS_[A-Z_]+) (0x[0-9a-fA-F]+)u", text))
    assert bits == {"MAR_STATUS_INDEX_RANGE": "0x1", "MAR_STATUS_INDEX_DUP": "0x2", "MAR_STATUS_TIMEOUT": "0x4"}
    for name, val in bits.items():
        assert getattr(mar, name) == int(val, 16)


def test_selftest_validation(lib):
    assert lib.mar_selftest_wait_timeout(0, FAKE, None) == -1          # limit below 1
    assert lib.mar_selftest_wait_timeout((1 << 20) + 1, FAKE, None) == -1
    assert lib.mar_selftest_wait_timeout(100, None, None) == -1        # no status word


FAKE = 1 << 20  # a 16-byte aligned non-null address that host validation never dereferences


def _shape(B=2, H=2, N=64, d=64, dtype=1):
    return ctypes.byref(mar.MarShape(B, H, N, d, dtype))


def test_attn_full_validation(lib):
    P = ctypes.c_void_p
    args = lambda s, q=FAKE, ws=None, wb=0, gen=None, G=0, score=None: (
        s, P(q), P(FAKE), P(FAKE), P(FAKE), ctypes.c_float(0), P(gen), G, P(score), None, P(ws), wb,
        None, None)
    assert lib.mar_attn_full(*args(_shape(d=48))) == -2          # unsupported head dim
    assert lib.mar_attn_full(*args(_shape(dtype=7))) == -3       # unknown dtype
    assert lib.mar_attn_full(*args(_shape(), q=0)) == -1          # NULL Q
    assert lib.mar_attn_full(*args(_shape(), q=FAKE + 8)) == -4   # misaligned
    assert lib.mar_attn_full(*args(_shape(), score=FAKE, G=0, gen=FAKE)) == -1  # score needs G >= 1
    need = lib.mar_attn_full_workspace_bytes(_shape(), 4, 1)
    assert need == 4 * 2 * 2 * 4 * 64 + 256 and need % 256 == 0  # raw-score rows + (m, l) (bf16, d = 64)
    # up to 16 heads the separate score launch needs no scratch; with more it keeps fp64
    # per-head partials
    assert lib.mar_attn_full_min_workspace_bytes(_shape(), 4, 1) == 0
    assert lib.mar_attn_full_workspace_bytes(_shape(d=32), 4, 1) == 0       # no raw-score form
    assert lib.mar_attn_full_workspace_bytes(_shape(), 33, 1) == 0          # G above 32
    least = lib.mar_attn_full_min_workspace_bytes(_shape(H=20), 4, 1)
    assert least == 8 * 2 * 20 * 64
    assert lib.mar_attn_full_workspace_bytes(_shape(H=20, d=32), 4, 1) == least
    # a score without the scratch it needs (20 heads): rejected before any launch
    assert lib.mar_attn_full(*args(_shape(H=20), score=FAKE, G=4, gen=FAKE)) == -5
    assert lib.mar_attn_full(*args(_shape(H=20), score=FAKE, G=4, gen=FAKE, ws=FAKE, wb=least - 1)) == -5
    assert lib.mar_attn_full(*args(_shape(B=0))) == 0             # empty: no-op


def test_cache_aware_validation(lib):
    P = ctypes.c_void_p
    def call(s, A, idx=FAKE, flags=0):
        return lib.mar_attn_cache_aware(s, A, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(idx),
                                        P(FAKE), ctypes.c_float(0), None, flags, None, 0, None, None)
    assert call(_shape(), 0) == 0            # A == 0 is a no-op
    assert call(_shape(), 0, flags=4) == -1  # an undefined flag bit
    assert call(_shape(), 0, flags=8) == -1
    assert call(_shape(), 65) == -1          # A > N
    assert call(_shape(), 8, idx=0) == -1    # NULL idx
    assert call(_shape(d=100), 8) == -2
    assert call(_shape(N=20000), 8) == -2    # beyond the cached-list limit


def test_topk_and_cfg_validation(lib):
    P = ctypes.c_void_p
    assert lib.mar_refresh_topk(2, 10, P(FAKE), P(FAKE), 4, 7, P(FAKE), None, None, None) == -1  # K > N-E
    assert lib.mar_refresh_topk(2, 5000, P(FAKE), P(FAKE), 4, 7, P(FAKE), None, None, None) == -2
    assert lib.mar_refresh_topk(2, 10, P(FAKE), P(FAKE), 4, 3, None, None, None, None) == -1  # no output
    assert lib.mar_refresh_topk(2, 10, P(FAKE), P(FAKE), 4, 0, None, None, None, None) == 0   # K = 0
    assert lib.mar_cfg_residual(5, 10, P(FAKE), P(FAKE), P(FAKE), ctypes.c_float(0), None, None) == -1
    assert lib.mar_cfg_residual(0, 0, None, None, None, ctypes.c_float(0), None, None) == 0


def test_rows_validation(lib):
    P = ctypes.c_void_p
    assert lib.mar_kv_scatter(_shape(), 8, P(FAKE), P(FAKE), None, P(FAKE), P(FAKE), None, None) == -1
    arr = (P * 1)(FAKE)
    assert lib.mar_kv_gather(_shape(), 8, 4, arr, arr, P(FAKE), None, None) == -1  # n_tensors > 3
    assert lib.mar_kv_gather(_shape(), 8, 1, arr, arr, None, None, None) == -1     # NULL idx


def test_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 8, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mar.mar_attn_full(x, x, x)


def test_attn_full_refresh_validation(lib):
    def call(shape, q=FAKE, k=FAKE + 256, v=FAKE + 512, o=FAKE + 768, kc=FAKE + 1024, vc=FAKE + 1280, lse=None):
        return lib.mar_attn_full_refresh(shape, q, k, v, o, kc, vc, 0.0, lse, None, None)
    assert call(_shape(d=48)) == -2                 # unsupported head dim
    assert call(_shape(), kc=None) == -1            # NULL cache
    assert call(_shape(), kc=FAKE + 256) == -1      # K cache aliases K
    assert call(_shape(), vc=FAKE + 1024) == -1     # V cache aliases K cache
    assert call(_shape(), vc=FAKE + 1288) == -4     # misaligned cache
    assert call(_shape(B=0)) == 0                   # empty: no-op


def test_next_rows_validation(lib):
    sh = lambda **k: _shape(**k)
    # token cosine: any d with whole 16-byte chunks
    assert lib.mar_token_cosine(sh(d=12), FAKE, FAKE, FAKE, None) == -2          # 24 bytes per row
    assert lib.mar_token_cosine(sh(dtype=7), FAKE, FAKE, FAKE, None) == -3
    assert lib.mar_token_cosine(sh(), None, FAKE, FAKE, None) == -1
    assert lib.mar_token_cosine(sh(), FAKE + 8, FAKE, FAKE, None) == -4
    assert lib.mar_token_cosine(sh(B=0), None, None, None, None) == 0
    # recompute set
    assert lib.mar_select_recompute(2, 16385, FAKE, 0.5, None, 0, FAKE, FAKE, None, None) == -2
    assert lib.mar_select_recompute(2, 10, FAKE, 0.5, None, 3, FAKE, FAKE, None, None) == -1   # F > 0, no force
    assert lib.mar_select_recompute(-1, 10, FAKE, 0.5, None, 0, FAKE, FAKE, None, None) == -1
    assert lib.mar_select_recompute(0, 10, None, 0.5, None, 0, None, None, None, None) == 0
    # shared refresh set
    assert lib.mar_refresh_topk_pairs(2, 4097, FAKE, FAKE, 1, 1, FAKE, None, None, None) == -2
    assert lib.mar_refresh_topk_pairs(2, 10, FAKE, FAKE, 5, 6, FAKE, None, None, None) == -1   # K > N - E
    assert lib.mar_refresh_topk_pairs(2, 10, FAKE, FAKE, 2, 3, None, None, None, None) == -1   # no output


def test_attn_full_select_validation(lib):
    need = lib.mar_attn_full_workspace_bytes(_shape(), 4, 1)
    def call(score=FAKE, G=4, gen=FAKE, excl=FAKE, E=8, K=4, out=FAKE, act=None, shape=None):
        return lib.mar_attn_full_select(shape or _shape(), FAKE, FAKE + 256, FAKE + 512, FAKE + 768, 0.0, gen, G,
                                        excl, E, K, score, out, act, None, FAKE + 4096, need, None, None)
    assert call(score=None) == -1                   # the score is required
    assert call(K=57) == -1                         # K > N - E
    assert call(excl=None) == -1                    # E > 0 without exclusions
    assert call(out=None) == -1                     # nowhere to write the selection
    assert call(out=FAKE + 2) == -4                 # misaligned
    assert call(shape=_shape(N=5000)) == -2         # top-K limit


def test_cache_aware_gather_validation(lib):
    def call(shape, A=8, q=FAKE, k=FAKE + 256, v=FAKE + 512, kc=FAKE + 1024, vc=FAKE + 1280, idx=FAKE + 2048,
             o=FAKE + 4096, flags=1):
        return lib.mar_attn_cache_aware_gather(shape, A, q, k, v, kc, vc, idx, o, 0.0, None, flags, None, None)
    assert call(_shape(), A=0) == 0                 # A == 0 is a no-op
    assert call(_shape(), A=0, flags=3) == 0        # both defined bits
    assert call(_shape(), A=0, flags=5) == -1       # an undefined flag bit
    assert call(_shape(), A=65) == -1               # A > N
    assert call(_shape(), idx=None) == -1           # NULL positions
    assert call(_shape(), kc=FAKE + 256) == -1      # K cache is the fresh K
    assert call(_shape(), vc=FAKE) == -1            # V cache is the fresh Q
    assert call(_shape(), o=FAKE + 4104) == -4      # misaligned output
    assert call(_shape(d=100)) == -2                # unsupported head dim
    assert call(_shape(N=20000)) == -2              # beyond the cached-list limit
    assert call(_shape(B=4096, H=64, N=16384)) == -2  # gather rows past 2^31
