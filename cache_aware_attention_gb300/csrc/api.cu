// Host side of the C ABI declared in include/marattn.h: argument validation, workspace
// accounting and kernel dispatch. Every entry point validates on the host, launches on
// the caller's stream and returns without synchronising (except mar_status_read).
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "attn.h"
#include "marattn.h"
#include "score.h"

namespace {

thread_local int g_last_cuda = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda = (int)e;
    return MAR_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t elem_size(int dtype) { return dtype == MAR_BF16 ? 2 : 4; }

int check_shape(const mar_shape *s) {
    if (!s) return MAR_ERR_ARG;
    if (s->dtype != MAR_F32 && s->dtype != MAR_BF16) return MAR_ERR_DTYPE;
    if (s->B < 0 || s->H < 0 || s->N < 0) return MAR_ERR_ARG;
    if (s->d != 32 && s->d != 64 && s->d != 80 && s->d != 128) return MAR_ERR_SHAPE;
    return MAR_OK;
}

// Row copies take any row of whole 16-byte vectors (up to 16384 elements), e.g. hidden
// states [B, 1, N, D] of a token cache.
int check_rows_shape(const mar_shape *s) {
    if (!s) return MAR_ERR_ARG;
    if (s->dtype != MAR_F32 && s->dtype != MAR_BF16) return MAR_ERR_DTYPE;
    if (s->B < 0 || s->H < 0 || s->N < 0 || s->d < 0) return MAR_ERR_ARG;
    if (s->d == 0 || s->d > 16384 || (s->d * (int)elem_size(s->dtype)) % 16 != 0) return MAR_ERR_SHAPE;
    return MAR_OK;
}

constexpr size_t kWsAlign = 256;
size_t round_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

// Largest N for which the list of cached positions fits in shared memory.
constexpr int kMaxCacheN = 16384;

float resolve_scale(float scale, int d) { return scale > 0.f ? scale : 1.0f / std::sqrt((float)d); }

}  // namespace

namespace mar {
// Lets other translation units of the library report a failed CUDA call.
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }
}  // namespace mar

extern "C" {

const char *mar_error_string(int code) {
    switch (code) {
        case MAR_OK: return "ok";
        case MAR_ERR_ARG: return "invalid argument";
        case MAR_ERR_SHAPE: return "unsupported shape (head dim must be 32, 64, 80 or 128; size limits)";
        case MAR_ERR_DTYPE: return "unsupported element type";
        case MAR_ERR_ALIGN: return "pointer not aligned (16 bytes for tensors, 4 for fp32 arrays)";
        case MAR_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case MAR_ERR_CUDA: return "CUDA error (see mar_last_cuda_error)";
        case MAR_ERR_NODEV: return "no usable CUDA device";
        case MAR_ERR_SCRATCH_LIMIT:
            return "shape needs more scratch than the library's built-in no-allocation buffer holds";
        default: return "unknown error";
    }
}

int mar_last_cuda_error(void) { return g_last_cuda; }

int mar_version(void) { return 10000; }

// Score scratch: with the tcgen05 attention (bf16, d = 64 or 80), G <= 32 and N % 4 == 0 the attention
// launch leaves the generating rows' raw scores (fp32 [B*H, G, N]) for a small reduction;
// otherwise a separate score launch computes the score, which needs scratch only with more
// than 16 heads (per-head fp64 partials [B*H, N]; up to 16 heads it sums in a cluster).
static constexpr int kMaxFusedG = 32;
static bool fused_score_shape(const mar_shape *s, int32_t G) {
    if (s->dtype != MAR_BF16 || G <= 0 || G > kMaxFusedG || (long long)s->H * G * 16 > 40 * 1024 || (s->N & 3))
        return false;
    mar::AttnParams p{};
    p.d = s->d;
    return mar::attn_tc5_supported(p);
}
static size_t ws_rows(const mar_shape *s, int32_t G) {  // raw scores, then (m, l) per row
    return round_up(sizeof(float) * (size_t)s->B * s->H * G * s->N) + round_up(sizeof(float) * 2 * s->B * s->H * G);
}
static size_t ws_partials(const mar_shape *s) {
    return mar::score_uses_partials(s->H) ? round_up(sizeof(double) * (size_t)s->B * s->H * s->N) : 0;
}

size_t mar_attn_full_workspace_bytes(const mar_shape *s, int32_t G, int want_score) {
    if (check_shape(s) != MAR_OK || !want_score || G <= 0) return 0;
    return fused_score_shape(s, G) ? ws_rows(s, G) : ws_partials(s);
}

size_t mar_attn_full_min_workspace_bytes(const mar_shape *s, int32_t G, int want_score) {
    const size_t need = mar_attn_full_workspace_bytes(s, G, want_score);
    return need ? std::min(need, ws_partials(s)) : 0;
}

// Full attention, optionally with the layer-2 score and, when `select`, the top-K refresh
// set and active set built on it.
static int attn_full_core(const mar_shape *s, const void *Q, const void *K, const void *V, void *O, float scale,
                          const int32_t *gen_idx, int32_t G, float *score_out, float *lse_out, void *workspace,
                          size_t workspace_bytes, uint32_t *d_status, mar_stream_t stream, bool select,
                          const int32_t *exclude_idx, int32_t E, int32_t Ksel, int32_t *out_idx,
                          int32_t *active_out) {
    int rc = check_shape(s);
    if (rc != MAR_OK) return rc;
    if (s->B == 0 || s->H == 0 || s->N == 0) return MAR_OK;
    if (!Q || !K || !V || !O) return MAR_ERR_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return MAR_ERR_ALIGN;
    if (!aligned4(lse_out) || !aligned4(score_out)) return MAR_ERR_ALIGN;
    const bool want_score = score_out != nullptr;
    if (want_score && (G <= 0 || !gen_idx)) return MAR_ERR_ARG;
    if (want_score && mar::score_smem_bytes(s->N, s->d) > 220 * 1024) return MAR_ERR_SHAPE;
    if (select) {
        if (!want_score || E < 0 || Ksel < 0) return MAR_ERR_ARG;
        if (s->N > 4096) return MAR_ERR_SHAPE;
        if (E > s->N || Ksel > s->N - E) return MAR_ERR_ARG;
        if (E > 0 && !exclude_idx) return MAR_ERR_ARG;
        if (!out_idx && !active_out && Ksel > 0) return MAR_ERR_ARG;
        if (!aligned4(out_idx) || !aligned4(active_out)) return MAR_ERR_ALIGN;
    }
    // the score's scratch: the raw-row form when it fits (see mar_attn_full_workspace_bytes),
    // else the per-head partials of the separate score kernel
    const bool ws_ok = workspace && !(reinterpret_cast<uintptr_t>(workspace) % kWsAlign);
    const bool fused = want_score && fused_score_shape(s, G) && ws_ok && workspace_bytes >= ws_rows(s, G);
    const size_t need_partials = ws_partials(s);
    if (want_score && !fused && need_partials && (!ws_ok || workspace_bytes < need_partials)) return MAR_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    mar::AttnParams p{};
    p.Q = Q; p.Kd = K; p.Vd = V; p.Kc = nullptr; p.Vc = nullptr; p.idx = nullptr;
    p.O = O; p.lse = lse_out; p.status = d_status;
    p.B = s->B; p.H = s->H; p.N = s->N; p.d = s->d;
    p.nq = s->N; p.n_dense = s->N; p.A = 0; p.fuse_scatter = 0;
    p.scale = resolve_scale(scale, s->d);
    if (fused) {
        p.gen = gen_idx; p.G = G; p.gen_s = static_cast<float *>(workspace);
        p.gen_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                              round_up(sizeof(float) * (size_t)s->B * s->H * G * s->N));
    }
    cudaError_t e = (s->dtype == MAR_BF16) ? mar::launch_attn_bf16(p, st) : mar::launch_attn_f32(p, st);
    if (e != cudaSuccess) return cuda_fail(e);

    if (fused) {
        e = mar::launch_score_rows(p.gen_s, p.gen_ml, gen_idx, score_out, s->B, s->H, G, s->N, p.scale, st);
        if (e != cudaSuccess) return cuda_fail(e);
    } else if (want_score) {
        mar::ScoreParams sp{};
        sp.Q = Q; sp.K = K; sp.gen = gen_idx;
        sp.partial = need_partials ? static_cast<double *>(workspace) : nullptr;
        sp.score = score_out; sp.status = d_status;
        sp.B = s->B; sp.H = s->H; sp.N = s->N; sp.d = s->d; sp.G = G;
        sp.bf16 = s->dtype == MAR_BF16;
        sp.scale = p.scale;
        e = mar::launch_score(sp, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (want_score && select && (out_idx || active_out)) {
        mar::TopkParams tp{};
        tp.score = score_out; tp.exclude = exclude_idx; tp.out = out_idx; tp.active = active_out;
        tp.status = d_status; tp.B = s->B; tp.N = s->N; tp.E = E; tp.K = Ksel;
        e = mar::launch_topk(tp, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return MAR_OK;
}

int mar_attn_full(const mar_shape *s, const void *Q, const void *K, const void *V, void *O,
                  float scale, const int32_t *gen_idx, int32_t G, float *score_out, float *lse_out,
                  void *workspace, size_t workspace_bytes, uint32_t *d_status, mar_stream_t stream) {
    return attn_full_core(s, Q, K, V, O, scale, gen_idx, G, score_out, lse_out, workspace, workspace_bytes,
                          d_status, stream, false, nullptr, 0, 0, nullptr, nullptr);
}

int mar_attn_full_select(const mar_shape *s, const void *Q, const void *K, const void *V, void *O, float scale,
                         const int32_t *gen_idx, int32_t G, const int32_t *exclude_idx, int32_t E, int32_t Ksel,
                         float *score_out, int32_t *out_idx, int32_t *active_out, float *lse_out,
                         void *workspace, size_t workspace_bytes, uint32_t *d_status, mar_stream_t stream) {
    return attn_full_core(s, Q, K, V, O, scale, gen_idx, G, score_out, lse_out, workspace, workspace_bytes,
                          d_status, stream, true, exclude_idx, E, Ksel, out_idx, active_out);
}

int mar_attn_cache_aware_gather(const mar_shape *s, int32_t A, const void *Q, const void *K, const void *V,
                                void *K_cache, void *V_cache, const int32_t *active_idx, void *O_A, float scale,
                                float *lse_out, int32_t fuse_scatter, uint32_t *d_status, mar_stream_t stream) {
    int rc = check_shape(s);
    if (rc != MAR_OK) return rc;
    if (A < 0 || A > s->N) return MAR_ERR_ARG;
    if (fuse_scatter & ~(MAR_CA_FUSE_SCATTER | MAR_CA_STALE_FINITE)) return MAR_ERR_ARG;
    if (A == 0 || s->B == 0 || s->H == 0) return MAR_OK;
    if (!Q || !K || !V || !K_cache || !V_cache || !active_idx || !O_A) return MAR_ERR_ARG;
    // the cache is written (fused scatter) while the fresh tensors are read: distinct buffers
    if (K_cache == K || V_cache == V || K_cache == V_cache || K_cache == Q || V_cache == Q) return MAR_ERR_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(K_cache) || !aligned16(V_cache) ||
        !aligned16(O_A) || !aligned4(lse_out) || !aligned4(active_idx))
        return MAR_ERR_ALIGN;
    if (s->N > kMaxCacheN) return MAR_ERR_SHAPE;
    if ((long long)s->B * s->H * s->N > 0x7fffffffLL) return MAR_ERR_SHAPE;  // gather row coordinates
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    mar::AttnParams p{};
    p.Q = Q; p.Kd = K; p.Vd = V; p.Kc = K_cache; p.Vc = V_cache; p.idx = active_idx;
    p.O = O_A; p.lse = lse_out; p.status = d_status;
    p.B = s->B; p.H = s->H; p.N = s->N; p.d = s->d;
    p.nq = A; p.n_dense = A; p.A = A; p.fresh = 1;
    p.fuse_scatter = (fuse_scatter & MAR_CA_FUSE_SCATTER) ? 1 : 0;
    p.stale_finite = (fuse_scatter & MAR_CA_STALE_FINITE) ? 1 : 0;
    p.scale = resolve_scale(scale, s->d);
    cudaError_t e = (s->dtype == MAR_BF16) ? mar::launch_attn_bf16(p, st) : mar::launch_attn_f32(p, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return MAR_OK;
}

static int rows_common(const mar_shape *s, int32_t A, int n, const void *const *src, void *const *dst,
                       const int32_t *idx, int scatter, uint32_t *d_status, mar_stream_t stream);

int mar_attn_full_refresh(const mar_shape *s, const void *Q, const void *K, const void *V, void *O,
                          void *K_cache, void *V_cache, float scale, float *lse_out, uint32_t *d_status,
                          mar_stream_t stream) {
    int rc = check_shape(s);
    if (rc != MAR_OK) return rc;
    if (s->B == 0 || s->H == 0 || s->N == 0) return MAR_OK;
    if (!Q || !K || !V || !O || !K_cache || !V_cache) return MAR_ERR_ARG;
    if (K_cache == K || V_cache == V || K_cache == V_cache) return MAR_ERR_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(K_cache) ||
        !aligned16(V_cache))
        return MAR_ERR_ALIGN;
    if (!aligned4(lse_out)) return MAR_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    mar::AttnParams p{};
    p.Q = Q; p.Kd = K; p.Vd = V; p.Kc = K_cache; p.Vc = V_cache; p.idx = nullptr;
    p.O = O; p.lse = lse_out; p.status = d_status;
    p.B = s->B; p.H = s->H; p.N = s->N; p.d = s->d;
    p.nq = s->N; p.n_dense = s->N; p.A = 0; p.fuse_scatter = 0; p.store_kv = 1;
    p.scale = resolve_scale(scale, s->d);
    const bool fused = s->dtype == MAR_BF16 && mar::attn_tc5_supported(p);
    cudaError_t e = fused ? mar::launch_attn_bf16_tc5(p, st)
                          : (s->dtype == MAR_BF16 ? mar::launch_attn_bf16(p, st) : mar::launch_attn_f32(p, st));
    if (e != cudaSuccess) return cuda_fail(e);
    if (fused) return MAR_OK;
    // other kernels: the refresh as a second launch (a plain row copy)
    const void *src[2] = {K, V};
    void *dst[2] = {K_cache, V_cache};
    return rows_common(s, s->N, 2, src, dst, nullptr, 1, d_status, stream);
}

// The cache-aware kernels need no scratch; the workspace arguments are reserved.
size_t mar_attn_cache_aware_workspace_bytes(const mar_shape *s, int32_t A) {
    (void)s;
    (void)A;
    return 0;
}

int mar_attn_cache_aware(const mar_shape *s, int32_t A, const void *Q_A, const void *K_A,
                         const void *V_A, void *K_cache, void *V_cache, const int32_t *active_idx,
                         void *O_A, float scale, float *lse_out, int32_t fuse_scatter, void *workspace,
                         size_t workspace_bytes, uint32_t *d_status, mar_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    int rc = check_shape(s);
    if (rc != MAR_OK) return rc;
    if (A < 0 || A > s->N) return MAR_ERR_ARG;
    if (fuse_scatter & ~(MAR_CA_FUSE_SCATTER | MAR_CA_STALE_FINITE)) return MAR_ERR_ARG;
    if (A == 0 || s->B == 0 || s->H == 0) return MAR_OK;
    if (!Q_A || !K_A || !V_A || !K_cache || !V_cache || !active_idx || !O_A) return MAR_ERR_ARG;
    if (!aligned16(Q_A) || !aligned16(K_A) || !aligned16(V_A) || !aligned16(K_cache) ||
        !aligned16(V_cache) || !aligned16(O_A) || !aligned4(lse_out) || !aligned4(active_idx))
        return MAR_ERR_ALIGN;
    if (s->N > kMaxCacheN) return MAR_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    mar::AttnParams p{};
    p.Q = Q_A; p.Kd = K_A; p.Vd = V_A; p.Kc = K_cache; p.Vc = V_cache; p.idx = active_idx;
    p.O = O_A; p.lse = lse_out; p.status = d_status;
    p.B = s->B; p.H = s->H; p.N = s->N; p.d = s->d;
    p.nq = A; p.n_dense = A; p.A = A;
    p.fuse_scatter = (fuse_scatter & MAR_CA_FUSE_SCATTER) ? 1 : 0;
    p.stale_finite = (fuse_scatter & MAR_CA_STALE_FINITE) ? 1 : 0;
    p.scale = resolve_scale(scale, s->d);
    cudaError_t e = (s->dtype == MAR_BF16) ? mar::launch_attn_bf16(p, st) : mar::launch_attn_f32(p, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return MAR_OK;
}

static int rows_common(const mar_shape *s, int32_t A, int n, const void *const *src, void *const *dst,
                       const int32_t *idx, int scatter, uint32_t *d_status, mar_stream_t stream) {
    int rc = check_rows_shape(s);
    if (rc != MAR_OK) return rc;
    if (A < 0 || A > s->N || n < 1 || n > 3) return MAR_ERR_ARG;
    if (!idx && A != s->N) return MAR_ERR_ARG;
    if (A == 0 || s->B == 0 || s->H == 0) return MAR_OK;
    mar::RowCopyParams p{};
    int k = 0;
    for (int t = 0; t < n; ++t) {
        if (!src[t] && !dst[t]) continue;
        if (!src[t] || !dst[t]) return MAR_ERR_ARG;
        if (!aligned16(src[t]) || !aligned16(dst[t])) return MAR_ERR_ALIGN;
        p.src[k] = src[t];
        p.dst[k] = dst[t];
        ++k;
    }
    if (k == 0) return MAR_OK;
    p.n_tensors = k;
    p.idx = idx;
    p.status = d_status;
    p.B = s->B; p.H = s->H; p.N = s->N; p.A = A;
    p.row_bytes = (int)(s->d * elem_size(s->dtype));
    p.scatter = scatter;
    cudaError_t e = mar::launch_rows(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

int mar_kv_scatter(const mar_shape *s, int32_t A, const void *K_A, const void *V_A,
                   const int32_t *active_idx, void *K_cache, void *V_cache, uint32_t *d_status,
                   mar_stream_t stream) {
    const void *src[2] = {K_A, V_A};
    void *dst[2] = {K_cache, V_cache};
    return rows_common(s, A, 2, src, dst, active_idx, 1, d_status, stream);
}

int mar_kv_gather(const mar_shape *s, int32_t A, int32_t n_tensors, const void *const *src,
                  void *const *dst, const int32_t *active_idx, uint32_t *d_status, mar_stream_t stream) {
    if (!src || !dst || !active_idx) return MAR_ERR_ARG;
    return rows_common(s, A, n_tensors, src, dst, active_idx, 0, d_status, stream);
}

int mar_refresh_topk(int32_t B, int32_t N, const float *score, const int32_t *exclude_idx, int32_t E,
                     int32_t K, int32_t *out_idx, int32_t *active_out, uint32_t *d_status,
                     mar_stream_t stream) {
    if (B < 0 || N < 0 || E < 0 || K < 0) return MAR_ERR_ARG;
    if (N > 4096) return MAR_ERR_SHAPE;
    if (E > N || K > N - E) return MAR_ERR_ARG;
    if (B == 0 || N == 0) return MAR_OK;
    if (!score || (E > 0 && !exclude_idx)) return MAR_ERR_ARG;
    if (!out_idx && !active_out) return K == 0 ? MAR_OK : MAR_ERR_ARG;
    mar::TopkParams p{};
    p.score = score; p.exclude = exclude_idx; p.out = out_idx; p.active = active_out;
    p.status = d_status; p.B = B; p.N = N; p.E = E; p.K = K;
    cudaError_t e = mar::launch_topk(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

int mar_refresh_topk_pairs(int32_t B_pairs, int32_t N, const float *score, const int32_t *exclude_idx, int32_t E,
                           int32_t K, int32_t *out_idx, int32_t *active_out, uint32_t *d_status,
                           mar_stream_t stream) {
    if (B_pairs < 0 || N < 0 || E < 0 || K < 0) return MAR_ERR_ARG;
    if (N > 4096) return MAR_ERR_SHAPE;
    if (E > N || K > N - E) return MAR_ERR_ARG;
    if (B_pairs == 0 || N == 0) return MAR_OK;
    if (!score || (E > 0 && !exclude_idx)) return MAR_ERR_ARG;
    if (!out_idx && !active_out) return K == 0 ? MAR_OK : MAR_ERR_ARG;
    mar::TopkParams p{};
    p.score = score; p.exclude = exclude_idx; p.out = out_idx; p.active = active_out;
    p.status = d_status; p.B = B_pairs; p.N = N; p.E = E; p.K = K; p.pairs = 1;
    cudaError_t e = mar::launch_topk(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

int mar_token_cosine(const mar_shape *s, const void *X, const void *Y, float *cos_out, mar_stream_t stream) {
    if (!s) return MAR_ERR_ARG;
    if (s->B < 0 || s->H < 0 || s->N < 0 || s->d < 0) return MAR_ERR_ARG;
    if (s->dtype != MAR_BF16 && s->dtype != MAR_F32) return MAR_ERR_DTYPE;
    const int elem = s->dtype == MAR_BF16 ? 2 : 4;
    if (s->d == 0 || (s->d * elem) % 16 != 0 || s->d > 16384) return MAR_ERR_SHAPE;
    if (s->B == 0 || s->H == 0 || s->N == 0) return MAR_OK;
    if (!X || !Y || !cos_out) return MAR_ERR_ARG;
    if (!aligned16(X) || !aligned16(Y) || !aligned4(cos_out)) return MAR_ERR_ALIGN;
    cudaError_t e = mar::launch_token_cosine(X, Y, cos_out, s->B, s->H, s->N, s->d, s->dtype == MAR_BF16,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

int mar_select_recompute(int32_t B, int32_t N, const float *cos, float tau, const int32_t *force_idx, int32_t F,
                         int32_t *out_idx, int32_t *out_count, uint32_t *d_status, mar_stream_t stream) {
    if (B < 0 || N < 0 || F < 0) return MAR_ERR_ARG;
    if (N > 16384) return MAR_ERR_SHAPE;
    if (B == 0 || N == 0) return MAR_OK;
    if (!cos || !out_idx || !out_count || (F > 0 && !force_idx)) return MAR_ERR_ARG;
    if (!aligned4(cos) || !aligned4(out_idx) || !aligned4(out_count)) return MAR_ERR_ALIGN;
    mar::SelectParams p{};
    p.cos = cos; p.force = F > 0 ? force_idx : nullptr; p.out = out_idx; p.count = out_count;
    p.status = d_status; p.B = B; p.N = N; p.F = F; p.tau = tau;
    cudaError_t e = mar::launch_select_recompute(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

int mar_cfg_residual(int32_t mode, int64_t n, const float *cond, float *uncond, float *residual,
                     float w, float *guided, mar_stream_t stream) {
    if (mode != MAR_CFG_APPLY && mode != MAR_CFG_UPDATE) return MAR_ERR_ARG;
    if (n < 0) return MAR_ERR_ARG;
    if (n == 0) return MAR_OK;
    if (!cond || !uncond || !residual) return MAR_ERR_ARG;
    cudaError_t e = mar::launch_cfg(mode, n, cond, uncond, residual, w, guided,
                                    reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

int mar_status_read(const uint32_t *d_status, uint32_t *h_status, mar_stream_t stream) {
    if (!d_status || !h_status) return MAR_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(h_status, d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? MAR_OK : cuda_fail(e);
}

}  // extern "C"
