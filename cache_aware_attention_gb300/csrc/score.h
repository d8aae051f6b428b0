// Internal launch interface of the layer-2 score, top-K, row-copy and guidance kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mar {

struct ScoreParams {
    const void *Q;          // [B*H, N, d] (layer-2 queries of all tokens)
    const void *K;          // [B*H, N, d]
    const int32_t *gen;     // [B, G] generating positions
    double *partial;        // workspace [B*H, N]: per-head sum over g of softmax weights
    float *score;           // [B, N]
    uint32_t *status;
    int B, H, N, d, G;
    int bf16;               // element type of Q/K
    float scale;
};

// Heads per thread-block cluster of the main score kernel. Up to this many heads the
// head sum runs through distributed shared memory and `partial` is not used; more heads
// take the two-kernel path, which keeps per-head fp64 partials in the workspace.
constexpr int kScoreMaxClusterHeads = 16;
inline bool score_uses_partials(int H) { return H > kScoreMaxClusterHeads; }

size_t score_smem_bytes(int N, int d);
cudaError_t launch_score(const ScoreParams &p, cudaStream_t s);

// The layer-2 score from what the attention launch left for the generating rows: raw
// scores gen_s [B*H, G, N] (unscaled q . k) and per row the (m, l) of its online softmax
// (weight_j = 2^(s_j * scale * log2(e) - m) / l):
// score[b, j] = (1/(H G)) sum_{h,g} weight_{h,g,j} (generating positions out of range add 0).
cudaError_t launch_score_rows(const float *gen_s, const float2 *gen_ml, const int32_t *gen, float *score, int B,
                              int H, int G, int N, float scale, cudaStream_t s);

struct TopkParams {
    const float *score;     // [B, N] (pairs: [2B, N])
    const int32_t *exclude; // [B, E] or nullptr (pairs: [2B, E])
    int32_t *out;           // [B, K] or nullptr (pairs: [2B, K])
    int32_t *active;        // [B, E + K] or nullptr (pairs: [2B, E + K])
    uint32_t *status;
    int B, N, E, K;         // pairs: B = number of pairs
    int pairs;              // rows b and b + B share one set, selected on the fp32 sum of their scores
};

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s);

// Token-cache recompute set: per row the positions with not (cos > tau), or forced,
// ascending, then -1; count per row.
struct SelectParams {
    const float *cos;       // [B, N]
    const int32_t *force;   // [B, F] or nullptr
    int32_t *out;           // [B, N]
    int32_t *count;         // [B]
    uint32_t *status;
    int B, N, F;
    float tau;
};
cudaError_t launch_select_recompute(const SelectParams &p, cudaStream_t s);

// Per-token cosine similarity of two [B, H, N, d] tensors over each token's H*d values.
cudaError_t launch_token_cosine(const void *X, const void *Y, float *out, int B, int H, int N, int d, int is_bf16,
                                cudaStream_t s);

struct RowCopyParams {
    const void *src[3];
    void *dst[3];
    int n_tensors;
    const int32_t *idx;     // [B, A] positions, or nullptr for the identity map (A == N)
    uint32_t *status;
    int B, H, N, A;
    int row_bytes;          // multiple of 16
    int scatter;            // 1: dst[bh, idx] = src[bh, a]; 0: dst[bh, a] = src[bh, idx]
};

cudaError_t launch_rows(const RowCopyParams &p, cudaStream_t s);
cudaError_t launch_cfg(int mode, int64_t n, const float *cond, float *uncond, float *residual,
                       float w, float *guided, cudaStream_t s);

}  // namespace mar
