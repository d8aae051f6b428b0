// Internal launch interface of the attention kernels (host + device visible).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mar {

// One attention launch: for every (b, h) the queries Q[bh, 0..nq) attend over a key
// list made of
//   - the dense rows Kd/Vd[bh, 0..n_dense)                (fresh K_A/V_A, or all of K/V),
//   - followed, when idx != nullptr, by the cache rows Kc/Vc[bh, p] for every
//     position p in [0, N) that is not in idx[b, 0..A)  (the cached set, ascending).
// Full attention: Kd/Vd = K/V with n_dense = N, idx = nullptr; with store_kv the launch
// also copies K/V into Kc/Vc (the full cache refresh).
// Cache-aware attention: Kd/Vd = K_A/V_A with n_dense = A, idx = active positions.
// With `fresh` set, Q/Kd/Vd are the whole fresh tensors [B*H, N, d] and row a of the
// active set is read at row idx[b, a] (the active gather folded into the launch).
struct AttnParams {
    const void *Q;      // [B*H, nq, d]
    const void *Kd;     // [B*H, n_dense, d]
    const void *Vd;
    void *Kc;           // [B*H, N, d] cache (written at active rows when fuse_scatter,
                        // everywhere when store_kv)
    void *Vc;
    const int32_t *idx; // [B, A] active positions, or nullptr
    void *O;            // [B*H, nq, d]
    float *lse;         // [B*H, nq] natural-log LSE, or nullptr
    uint32_t *status;
    int B, H, N, d;
    int nq, n_dense, A;
    int fuse_scatter;
    int stale_finite;   // cache-aware: the V cache rows at active positions are finite, so the
                        // tensor-core kernel need not zero them before P.V (their P is 0)
    int fresh;          // cache-aware only: Q/Kd/Vd are [B*H, N, d], active row a at idx[b, a]
    // Full attention (tcgen05 kernel): the rows of the generating queries gen[b, 0..G) also
    // leave their raw scores and softmax statistics for the layer-2 score (under the first
    // slot g of a position listed more than once):
    //   gen_s[bh, g, j] = q_{gen[b,g]} . k_j (unscaled; the fp32 tensor-core accumulation the
    //   attention itself uses), gen_ml[bh, g] = (m, l) of the row's own online softmax:
    //   weight_j = 2^(gen_s * scale * log2(e) - m) / l.
    const int32_t *gen; // [B, G] or nullptr
    int G;              // <= 32
    float *gen_s;       // [B*H, G, N]
    float2 *gen_ml;     // [B*H, G]
    int store_kv;       // full attention only: Kc/Vc := Kd/Vd (tcgen05 kernel only)
    float scale;        // softmax scale
};

#ifdef __CUDACC__
// Row of Q/Kd/Vd holding dense row a of (b, h): a itself, or with `fresh` the active
// position idx[b, a] of the whole tensor (an out-of-range position reads row 0 of the slab;
// the bitmap build reports it).
__device__ __forceinline__ int64_t dense_row(const AttnParams &p, int bh, int b, int a, int rows) {
    if (!p.fresh) return (int64_t)bh * rows + a;
    const int pos = p.idx[(int64_t)b * p.A + a];
    return (int64_t)bh * p.N + ((pos >= 0 && pos < p.N) ? pos : 0);
}
#endif

// Launchers. Return the cudaError_t of the launch.
cudaError_t launch_attn_f32(const AttnParams &p, cudaStream_t s);
cudaError_t launch_attn_bf16_mma(const AttnParams &p, cudaStream_t s);
// tcgen05/TMEM/TMA kernel (head dim 64 or 80).
bool attn_tc5_supported(const AttnParams &p);
cudaError_t launch_attn_bf16_tc5(const AttnParams &p, cudaStream_t s);
// Cache-aware launches of 65 to 96 queries: 96-row Q buffers and one more K/V stage
// (attn_tc5_q96.cu).
cudaError_t launch_attn_bf16_tc5_q96(const AttnParams &p, cudaStream_t s);

// bf16 attention: the tcgen05 kernel where it supports the shape, else the mma.sync one.
inline cudaError_t launch_attn_bf16(const AttnParams &p, cudaStream_t s) {
    return attn_tc5_supported(p) ? launch_attn_bf16_tc5(p, s) : launch_attn_bf16_mma(p, s);
}

}  // namespace mar
