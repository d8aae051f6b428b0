// fp32 attention on CUDA cores: full attention and cache-aware attention.
//
// MARché notes, Key Design 2: each active query attends over fresh active K/V and
// stored cached K/V; the two softmax partial sums share one running max and running
// sum (safe online softmax), so no concatenated key buffer is ever built. Here one
// warp owns one query row and walks the key list in order: first the dense rows,
// then the cached rows of the cached set; each key updates (m, l, o) with the online
// rule  m' = max(m, s), l' = l e^(m-m') + e^(s-m'), o' = o e^(m-m') + e^(s-m') v.
// The fp32 path exists for exact-precision work; the bf16 path is the fast one.
#include <cmath>

#include "attn.h"
#include "common.cuh"

namespace mar {
namespace {

constexpr int kWarps = 8;

template <int MAXC>  // ceil(d / 32) values per lane
__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(const AttnParams p) {
    extern __shared__ int32_t smem_i[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nqt = (p.nq + kWarps - 1) / kWarps;
    const int qt = blockIdx.x % nqt, bh = blockIdx.x / nqt, b = bh / p.H;
    const int d = p.d;
    const float *__restrict__ Q = static_cast<const float *>(p.Q);
    const float *__restrict__ Kd = static_cast<const float *>(p.Kd);
    const float *__restrict__ Vd = static_cast<const float *>(p.Vd);
    float *Kc = static_cast<float *>(p.Kc);
    float *Vc = static_cast<float *>(p.Vc);

    int C = 0;
    int32_t *cached = smem_i;
    if (p.idx) {
        uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem_i + p.N);
        int32_t *wt = smem_i + p.N + ((p.N + 31) >> 5);
        C = build_cached_list(p.idx + (int64_t)b * p.A, p.A, p.N, bitmap, cached, wt, p.status);
        if (p.fuse_scatter && qt == 0) {
            // Write fresh K_A/V_A into the cache rows of the active positions. No query
            // of this launch reads those rows (they are excluded from the cached set).
            const int vec = d / 4;  // float4 per row
            for (int t = tid; t < p.A * vec; t += blockDim.x) {
                int a = t / vec, c = t % vec;
                int pos = p.idx[(int64_t)b * p.A + a];
                if (pos < 0 || pos >= p.N) continue;
                const int64_t src = dense_row(p, bh, b, a, p.n_dense) * d + 4 * c;
                const int64_t dst = ((int64_t)bh * p.N + pos) * d + 4 * c;
                *reinterpret_cast<float4 *>(Kc + dst) = *reinterpret_cast<const float4 *>(Kd + src);
                *reinterpret_cast<float4 *>(Vc + dst) = *reinterpret_cast<const float4 *>(Vd + src);
            }
        }
    }
    const int i = qt * kWarps + warp;
    if (i >= p.nq) return;

    const int64_t qrow = dense_row(p, bh, b, i, p.nq);
    float q[MAXC], o[MAXC];
#pragma unroll
    for (int k = 0; k < MAXC; ++k) {
        int c = lane + 32 * k;
        q[k] = (c < d) ? Q[qrow * d + c] : 0.f;
        o[k] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int n_keys = p.n_dense + C;
    for (int t = 0; t < n_keys; ++t) {
        const float *kr, *vr;
        if (t < p.n_dense) {
            const int64_t r = dense_row(p, bh, b, t, p.n_dense);
            kr = Kd + r * d;
            vr = Vd + r * d;
        } else {
            int pos = cached[t - p.n_dense];
            kr = Kc + ((int64_t)bh * p.N + pos) * d;
            vr = Vc + ((int64_t)bh * p.N + pos) * d;
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < MAXC; ++k) {
            int c = lane + 32 * k;
            if (c < d) dot = fmaf(q[k], kr[c], dot);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float s = dot * p.scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);  // m = -inf on the first key -> 0
        const float e = expf(s - m_new);
        l = l * alpha + e;
#pragma unroll
        for (int k = 0; k < MAXC; ++k) {
            int c = lane + 32 * k;
            if (c < d) o[k] = o[k] * alpha + e * vr[c];
        }
        m = m_new;
    }
    const float inv = 1.f / l;
    float *O = static_cast<float *>(p.O);
#pragma unroll
    for (int k = 0; k < MAXC; ++k) {
        int c = lane + 32 * k;
        if (c < d) O[((int64_t)bh * p.nq + i) * d + c] = o[k] * inv;
    }
    if (p.lse && lane == 0) p.lse[(int64_t)bh * p.nq + i] = m + logf(l);
}

template <int MAXC>
cudaError_t launch(const AttnParams &p, cudaStream_t s) {
    static int configured[64] = {0};
    size_t smem = 0;
    if (p.idx) smem = sizeof(int32_t) * (p.N + ((p.N + 31) / 32) + kWarps);
    cudaError_t e = ensure_smem(attn_f32_kernel<MAXC>, smem, configured);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)((p.nq + kWarps - 1) / kWarps) * p.B * p.H;
    attn_f32_kernel<MAXC><<<(unsigned)blocks, kWarps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_f32(const AttnParams &p, cudaStream_t s) {
    if (p.d <= 32) return launch<1>(p, s);
    if (p.d <= 64) return launch<2>(p, s);
    if (p.d <= 96) return launch<3>(p, s);
    return launch<4>(p, s);
}

}  // namespace mar
