// Layer-2 head-averaged relevance score.
//
// MARché notes, Key Design 1: during layer-2 full attention the softmax weights from
// every generating query to every token are averaged across heads (and here across the
// generating queries) into one relevance score per token; the top-K tokens become the
// refreshing tokens:
//   score[b, j] = 1/(H G) sum_h sum_g exp(s_hgj - lse_hg),  s_hgj = scale <q_{h,gen_g}, k_{h,j}>.
//
// The refresh set must match an exact evaluation except where two candidates lie within
// 1e-6 (relative) of each other, so this path is kept well below that error: bf16
// products are exact in fp32, dot products accumulate in fp32 in a fixed order, the
// exponentials use the accurate expf, and every sum over keys, generating queries and
// heads is accumulated in fp64 in a fixed order (deterministic, no atomics).
//
// Two kernels: per-(b, h) partial sums over g into a workspace [B, H, N], then a fixed
// order reduction over h.
#include <cmath>

#include "common.cuh"
#include "score.h"

namespace mar {
namespace {

constexpr int kThreads = 256;
constexpr int GC = 4;  // generating queries per pass

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) score_partial_kernel(ScoreParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    double *acc = reinterpret_cast<double *>(smem_raw);        // [N] sum over g of p_gj
    float *s = reinterpret_cast<float *>(acc + p.N);            // [GC][N] logits
    float *qs = s + GC * p.N;                                   // [GC][D]
    double *red = reinterpret_cast<double *>(qs + GC * D);     // [kThreads]
    float *stat = reinterpret_cast<float *>(red + kThreads);    // [2*GC]: max, 1/l
    __shared__ int valid[GC];

    const int tid = threadIdx.x;
    const int bh = blockIdx.x, b = bh / p.H;
    const T *__restrict__ Q = static_cast<const T *>(p.Q);
    const T *__restrict__ K = static_cast<const T *>(p.K);
    const T *__restrict__ Kbh = K + (int64_t)bh * p.N * D;

    for (int j = tid; j < p.N; j += kThreads) acc[j] = 0.0;

    for (int g0 = 0; g0 < p.G; g0 += GC) {
        const int gn = min(GC, p.G - g0);
        __syncthreads();
        if (tid < GC) {
            int ok = 0;
            if (tid < gn) {
                int pos = p.gen[(int64_t)b * p.G + g0 + tid];
                ok = (pos >= 0 && pos < p.N);
                if (!ok) report(p.status, MAR_STATUS_INDEX_RANGE);
            }
            valid[tid] = ok;
        }
        __syncthreads();
        for (int t = tid; t < GC * D; t += kThreads) {
            int g = t / D, c = t % D;
            float v = 0.f;
            if (g < gn && valid[g]) {
                int pos = p.gen[(int64_t)b * p.G + g0 + g];
                v = to_f32(Q[((int64_t)bh * p.N + pos) * D + c]);
            }
            qs[t] = v;
        }
        __syncthreads();
        // logits s[g][j] (fixed accumulation order over c)
        for (int j = tid; j < p.N; j += kThreads) {
            float dot[GC];
#pragma unroll
            for (int g = 0; g < GC; ++g) dot[g] = 0.f;
            const T *kr = Kbh + (int64_t)j * D;
#pragma unroll 4
            for (int c = 0; c < D; ++c) {
                const float kv = to_f32(kr[c]);
#pragma unroll
                for (int g = 0; g < GC; ++g) dot[g] = fmaf(qs[g * D + c], kv, dot[g]);
            }
#pragma unroll
            for (int g = 0; g < GC; ++g) s[g * p.N + j] = dot[g] * p.scale;
        }
        __syncthreads();
        // per generating query: max and (fp64) sum of exponentials
        for (int g = 0; g < gn; ++g) {
            float mx = -INFINITY;
            for (int j = tid; j < p.N; j += kThreads) mx = fmaxf(mx, s[g * p.N + j]);
            red[tid] = (double)mx;
            __syncthreads();
            for (int w = kThreads / 2; w > 0; w >>= 1) {
                if (tid < w) red[tid] = fmax(red[tid], red[tid + w]);
                __syncthreads();
            }
            const float m = (float)red[0];
            __syncthreads();
            double l = 0.0;
            for (int j = tid; j < p.N; j += kThreads) l += (double)expf(s[g * p.N + j] - m);
            red[tid] = l;
            __syncthreads();
            for (int w = kThreads / 2; w > 0; w >>= 1) {
                if (tid < w) red[tid] += red[tid + w];
                __syncthreads();
            }
            if (tid == 0) {
                stat[2 * g] = m;
                stat[2 * g + 1] = (float)(1.0 / red[0]);
            }
            __syncthreads();
        }
        // accumulate the normalised weights over g (fixed order g = 0..gn-1)
        for (int j = tid; j < p.N; j += kThreads) {
            double a = acc[j];
            for (int g = 0; g < gn; ++g)
                if (valid[g]) a += (double)(expf(s[g * p.N + j] - stat[2 * g]) * stat[2 * g + 1]);
            acc[j] = a;
        }
    }
    __syncthreads();
    for (int j = tid; j < p.N; j += kThreads) p.partial[(int64_t)bh * p.N + j] = acc[j];
}

__global__ void __launch_bounds__(kThreads) score_reduce_kernel(ScoreParams p) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * kThreads + threadIdx.x;
    if (j >= p.N) return;
    double a = 0.0;
    for (int h = 0; h < p.H; ++h) a += p.partial[((int64_t)b * p.H + h) * p.N + j];
    p.score[(int64_t)b * p.N + j] = (float)(a / ((double)p.H * (double)p.G));
}

template <typename T, int D>
cudaError_t launch_partial(const ScoreParams &p, cudaStream_t s) {
    static int configured[64] = {0};
    const size_t smem = score_smem_bytes(p.N, D);
    cudaError_t e = ensure_smem(score_partial_kernel<T, D>, smem, configured);
    if (e != cudaSuccess) return e;
    score_partial_kernel<T, D><<<p.B * p.H, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_partial_d(const ScoreParams &p, cudaStream_t s) {
    switch (p.d) {
        case 32: return launch_partial<T, 32>(p, s);
        case 64: return launch_partial<T, 64>(p, s);
        case 80: return launch_partial<T, 80>(p, s);
        case 128: return launch_partial<T, 128>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t score_smem_bytes(int N, int d) {
    return sizeof(double) * N + sizeof(float) * (GC * N + GC * d) + sizeof(double) * kThreads +
           sizeof(float) * 2 * GC;
}

cudaError_t launch_score(const ScoreParams &p, cudaStream_t s) {
    cudaError_t e = p.bf16 ? launch_partial_d<bf16>(p, s) : launch_partial_d<float>(p, s);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kThreads - 1) / kThreads, p.B);
    score_reduce_kernel<<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mar
