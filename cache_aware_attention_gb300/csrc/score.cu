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
// products are exact in fp32, each dot product accumulates in fp32 in a fixed order,
// the exponentials use the accurate expf, and every sum over keys, generating queries
// and heads is accumulated in fp64 in a fixed order (deterministic, no atomics).
//
// Kernel 1, one CTA per (b, h): every thread owns keys j = tid, tid + 128, ...; it reads
// each key row once and forms the logits of up to GCH generating queries at a time
// (query rows broadcast from shared memory). Each warp then reduces the max and the
// fp64 exponential sum of one generating query with shuffles, and every thread adds
// the normalised weights of its keys, g in order, into an fp64 accumulator.
// Kernel 2: fixed-order sum over heads, divided by H*G.
#include <cmath>

#include "common.cuh"
#include "score.h"

namespace mar {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int GCH = 8;  // generating queries per pass

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) score_partial_kernel(ScoreParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    double *acc = reinterpret_cast<double *>(smem_raw);          // [N]
    float *s = reinterpret_cast<float *>(acc + p.N);              // [GCH][N] logits
    float *qs = s + GCH * p.N;                                    // [GCH][D]
    float *stat = qs + GCH * D;                                   // [GCH][2]: max, 1/l
    __shared__ int valid[GCH];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / p.H;
    const T *__restrict__ Q = static_cast<const T *>(p.Q);
    const T *__restrict__ Kbh = static_cast<const T *>(p.K) + (int64_t)bh * p.N * D;

    for (int j = tid; j < p.N; j += kThreads) acc[j] = 0.0;

    for (int g0 = 0; g0 < p.G; g0 += GCH) {
        const int gn = min(GCH, p.G - g0);
        __syncthreads();  // previous pass done with s/qs/stat
        if (tid < GCH) {
            int ok = 0;
            if (tid < gn) {
                const int pos = p.gen[(int64_t)b * p.G + g0 + tid];
                ok = (pos >= 0 && pos < p.N);
                if (!ok) report(p.status, MAR_STATUS_INDEX_RANGE);
            }
            valid[tid] = ok;
        }
        __syncthreads();
        for (int t = tid; t < GCH * D; t += kThreads) {
            const int g = t / D, c = t % D;
            float v = 0.f;
            if (g < gn && valid[g]) {
                const int pos = p.gen[(int64_t)b * p.G + g0 + g];
                v = to_f32(Q[((int64_t)bh * p.N + pos) * D + c]);
            }
            qs[t] = v;
        }
        __syncthreads();
        // logits: one key row per thread, all generating queries of the pass. The key row
        // is held in registers 32 columns at a time; query rows are read from shared
        // memory as float4 broadcasts. Accumulation runs over c in ascending order.
        for (int j = tid; j < p.N; j += kThreads) {
            float dot[GCH];
#pragma unroll
            for (int g = 0; g < GCH; ++g) dot[g] = 0.f;
            const T *kr = Kbh + (int64_t)j * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float kv[32];
                const int w = (D - c0) < 32 ? (D - c0) : 32;   // 32, or 16 for the tail of d=80
#pragma unroll
                for (int e8 = 0; e8 < 4; ++e8) {
                    if (8 * e8 < w) {
                        if constexpr (sizeof(T) == 2) {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(kr + c0 + 8 * e8);
                            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(h2[e]);
                                kv[8 * e8 + 2 * e] = f.x;
                                kv[8 * e8 + 2 * e + 1] = f.y;
                            }
                        } else {
                            const float4 a = *reinterpret_cast<const float4 *>(kr + c0 + 8 * e8);
                            const float4 bq = *reinterpret_cast<const float4 *>(kr + c0 + 8 * e8 + 4);
                            kv[8 * e8 + 0] = a.x; kv[8 * e8 + 1] = a.y; kv[8 * e8 + 2] = a.z; kv[8 * e8 + 3] = a.w;
                            kv[8 * e8 + 4] = bq.x; kv[8 * e8 + 5] = bq.y; kv[8 * e8 + 6] = bq.z; kv[8 * e8 + 7] = bq.w;
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < GCH; ++g) {
                    if (g < gn) {
                        const float4 *q4 = reinterpret_cast<const float4 *>(qs + g * D + c0);
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            if (4 * e4 < w) {
                                const float4 q = q4[e4];
                                dot[g] = fmaf(q.x, kv[4 * e4 + 0], dot[g]);
                                dot[g] = fmaf(q.y, kv[4 * e4 + 1], dot[g]);
                                dot[g] = fmaf(q.z, kv[4 * e4 + 2], dot[g]);
                                dot[g] = fmaf(q.w, kv[4 * e4 + 3], dot[g]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < GCH; ++g)
                if (g < gn) s[g * p.N + j] = dot[g] * p.scale;
        }
        __syncthreads();
        // per generating query (one warp each): max and fp64 sum of exponentials
        for (int g = warp; g < gn; g += kWarps) {
            const float *sg = s + g * p.N;
            float mx = -INFINITY;
            for (int j = lane; j < p.N; j += 32) mx = fmaxf(mx, sg[j]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            double l = 0.0;
            for (int j = lane; j < p.N; j += 32) l += (double)expf(sg[j] - mx);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) {
                stat[2 * g] = mx;
                stat[2 * g + 1] = (float)(1.0 / l);
            }
        }
        __syncthreads();
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

__global__ void __launch_bounds__(256) score_reduce_kernel(ScoreParams p) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * 256 + threadIdx.x;
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
    return sizeof(double) * N + sizeof(float) * (GCH * N + GCH * d + 2 * GCH);
}

cudaError_t launch_score(const ScoreParams &p, cudaStream_t s) {
    cudaError_t e = p.bf16 ? launch_partial_d<bf16>(p, s) : launch_partial_d<float>(p, s);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + 255) / 256, p.B);
    score_reduce_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mar
