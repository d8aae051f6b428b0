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
// the exponentials use the accurate expf on an argument carried as an fp32 pair (so that
// peaked rows, whose tail weights have arguments of -50 and below, keep their relative
// accuracy; see exp_scaled_diff), and every sum over keys, generating queries
// and heads is accumulated with fp64-grade accuracy in a fixed order (deterministic,
// no atomics).
//
// Main path (H <= 16): one thread-block cluster of H CTAs per batch row, CTA h owning
// head h. The (b, h) key slab streams through two 12 KB shared-memory buffers filled by
// bulk copies. Each warp takes 4 key rows (d = 64) per step, one 16-byte chunk per lane,
// with that lane's chunk of up to 4 generating queries in registers; a chunk's products
// accumulate in fp32 in element order and the chunks of a row are added in a fixed
// shuffle order. One warp per generating query takes the max and the sum of
// exponentials; every thread adds the normalised weights of its keys, g in order. These
// sums use double-float arithmetic (an fp32 pair with error-free two-sums: fp64-grade
// accuracy without the fp64 pipe, which is slow on this part). After a cluster barrier
// CTA r sums a slice of the keys over the H heads' accumulators (distributed shared
// memory, h in order) and writes score = sum / (H G).
// Fallback (H > 16): kernel 1 per (b, h) writes the per-head accumulator to the
// workspace; kernel 2 sums over heads in the same order.
#include <cmath>

#include <cooperative_groups.h>

#include "common.cuh"
#include "gen_rows.cuh"
#include "score.h"
#include "tc5.cuh"

namespace mar {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int GCH = 8;  // generating queries per pass

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) score_partial_kernel(ScoreParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    double *acc = reinterpret_cast<double *>(smem_raw);          // [N]
    float *s = reinterpret_cast<float *>(acc + p.N);              // [GCH][N] dot products (unscaled)
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
                if (g < gn) s[g * p.N + j] = dot[g];
        }
        __syncthreads();
        // per generating query (one warp each): max and fp64 sum of exponentials (the scale
        // is positive, so the max of the unscaled dot products is the max logit)
        for (int g = warp; g < gn; g += kWarps) {
            const float *sg = s + g * p.N;
            float mx = -INFINITY;
            for (int j = lane; j < p.N; j += 32) mx = fmaxf(mx, sg[j]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            double l = 0.0;
            for (int j = lane; j < p.N; j += 32) l += (double)exp_scaled_diff(sg[j], mx, p.scale);
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
                if (valid[g]) a += (double)(exp_scaled_diff(s[g * p.N + j], stat[2 * g], p.scale) * stat[2 * g + 1]);
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

// ------------------------------------------------------------------------ cluster kernel
constexpr int kCThreads = 128;   // 4 warps: with <= 80 registers and ~33 KB, 6 CTAs per SM
constexpr int kCWarps = kCThreads / 32;
constexpr int kMaxCluster = kScoreMaxClusterHeads;
constexpr int kQReg = 4;                // generating queries per pass (held in registers)
constexpr int kBufBytes = 12 * 1024;    // one of two staging buffers for key rows

// key rows per staged chunk
inline int cluster_rows(int N, int row_bytes) {
    const int r = kBufBytes / row_bytes;
    return N < r ? N : r;
}

size_t cluster_smem_bytes(int N, int D, int elem) {
    const size_t kbuf = 2 * (size_t)cluster_rows(N, D * elem) * D * elem;
    return kbuf + sizeof(float) * ((size_t)2 * N + (size_t)kQReg * N);
}

template <typename T>
MAR_DEVINL void load_chunk(const T *src, float (&v)[16 / sizeof(T)]) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(src);
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            v[2 * e] = f.x;
            v[2 * e + 1] = f.y;
        }
    } else {
        v[0] = __uint_as_float(raw.x); v[1] = __uint_as_float(raw.y);
        v[2] = __uint_as_float(raw.z); v[3] = __uint_as_float(raw.w);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kCThreads, 6) score_cluster_kernel(ScoreParams p, int krows) {
    namespace cg = cooperative_groups;
    using namespace tc5;
    cg::cluster_group cluster = cg::this_cluster();
    constexpr int E = 16 / sizeof(T);      // elements per 16-byte chunk
    constexpr int CH = D / E;              // chunks per key row
    constexpr int RPW = 32 / CH;           // key rows per warp step
    static_assert(D % E == 0 && CH <= 32, "row must be whole 16-byte chunks, at most 32");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *kbuf = reinterpret_cast<T *>(smem_raw);                                          // [2][krows][D]
    float *acc_hi = reinterpret_cast<float *>(smem_raw + 2 * (size_t)krows * D * sizeof(T));  // [N]
    float *acc_lo = acc_hi + p.N;                                                       // [N]
    float *s = acc_lo + p.N;                                      // [kQReg][N] dot products (unscaled)
    __shared__ float stat[kQReg][2];                              // max, 1/l
    __shared__ int valid[kQReg];
    __shared__ __align__(8) uint64_t kbar[2];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, b = blockIdx.y, bh = b * p.H + h;
    const T *__restrict__ Q = static_cast<const T *>(p.Q);
    const T *__restrict__ Kbh = static_cast<const T *>(p.K) + (int64_t)bh * p.N * D;
    const int c = lane % CH, rsub = lane / CH;   // chunk of the row, row within the step
    const bool lane_used = rsub < RPW;
    const int nchunk = (p.N + krows - 1) / krows;
    const int npass = (p.G + kQReg - 1) / kQReg;
    const int nuse = npass * nchunk;             // staged chunks over all passes

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&kbar[0], 1);
        mbar_init(&kbar[1], 1);
        mbar_fence_init();
    }
    for (int j = tid; j < p.N; j += kCThreads) acc_hi[j] = acc_lo[j] = 0.f;
    __syncthreads();
    // chunk use u (u = pass * nchunk + ck) lands in buffer u % 2
    auto stage = [&](int u) {
        const int ck = u % nchunk, r0 = ck * krows, nr = min(krows, p.N - r0);
        const uint32_t bytes = (uint32_t)nr * D * sizeof(T);
        mbar_arrive_expect_tx(&kbar[u & 1], bytes);
        bulk_load(kbuf + (size_t)(u & 1) * krows * D, Kbh + (int64_t)r0 * D, bytes, &kbar[u & 1]);
    };
    if (tid == 0) {
        stage(0);
        if (nuse > 1) stage(1);
    }

    int u = 0;
    for (int pass = 0; pass < npass; ++pass) {
        const int g0 = pass * kQReg, gn = min(kQReg, p.G - g0);
        // this lane's chunk of every generating query of the pass, in registers
        float qr[kQReg][E];
        int okm = 0;
#pragma unroll
        for (int g = 0; g < kQReg; ++g) {
            int pos = -1;
            if (g < gn) {
                pos = p.gen[(int64_t)b * p.G + g0 + g];
                if (pos < 0 || pos >= p.N) pos = -1;
            }
            if (pos >= 0 && lane_used) {
                load_chunk<T>(Q + ((int64_t)bh * p.N + pos) * D + c * E, qr[g]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) qr[g][e] = 0.f;
            }
            okm |= (pos >= 0) << g;
        }
        if (tid < kQReg) {
            valid[tid] = (okm >> tid) & 1;
            if (tid < gn && !((okm >> tid) & 1) && h == 0) report(p.status, MAR_STATUS_INDEX_RANGE);
        }
        // logits: each warp takes RPW key rows per step, lane (rsub, c) holding chunk c of
        // row rsub; products accumulate in element order within a chunk, then the chunks of
        // a row are added in a fixed order (a butterfly when CH is a power of two, else
        // chunk 0, 1, ... CH-1).
        for (int ck = 0; ck < nchunk; ++ck, ++u) {
            // bounded wait; the outcome is made uniform so that every thread leaves together
            if (!__syncthreads_and(mbar_wait(&kbar[u & 1], (u >> 1) & 1, p.status, &abort_flag))) {
                u = nuse;
                break;
            }
            const T *kb = kbuf + (size_t)(u & 1) * krows * D;
            const int r0 = ck * krows, nr = min(krows, p.N - r0);
            for (int jl0 = warp * RPW; jl0 < nr; jl0 += kCWarps * RPW) {
                const int jl = jl0 + rsub;
                float kv[E];
                if (lane_used && jl < nr) {
                    load_chunk<T>(kb + (int64_t)jl * D + c * E, kv);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) kv[e] = 0.f;
                }
#pragma unroll
                for (int g = 0; g < kQReg; ++g) {
                    float part = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) part = fmaf(qr[g][e], kv[e], part);
                    float tot;
                    if constexpr ((CH & (CH - 1)) == 0) {
                        tot = part;
#pragma unroll
                        for (int off = CH / 2; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
                    } else {
                        const int base = rsub * CH;
                        tot = __shfl_sync(0xffffffffu, part, base & 31);
#pragma unroll
                        for (int cc = 1; cc < CH; ++cc) tot += __shfl_sync(0xffffffffu, part, (base + cc) & 31);
                    }
                    if (g < gn && lane_used && c == 0 && jl < nr) s[g * p.N + r0 + jl] = tot;
                }
            }
            __syncthreads();  // buffer u & 1 consumed
            if (tid == 0 && u + 2 < nuse && !abort_flag) stage(u + 2);
        }
        // per generating query (one warp each): max (of the unscaled dot products: the scale
        // is positive), then the double-float sum of the exponentials (lane-strided in key
        // order, then a butterfly over the lanes)
        for (int g = warp; g < gn; g += kCWarps) {
            const float *sg = s + g * p.N;
            float mx = -INFINITY;
            for (int j = lane; j < p.N; j += 32) mx = fmaxf(mx, sg[j]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            float hi = 0.f, lo = 0.f;
            for (int j = lane; j < p.N; j += 32) df_add(hi, lo, exp_scaled_diff(sg[j], mx, p.scale));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float h2 = __shfl_xor_sync(0xffffffffu, hi, off), l2 = __shfl_xor_sync(0xffffffffu, lo, off);
                df_merge(hi, lo, h2, l2);
            }
            if (lane == 0) {
                stat[g][0] = mx;
                stat[g][1] = __frcp_rn(hi + lo);
            }
        }
        __syncthreads();
        for (int j = tid; j < p.N; j += kCThreads) {
            float hi = acc_hi[j], lo = acc_lo[j];
            for (int g = 0; g < gn; ++g)
                if (valid[g]) df_add(hi, lo, exp_scaled_diff(s[g * p.N + j], stat[g][0], p.scale) * stat[g][1]);
            acc_hi[j] = hi;
            acc_lo[j] = lo;
        }
        __syncthreads();  // valid / stat / s reused by the next pass
    }
    // every head's accumulator is complete: CTA h sums its slice of the keys over the
    // heads (distributed shared memory, h in order)
    cluster.sync();
    const int per = (p.N + p.H - 1) / p.H;
    const int j_lo = h * per, j_hi = min(p.N, j_lo + per);
    const float hg = (float)p.H * (float)p.G;
    for (int j = j_lo + tid; j < j_hi; j += kCThreads) {
        // remote loads in batches of 8 (issued together), merged in head order
        float hi = 0.f, lo = 0.f;
        for (int h0 = 0; h0 < p.H; h0 += 8) {
            float his[8], los[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                his[k] = los[k] = 0.f;
                if (h0 + k < p.H) {
                    his[k] = cluster.map_shared_rank(acc_hi, h0 + k)[j];
                    los[k] = cluster.map_shared_rank(acc_lo, h0 + k)[j];
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (h0 + k < p.H) df_merge(hi, lo, his[k], los[k]);
        }
        p.score[(int64_t)b * p.N + j] = __fdiv_rn(hi + lo, hg);
    }
    cluster.sync();  // no CTA leaves while another reads its accumulator
}

template <typename T, int D>
cudaError_t launch_cluster(const ScoreParams &p, cudaStream_t s) {
    static int configured[64] = {0};
    const int krows = cluster_rows(p.N, D * (int)sizeof(T));
    const size_t smem = cluster_smem_bytes(p.N, D, (int)sizeof(T));
    cudaError_t e = ensure_smem(score_cluster_kernel<T, D>, smem, configured);
    if (e != cudaSuccess) return e;
    if (p.H > 8) {
        e = cudaFuncSetAttribute(score_cluster_kernel<T, D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.H, (unsigned)p.B, 1);
    cfg.blockDim = dim3(kCThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.H;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, score_cluster_kernel<T, D>, p, krows);
}

template <typename T>
cudaError_t launch_cluster_d(const ScoreParams &p, cudaStream_t s) {
    switch (p.d) {
        case 32: return launch_cluster<T, 32>(p, s);
        case 64: return launch_cluster<T, 64>(p, s);
        case 80: return launch_cluster<T, 80>(p, s);
        case 128: return launch_cluster<T, 128>(p, s);
        default: return cudaErrorInvalidValue;
    }
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

// Grid (batch row b, chunk of 32 keys), 128 threads: one score group per warp, one key
// per thread; the groups' sums are merged in group order (see gen_rows.cuh). Chunks of 64
// keys (256 threads) measured 2 us slower per call at the MAR-H shape.
constexpr int kRKeys = 32, kRThreads = kRKeys * kScoreGroups;

__global__ void __launch_bounds__(kRThreads) score_rows_kernel(const float *__restrict__ gen_s,
                                                               const float2 *__restrict__ gen_ml,
                                                               const int32_t *__restrict__ gen,
                                                               float *__restrict__ score, int H, int G, int N,
                                                               float sl2, float sl2_lo) {
    extern __shared__ RowStat rstat[];  // [H * G]
    __shared__ float part[2][kScoreGroups][kRKeys];
    const int b = blockIdx.x, rows = H * G, tid = threadIdx.x;
    load_row_stats(rstat, gen_ml, gen, b, H, G, N, tid, kRThreads);
    __syncthreads();
    const int q = tid / kRKeys, kk = tid % kRKeys, j = blockIdx.y * kRKeys + kk;
    float hi = 0.f, lo = 0.f;
    if (j < N) score_group_sum<8>(gen_s + (int64_t)b * rows * N + j, rstat, rows, q, N, sl2, sl2_lo, hi, lo);
    part[0][q][kk] = hi;
    part[1][q][kk] = lo;
    __syncthreads();
    if (q == 0 && j < N) {
        for (int u = 1; u < kScoreGroups; ++u) df_merge(hi, lo, part[0][u][kk], part[1][u][kk]);
        score[(int64_t)b * N + j] = __fdiv_rn(hi + lo, (float)rows);
    }
}

}  // namespace

cudaError_t launch_score_rows(const float *gen_s, const float2 *gen_ml, const int32_t *gen, float *score, int B,
                              int H, int G, int N, float scale, cudaStream_t s) {
    const size_t smem = sizeof(RowStat) * (size_t)H * G;
    if (smem > 40 * 1024 || B <= 0) return B <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    // scale * log2(e) as an fp32 pair (hi, lo), formed in double
    const double c = (double)scale * 1.4426950408889634;
    const float c_hi = (float)c, c_lo = (float)(c - (double)c_hi);
    score_rows_kernel<<<dim3(B, (N + kRKeys - 1) / kRKeys), kRThreads, smem, s>>>(
        gen_s, gen_ml, gen, score, H, G, N, c_hi, c_lo);
    return cudaGetLastError();
}

size_t score_smem_bytes(int N, int d) {
    return sizeof(double) * N + sizeof(float) * (GCH * N + GCH * d + 2 * GCH);
}

cudaError_t launch_score(const ScoreParams &p, cudaStream_t s) {
    if (p.H >= 1 && !score_uses_partials(p.H))
        return p.bf16 ? launch_cluster_d<bf16>(p, s) : launch_cluster_d<float>(p, s);
    cudaError_t e = p.bf16 ? launch_partial_d<bf16>(p, s) : launch_partial_d<float>(p, s);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + 255) / 256, p.B);
    score_reduce_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mar
