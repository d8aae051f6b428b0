// Per-token cosine similarity between two feature tensors of the same layout.
//
// LazyMAR notes, Token Cache: in the deeper layers a token whose current feature is close,
// in cosine similarity, to its cached feature reuses the cached value; only the others are
// recomputed. MARche notes, Figure 1 and Figures 10-11: the same cosine between the key
// (value) projections of consecutive decoding steps shows which tokens drift, the quantity
// behind the choice of caching and refreshing tokens.
//
// Layout [B, H, N, d]: token (b, n) has the H*d values X[b, h, n, :] over all h, and
//   cos(b, n) = <x, y> / (|x| |y|),   both zero -> 1, one zero -> 0.
// One warp per token. Lane l takes the 16-byte chunks t = l, l + 32, ... of the token
// (chunk t = head t / CH, columns (t % CH) * E ..); a chunk's products accumulate in fp32 in
// element order and the chunk sums are added as fp32 pairs (error-free two-sums), then
// combined across the lanes in a fixed butterfly: the three sums are fp64-grade and the
// result is deterministic.
#include "common.cuh"
#include "score.h"

namespace mar {
namespace {

constexpr int kWarpsPerBlock = 8;

template <typename T>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) token_cosine_kernel(const T *__restrict__ X,
                                                                          const T *__restrict__ Y, float *out,
                                                                          int B, int H, int N, int d) {
    constexpr int E = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (tok >= (int64_t)B * N) return;
    const int b = (int)(tok / N), n = (int)(tok - (int64_t)b * N);
    const int CH = d / E;
    float xy_h = 0.f, xy_l = 0.f, xx_h = 0.f, xx_l = 0.f, yy_h = 0.f, yy_l = 0.f;
    for (int t = lane; t < H * CH; t += 32) {
        const int h = t / CH, c = t - h * CH;
        const int64_t off = (((int64_t)b * H + h) * N + n) * d + (int64_t)c * E;
        const uint4 rx = *reinterpret_cast<const uint4 *>(X + off);
        const uint4 ry = *reinterpret_cast<const uint4 *>(Y + off);
        float x[E], y[E];
        if constexpr (sizeof(T) == 2) {
            const __nv_bfloat162 *hx = reinterpret_cast<const __nv_bfloat162 *>(&rx);
            const __nv_bfloat162 *hy = reinterpret_cast<const __nv_bfloat162 *>(&ry);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fx = __bfloat1622float2(hx[e]), fy = __bfloat1622float2(hy[e]);
                x[2 * e] = fx.x; x[2 * e + 1] = fx.y;
                y[2 * e] = fy.x; y[2 * e + 1] = fy.y;
            }
        } else {
            x[0] = __uint_as_float(rx.x); x[1] = __uint_as_float(rx.y);
            x[2] = __uint_as_float(rx.z); x[3] = __uint_as_float(rx.w);
            y[0] = __uint_as_float(ry.x); y[1] = __uint_as_float(ry.y);
            y[2] = __uint_as_float(ry.z); y[3] = __uint_as_float(ry.w);
        }
        float pxy = 0.f, pxx = 0.f, pyy = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            pxy = fmaf(x[e], y[e], pxy);
            pxx = fmaf(x[e], x[e], pxx);
            pyy = fmaf(y[e], y[e], pyy);
        }
        df_add(xy_h, xy_l, pxy);
        df_add(xx_h, xx_l, pxx);
        df_add(yy_h, yy_l, pyy);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float a, c;
        a = __shfl_xor_sync(0xffffffffu, xy_h, off); c = __shfl_xor_sync(0xffffffffu, xy_l, off); df_merge(xy_h, xy_l, a, c);
        a = __shfl_xor_sync(0xffffffffu, xx_h, off); c = __shfl_xor_sync(0xffffffffu, xx_l, off); df_merge(xx_h, xx_l, a, c);
        a = __shfl_xor_sync(0xffffffffu, yy_h, off); c = __shfl_xor_sync(0xffffffffu, yy_l, off); df_merge(yy_h, yy_l, a, c);
    }
    if (lane == 0) {
        const float xy = xy_h + xy_l, xx = xx_h + xx_l, yy = yy_h + yy_l;
        float cs;
        if (xx == 0.f && yy == 0.f) cs = 1.f;
        else if (xx == 0.f || yy == 0.f) cs = 0.f;
        else cs = __fdiv_rn(xy, __fmul_rn(__fsqrt_rn(xx), __fsqrt_rn(yy)));
        out[tok] = cs;
    }
}

}  // namespace

cudaError_t launch_token_cosine(const void *X, const void *Y, float *out, int B, int H, int N, int d, int is_bf16,
                                cudaStream_t s) {
    const int64_t tokens = (int64_t)B * N;
    if (tokens == 0) return cudaSuccess;
    const int64_t blocks = (tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (is_bf16)
        token_cosine_kernel<bf16><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, s>>>(
            static_cast<const bf16 *>(X), static_cast<const bf16 *>(Y), out, B, H, N, d);
    else
        token_cosine_kernel<float><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, s>>>(
            static_cast<const float *>(X), static_cast<const float *>(Y), out, B, H, N, d);
    return cudaGetLastError();
}

}  // namespace mar
