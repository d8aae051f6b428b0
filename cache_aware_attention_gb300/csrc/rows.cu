// Row movement for the KV cache and the LazyMAR condition cache.
//
// MARché notes, Key Design 2: active tokens carry freshly projected K/V that replace
// their stored rows in the per-layer cache (scatter), and the active rows of a full
// tensor are pulled into a dense block (gather); Key Design 3: a full-refresh step
// overwrites every row. All of these are bit copies in 16-byte vectors.
// LazyMAR notes, Condition Cache: uncond = cond - residual on cached steps, residual =
// cond - uncond on full steps (elementwise fp32).
#include "common.cuh"
#include "score.h"

namespace mar {
namespace {

constexpr int kThreads = 256;

// blockIdx.x and the thread index cover one batch row's (tensor, row, chunk) 16-byte
// vectors, neighbouring threads moving neighbouring chunks of a row; blockIdx.y steps over
// the batch rows. A thread reads its row's position once and copies that chunk for every
// head, the head loop unrolled so that its loads are in flight together. 32-bit index
// arithmetic only.
__global__ void __launch_bounds__(kThreads) rows_kernel(RowCopyParams p) {
    const int vec = p.row_bytes >> 4;
    const int av = p.A * vec;
    const int i = (int)blockIdx.x * kThreads + (int)threadIdx.x;
    if (i >= av * p.n_tensors) return;
    const int tensor = i / av;
    const int r = i - tensor * av;
    const int a = r / vec, c = r - a * vec;
    const char *src_base = static_cast<const char *>(p.src[tensor]);
    char *dst_base = static_cast<char *>(p.dst[tensor]);
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        int pos = a;
        if (p.idx) {
            pos = p.idx[(int64_t)b * p.A + a];
            if (pos < 0 || pos >= p.N) {
                // -1 pads a row of positions (as the recompute set is written); anything
                // else outside [0, N) is an error
                if (pos != -1 && tensor == 0 && c == 0) report(p.status, MAR_STATUS_INDEX_RANGE);
                continue;
            }
        }
        const int64_t bh0 = (int64_t)b * p.H;
        const int64_t dense0 = bh0 * p.A + a, full0 = bh0 * p.N + pos;
        const int64_t src0 = p.scatter ? dense0 : full0, dst0 = p.scatter ? full0 : dense0;
        const int64_t src_step = (int64_t)(p.scatter ? p.A : p.N) * p.row_bytes;
        const int64_t dst_step = (int64_t)(p.scatter ? p.N : p.A) * p.row_bytes;
        const char *sp = src_base + src0 * p.row_bytes + 16 * c;
        char *dp = dst_base + dst0 * p.row_bytes + 16 * c;
#pragma unroll 4
        for (int h = 0; h < p.H; ++h) {
            const uint4 v = *reinterpret_cast<const uint4 *>(sp + h * src_step);
            *reinterpret_cast<uint4 *>(dp + h * dst_step) = v;
        }
    }
}

__global__ void __launch_bounds__(kThreads) cfg_kernel(int mode, int64_t n, const float *__restrict__ cond,
                                                       float *uncond, float *residual, float w,
                                                       float *guided) {
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
        const float c = cond[i];
        float u;
        if (mode == MAR_CFG_APPLY) {
            u = __fsub_rn(c, residual[i]);
            uncond[i] = u;
        } else {
            u = uncond[i];
            residual[i] = __fsub_rn(c, u);
        }
        if (guided) guided[i] = __fadd_rn(u, __fmul_rn(w, __fsub_rn(c, u)));
    }
}

MAR_DEVINL float guide1(float u, float c, float w) { return __fadd_rn(u, __fmul_rn(w, __fsub_rn(c, u))); }

__global__ void __launch_bounds__(kThreads) cfg_kernel_v4(int mode, int64_t n4, const float4 *__restrict__ cond,
                                                          float4 *uncond, float4 *residual, float w,
                                                          float4 *guided) {
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n4; i += (int64_t)gridDim.x * kThreads) {
        const float4 c = cond[i];
        float4 u;
        if (mode == MAR_CFG_APPLY) {
            const float4 r = residual[i];
            u = make_float4(__fsub_rn(c.x, r.x), __fsub_rn(c.y, r.y), __fsub_rn(c.z, r.z), __fsub_rn(c.w, r.w));
            uncond[i] = u;
        } else {
            u = uncond[i];
            residual[i] = make_float4(__fsub_rn(c.x, u.x), __fsub_rn(c.y, u.y), __fsub_rn(c.z, u.z),
                                      __fsub_rn(c.w, u.w));
        }
        if (guided)
            guided[i] = make_float4(guide1(u.x, c.x, w), guide1(u.y, c.y, w), guide1(u.z, c.z, w),
                                    guide1(u.w, c.w, w));
    }
}

int grid_for(int64_t work) {
    int64_t blocks = (work + kThreads - 1) / kThreads;
    const int64_t cap = 152 * 16;  // a few resident waves over the 152 SMs; grid-stride beyond
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

cudaError_t launch_rows(const RowCopyParams &p, cudaStream_t s) {
    const int64_t per_bh = (int64_t)p.A * (p.row_bytes / 16) * p.n_tensors;
    if (per_bh == 0 || p.B == 0 || p.H == 0) return cudaSuccess;
    if (per_bh > 0x7fffffffLL - kThreads) return cudaErrorInvalidValue;
    const unsigned gx = (unsigned)((per_bh + kThreads - 1) / kThreads);
    const unsigned gy = (unsigned)(p.B < 65535 ? p.B : 65535);
    rows_kernel<<<dim3(gx, gy), kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cfg(int mode, int64_t n, const float *cond, float *uncond, float *residual, float w,
                       float *guided, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const bool v4 = (n % 4 == 0) && ((reinterpret_cast<uintptr_t>(cond) | reinterpret_cast<uintptr_t>(uncond) |
                                      reinterpret_cast<uintptr_t>(residual) |
                                      reinterpret_cast<uintptr_t>(guided)) % 16 == 0);
    if (v4) {
        cfg_kernel_v4<<<grid_for(n / 4), kThreads, 0, s>>>(
            mode, n / 4, reinterpret_cast<const float4 *>(cond), reinterpret_cast<float4 *>(uncond),
            reinterpret_cast<float4 *>(residual), w, reinterpret_cast<float4 *>(guided));
    } else {
        cfg_kernel<<<grid_for(n), kThreads, 0, s>>>(mode, n, cond, uncond, residual, w, guided);
    }
    return cudaGetLastError();
}

}  // namespace mar
