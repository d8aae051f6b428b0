// Device-side helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "marattn.h"

#define MAR_DEVINL __device__ __forceinline__

namespace mar {

using bf16 = __nv_bfloat16;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- status word
MAR_DEVINL void report(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------- element conversion
template <typename T> MAR_DEVINL float to_f32(T x);
template <> MAR_DEVINL float to_f32<float>(float x) { return x; }
template <> MAR_DEVINL float to_f32<bf16>(bf16 x) { return __bfloat162float(x); }

MAR_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---------------------------------------------------------------- cp.async (16 B)
MAR_DEVINL uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Copies 16 bytes global -> shared; src_bytes < 16 zero-fills the remainder.
MAR_DEVINL void cp_async16(void *smem_dst, const void *gmem_src, int src_bytes = 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(src_bytes));
}
MAR_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> MAR_DEVINL void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---------------------------------------------------------------- ldmatrix / mma.sync
MAR_DEVINL void ldmatrix_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                            const void *smem_row_ptr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(smem_row_ptr)));
}
MAR_DEVINL void ldmatrix_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                  const void *smem_row_ptr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(smem_row_ptr)));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
MAR_DEVINL void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Hardware base-2 exponential (PTX ex2.approx); ex2(-inf) = +0.
MAR_DEVINL float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- packed fp32 pairs (sm_100+)
// Two fp32 values in one 64-bit register pair; one instruction operates on both.
using f32x2 = unsigned long long;
MAR_DEVINL f32x2 f2_pack(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
MAR_DEVINL void f2_unpack(f32x2 r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(r));
}
MAR_DEVINL f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
MAR_DEVINL f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// max of three (sm_100+ three-input form)
MAR_DEVINL float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ---------------------------------------------------------------- double-float sums
// (hi, lo) += x with the error-free two-sum, so that a sum of fp32 terms keeps about 48
// bits (fp64-grade for these sums) without the fp64 pipe, which is slow on this part.
// The result is a pure function of the operand sequence (deterministic).
MAR_DEVINL void df_add(float &hi, float &lo, float x) {
    const float s = hi + x;
    const float bb = s - hi;
    const float err = (hi - (s - bb)) + (x - bb);
    hi = s;
    lo += err;
}
// (hi, lo) += (hi2, lo2); symmetric in its operands (both sides of a butterfly agree)
MAR_DEVINL void df_merge(float &hi, float &lo, float hi2, float lo2) {
    const float s = hi + hi2;
    const float bb = s - hi;
    const float err = (hi - (s - bb)) + (hi2 - bb);
    hi = s;
    lo = (lo + lo2) + err;
}

// ---------------------------------------------------------------- exponentials of large arguments
// A softmax weight is an exponential of a difference of logits. Evaluated as exp(fl(arg)),
// its relative error is |arg| * 2^-24 from the rounding of the argument alone: 3e-6 at an
// argument of 50, which the layer-2 score's 1e-6 bound does not allow for peaked rows.
// These forms carry the argument as an unevaluated fp32 pair (a two-sum for the
// difference, the FMA residual for the product) and apply the low part as a first-order
// correction, leaving the exponential's own error (a few ulp) and O(2^-48) terms.

// exp(scale * (a - b)), scale > 0 (the natural-base form of the separate score kernel)
MAR_DEVINL float exp_scaled_diff(float a, float b, float scale) {
    const float d = a - b;
    const float bb = d - a;
    const float de = (a - (d - bb)) + (-b - bb);      // a - b == d + de exactly
    const float y = d * scale;
    const float ye = fmaf(d, scale, -y) + de * scale;  // d * scale == y + residual exactly
    const float e = expf(y);
    return fmaf(e, ye, e);
}

// 2^(s * (c_hi + c_lo) - m) with c_hi + c_lo = scale * log2(e) to about 2^-48 (the base-2
// form of the raw-score reduction)
MAR_DEVINL float exp2_fma_acc(float s, float c_hi, float c_lo, float m) {
    const float th = s * c_hi;
    const float tl = fmaf(s, c_hi, -th);               // s * c_hi == th + tl exactly
    const float u = th - m;
    const float bb = u - th;
    const float ue = (th - (u - bb)) + (-m - bb);      // th - m == u + ue exactly
    const float c = ue + fmaf(s, c_lo, tl);
    const float e = fast_exp2(u);
    return fmaf(e, c * kLn2, e);
}

// ---------------------------------------------------------------- active/cached partition
// Builds, in shared memory, the ascending list of positions of one batch row that are
// NOT in idx[0..A) (the cached set), using a bitmap of N bits. All threads of the
// block must call it. Returns the cached count C. Reports out-of-range and repeated
// positions through `status`; such entries are ignored.
// bitmap: ceil(N/32) words; cached: N ints; warp_tot: blockDim/32 ints.
MAR_DEVINL int build_cached_list(const int32_t *__restrict__ idx, int A, int N,
                                 uint32_t *bitmap, int32_t *cached, int32_t *warp_tot,
                                 uint32_t *status) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int words = (N + 31) >> 5;
    for (int w = tid; w < words; w += nthr) bitmap[w] = 0u;
    __syncthreads();
    uint32_t bad = 0;
    for (int a = tid; a < A; a += nthr) {
        int p = idx[a];
        if (p < 0 || p >= N) {
            bad |= MAR_STATUS_INDEX_RANGE;
            continue;
        }
        uint32_t old = atomicOr(&bitmap[p >> 5], 1u << (p & 31));
        if (old & (1u << (p & 31))) bad |= MAR_STATUS_INDEX_DUP;
    }
    if (bad) report(status, bad);
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5, nwarp = nthr >> 5;
    int base = 0;
    for (int p0 = 0; p0 < N; p0 += nthr) {
        int p = p0 + tid;
        bool is_cached = (p < N) && !((bitmap[p >> 5] >> (p & 31)) & 1u);
        uint32_t ball = __ballot_sync(0xffffffffu, is_cached);
        int within = __popc(ball & ((1u << lane) - 1u));
        if (lane == 0) warp_tot[warp] = __popc(ball);
        __syncthreads();
        int off = base;
        for (int w = 0; w < warp; ++w) off += warp_tot[w];
        if (is_cached) cached[off + within] = p;
        int tot = 0;
        for (int w = 0; w < nwarp; ++w) tot += warp_tot[w];
        base += tot;
        __syncthreads();
    }
    return base;
}

// Raises the dynamic shared memory limit of `func` to `bytes` once per device. With
// max_carveout the kernel also asks for the largest shared-memory carveout of the SM, so
// that as many CTAs as the shared memory allows can be resident (the default carveout
// can be one step too small for two ~100 KB CTAs).
template <typename F>
inline cudaError_t ensure_smem(F *func, size_t bytes, int *configured /* [64] */, bool max_carveout = false) {
    if (bytes <= 48 * 1024 && !max_carveout) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && configured[dev] >= (int)bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && dev < 64) configured[dev] = (int)bytes;
    return e;
}

}  // namespace mar
