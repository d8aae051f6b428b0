// Top-K refresh selection and active-set assembly.
//
// MARché notes, Key Design 1: the K tokens with the highest layer-2 relevance score
// become the refreshing tokens; with the generating and just-decoded (caching) tokens
// they form the active set. Candidates exclude the generating and just-decoded tokens.
//
// One CTA per batch row. Scores map to 32-bit keys that order like the floats
// (sign-magnitude flip), so the selection is exact on the fp32 values. A candidate j is
// selected when fewer than K candidates precede it in the order (key desc, position
// asc). For N <= kRankN each thread counts that rank directly against all candidates
// in shared memory (one pass, broadcast reads). Larger rows use a 4-pass MSB-first radix
// select over the keys, which finds the K-th largest value T and how many candidates
// equal to T are taken (the lowest positions first). Selected positions are written in
// ascending order by a block-wide prefix sum, so the result is deterministic.
#include "common.cuh"
#include "score.h"

namespace mar {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxN = 4096;
constexpr int kRankN = 1152;

MAR_DEVINL uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of `v` over the block in thread order; the block total is
// returned through *total. All threads must call it.
MAR_DEVINL int block_excl_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < nw; ++w) {
        int ws = warp_sums[w];
        if (w < warp) before += ws;
        tot += ws;
    }
    __syncthreads();
    *total = tot;
    return before + x - v;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkParams p) {
    __shared__ uint32_t keys[kMaxN];
    __shared__ unsigned char cand[kMaxN];
    __shared__ uint64_t wide[kRankN];
    __shared__ int hist[256];
    __shared__ int warp_sums[kThreads / 32];
    __shared__ uint32_t sel_prefix;
    __shared__ int sel_remaining;

    const int tid = threadIdx.x, b = blockIdx.x;
    const int N = p.N;
    for (int j = tid; j < N; j += kThreads) {
        keys[j] = order_key(p.score[(int64_t)b * N + j]);
        cand[j] = 1;
    }
    __syncthreads();
    for (int e = tid; e < p.E; e += kThreads) {
        int pos = p.exclude[(int64_t)b * p.E + e];
        if (p.active) p.active[(int64_t)b * (p.E + p.K) + e] = pos;  // copied as given
        if (pos < 0 || pos >= N) {
            report(p.status, MAR_STATUS_INDEX_RANGE);
            continue;
        }
        cand[pos] = 0;
    }
    if (p.K == 0) return;
    if (N <= kRankN) {
        // rank = number of candidates before j in (key desc, position asc) order; one
        // 64-bit compare per candidate (non-candidates map to 0 and never precede).
        __syncthreads();  // exclusion flags written above
        for (int j = tid; j < N; j += kThreads)
            wide[j] = cand[j] ? (((uint64_t)keys[j] << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)j)) : 0ull;
        __syncthreads();
        int base = 0;
        for (int j0 = 0; j0 < N; j0 += kThreads) {
            const int j = j0 + tid;
            bool sel = false;
            if (j < N && cand[j]) {
                const uint64_t kj = wide[j];
                int rank = 0;
                for (int i = 0; i < N; ++i) rank += (wide[i] > kj) ? 1 : 0;
                sel = rank < p.K;
            }
            int tot;
            const int slot = base + block_excl_scan(sel ? 1 : 0, warp_sums, &tot);
            base += tot;
            if (sel && slot < p.K) {
                if (p.out) p.out[(int64_t)b * p.K + slot] = j;
                if (p.active) p.active[(int64_t)b * (p.E + p.K) + p.E + slot] = j;
            }
        }
        return;
    }
    if (tid == 0) {
        sel_prefix = 0u;
        sel_remaining = p.K;
    }
    __syncthreads();

    // radix select of the K-th largest key among candidates
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = sel_prefix;
        for (int j = tid; j < N; j += kThreads)
            if (cand[j] && (keys[j] & mask) == prefix) atomicAdd(&hist[(keys[j] >> shift) & 255u], 1);
        __syncthreads();
        if (tid == 0) {
            int rem = sel_remaining, bin = 255;
            for (; bin > 0; --bin) {
                if (hist[bin] >= rem) break;
                rem -= hist[bin];
            }
            sel_prefix = prefix | ((uint32_t)bin << shift);
            sel_remaining = rem;
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t T = sel_prefix;
    const int take = sel_remaining;  // candidates equal to T to select, lowest positions first

    // rank of equal-to-T candidates by position, then selection flags and output slots
    int eq_base = 0, out_base = 0;
    for (int j0 = 0; j0 < N; j0 += kThreads) {
        const int j = j0 + tid;
        const bool c = (j < N) && cand[j];
        const bool eq = c && keys[j] == T;
        int tot;
        const int eq_rank = eq_base + block_excl_scan(eq ? 1 : 0, warp_sums, &tot);
        eq_base += tot;
        const bool sel = c && (keys[j] > T || (eq && eq_rank < take));
        const int slot = out_base + block_excl_scan(sel ? 1 : 0, warp_sums, &tot);
        out_base += tot;
        if (sel && slot < p.K) {
            if (p.out) p.out[(int64_t)b * p.K + slot] = j;
            if (p.active) p.active[(int64_t)b * (p.E + p.K) + p.E + slot] = j;
        }
    }
}

}  // namespace

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s) {
    if (p.N > kMaxN) return cudaErrorInvalidValue;
    topk_kernel<<<p.B, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mar
