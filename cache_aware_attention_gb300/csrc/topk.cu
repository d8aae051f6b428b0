// Top-K refresh selection and active-set assembly.
//
// MARché notes, Key Design 1: the K tokens with the highest layer-2 relevance score
// become the refreshing tokens; with the generating and just-decoded (caching) tokens
// they form the active set. Candidates exclude the generating and just-decoded tokens.
//
// Scores map to 32-bit keys that order like the floats (sign-magnitude flip), so the
// selection is exact on the fp32 values: the K candidates first in the order (key desc,
// position asc). Rows of up to 1152 scores: one warp per row (topk_warp_kernel below).
// Longer rows: one CTA per row and a 4-pass MSB-first radix select over the keys, which
// finds the K-th largest value T and how many candidates equal to T are taken (the lowest
// positions first); selected positions are written in ascending order by a block-wide
// prefix sum, so the result is deterministic. (The CTA form also keeps a rank-counting
// pass for rows up to kRankN, used when the warp form does not apply.)
#include "common.cuh"
#include "score.h"

namespace mar {
namespace {

constexpr int kThreads = 512;
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
    // pairs: rows b (conditional) and b + B (unconditional) share the selection, made on
    // the fp32 sum of their scores with row b's exclusions
    const int b2 = b + p.B;
    for (int j = tid; j < N; j += kThreads) {
        const float sc = p.pairs ? __fadd_rn(p.score[(int64_t)b * N + j], p.score[(int64_t)b2 * N + j])
                                 : p.score[(int64_t)b * N + j];
        keys[j] = order_key(sc);
        cand[j] = 1;
    }
    __syncthreads();
    for (int e = tid; e < p.E; e += kThreads) {
        int pos = p.exclude[(int64_t)b * p.E + e];
        if (p.active) {
            p.active[(int64_t)b * (p.E + p.K) + e] = pos;  // copied as given
            if (p.pairs) p.active[(int64_t)b2 * (p.E + p.K) + e] = p.exclude[(int64_t)b2 * p.E + e];
        }
        if (pos < 0 || pos >= N) {
            report(p.status, MAR_STATUS_INDEX_RANGE);
            continue;
        }
        cand[pos] = 0;
    }
    auto emit = [&](int slot, int j) {
        if (p.out) p.out[(int64_t)b * p.K + slot] = j;
        if (p.active) p.active[(int64_t)b * (p.E + p.K) + p.E + slot] = j;
        if (p.pairs) {
            if (p.out) p.out[(int64_t)b2 * p.K + slot] = j;
            if (p.active) p.active[(int64_t)b2 * (p.E + p.K) + p.E + slot] = j;
        }
    };
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
            if (sel && slot < p.K) emit(slot, j);
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
        if (sel && slot < p.K) emit(slot, j);
    }
}

// Warp-level form for rows of at most kWarpN scores: one warp per batch row, the row's keys
// in registers (lane l holds positions l, l + 32, ...). An MSB-first radix select over the
// 32 key bits finds the K-th largest key T among the candidates: at each bit the warp
// counts the candidates that match the prefix chosen so far with that bit set (a per-lane
// count, then a butterfly sum) and keeps the bit if at least the remaining number of
// picks does. The candidates above T are taken, and of those equal to T the `take` lowest
// positions; positions are written in ascending order by ballot prefix counts. Exactly
// the selection of the block form.
constexpr int kWarpN = 1152;
constexpr int kWarpsPerCta = 4;

template <int kWarpNPL>  // keys per lane: rows of up to 32 * kWarpNPL scores
__global__ void __launch_bounds__(32 * kWarpsPerCta) topk_warp_kernel(TopkParams p) {
    __shared__ uint32_t excl_bits[kWarpsPerCta][kWarpN / 32];
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const int b = blockIdx.x * kWarpsPerCta + wi;
    if (b >= p.B) return;  // whole warps leave together
    const int N = p.N, b2 = b + p.B;
    uint32_t *ex = excl_bits[wi];
    for (int w = lane; w < (N + 31) / 32; w += 32) ex[w] = 0u;
    __syncwarp();
    for (int e = lane; e < p.E; e += 32) {
        const int pos = p.exclude[(int64_t)b * p.E + e];
        if (p.active) {
            p.active[(int64_t)b * (p.E + p.K) + e] = pos;  // copied as given
            if (p.pairs) p.active[(int64_t)b2 * (p.E + p.K) + e] = p.exclude[(int64_t)b2 * p.E + e];
        }
        if (pos < 0 || pos >= N) {
            report(p.status, MAR_STATUS_INDEX_RANGE);
            continue;
        }
        atomicOr(&ex[pos >> 5], 1u << (pos & 31));
    }
    __syncwarp();
    if (p.K == 0) return;
    uint32_t key[kWarpNPL];
    uint64_t cand = 0;  // bit i: position lane + 32 i is a candidate
#pragma unroll
    for (int i = 0; i < kWarpNPL; ++i) {
        const int j = lane + 32 * i;
        key[i] = 0u;
        if (j < N) {
            const float sc = p.pairs ? __fadd_rn(p.score[(int64_t)b * N + j], p.score[(int64_t)b2 * N + j])
                                     : p.score[(int64_t)b * N + j];
            key[i] = order_key(sc);
            if (!((ex[i] >> lane) & 1u)) cand |= 1ull << i;
        }
    }
    // radix select: T = the K-th largest candidate key, `take` = how many keys equal to T
    uint32_t T = 0u;
    int take = p.K;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t want = T | (1u << bit);
        const int sh = bit;  // compare the bits at and above `bit`
        int c = 0;
#pragma unroll
        for (int i = 0; i < kWarpNPL; ++i)
            c += (((cand >> i) & 1ull) && (key[i] >> sh) == (want >> sh)) ? 1 : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
        if (c >= take) T = want;
        else take -= c;
    }
    // ascending positions: the candidates above T, and the first `take` equal to T
    const uint32_t lt = (1u << lane) - 1u;
    int base = 0, eq_base = 0;
    auto emit = [&](int slot, int j) {
        if (p.out) p.out[(int64_t)b * p.K + slot] = j;
        if (p.active) p.active[(int64_t)b * (p.E + p.K) + p.E + slot] = j;
        if (p.pairs) {
            if (p.out) p.out[(int64_t)b2 * p.K + slot] = j;
            if (p.active) p.active[(int64_t)b2 * (p.E + p.K) + p.E + slot] = j;
        }
    };
#pragma unroll
    for (int i = 0; i < kWarpNPL; ++i) {
        if (32 * i >= N) break;  // warp-uniform
        const bool c = (cand >> i) & 1ull;
        const bool eq = c && key[i] == T;
        const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
        const bool sel = c && (key[i] > T || (eq && eq_base + __popc(eqm & lt) < take));
        eq_base += __popc(eqm);
        const uint32_t selm = __ballot_sync(0xffffffffu, sel);
        if (sel) {
            const int slot = base + __popc(selm & lt);
            if (slot < p.K) emit(slot, lane + 32 * i);
        }
        base += __popc(selm);
    }
}

constexpr int kSelectMaxN = 16384;

// Token-cache recompute set (LazyMAR notes, Token Cache): one CTA per row; position j is
// recomputed when it is forced or not (cos > tau) (a NaN similarity is recomputed). The
// positions are written in ascending order by a block-wide prefix sum, the remaining
// slots get -1.
__global__ void __launch_bounds__(kThreads) select_recompute_kernel(SelectParams p) {
    __shared__ uint32_t forced[kSelectMaxN / 32];
    __shared__ int warp_sums[kThreads / 32];
    const int tid = threadIdx.x, b = blockIdx.x, N = p.N;
    const int words = (N + 31) >> 5;
    for (int w = tid; w < words; w += kThreads) forced[w] = 0u;
    __syncthreads();
    for (int f = tid; f < p.F; f += kThreads) {
        const int pos = p.force[(int64_t)b * p.F + f];
        if (pos < 0 || pos >= N) {
            report(p.status, MAR_STATUS_INDEX_RANGE);
            continue;
        }
        atomicOr(&forced[pos >> 5], 1u << (pos & 31));
    }
    __syncthreads();
    int base = 0;
    for (int j0 = 0; j0 < N; j0 += kThreads) {
        const int j = j0 + tid;
        bool sel = false;
        if (j < N) sel = ((forced[j >> 5] >> (j & 31)) & 1u) || !(p.cos[(int64_t)b * N + j] > p.tau);
        int tot;
        const int slot = base + block_excl_scan(sel ? 1 : 0, warp_sums, &tot);
        base += tot;
        if (sel) p.out[(int64_t)b * N + slot] = j;
    }
    for (int j = base + tid; j < N; j += kThreads) p.out[(int64_t)b * N + j] = -1;
    if (tid == 0) p.count[b] = base;
}

}  // namespace

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s) {
    if (p.N > kMaxN) return cudaErrorInvalidValue;
    if (p.B == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((p.B + kWarpsPerCta - 1) / kWarpsPerCta);
    if (p.N <= 320)
        topk_warp_kernel<10><<<grid, 32 * kWarpsPerCta, 0, s>>>(p);
    else if (p.N <= 640)
        topk_warp_kernel<20><<<grid, 32 * kWarpsPerCta, 0, s>>>(p);
    else if (p.N <= kWarpN)
        topk_warp_kernel<kWarpN / 32><<<grid, 32 * kWarpsPerCta, 0, s>>>(p);
    else
        topk_kernel<<<p.B, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mar

namespace mar {

cudaError_t launch_select_recompute(const SelectParams &p, cudaStream_t s) {
    if (p.N > kSelectMaxN) return cudaErrorInvalidValue;
    if (p.B == 0 || p.N == 0) return cudaSuccess;
    select_recompute_kernel<<<p.B, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mar
