// Layer-2 score from the generating rows the attention launch left behind (raw scores and
// the (m, l) of each row's online softmax), as the reduction kernel computes it.
//
// The score of key j is (1/(H G)) sum over rows r = h * G + g of 2^(s_rj * sl2 - m_r) / l_r
// (sl2 = scale * log2(e) as an fp32 pair, the exponent argument carried to fp64-grade
// accuracy by exp2_fma_acc), summed in a fixed order: the rows are cut into kScoreGroups
// consecutive groups; a group is summed in row order with two double-float accumulators
// taking alternate rows (counted from the group's first row), merged at the end; the groups
// are merged in group order.
#pragma once

#include "common.cuh"

namespace mar {

constexpr int kScoreGroups = 4;

struct RowStat {
    float m, rl;  // max, 1 / l; rl == 0: no row (a generating position out of range)
    int src;      // row of gen_s holding the slot's scores (a repeated position: its first slot)
    int pad;
};

// rstat[r] for the rows r of batch row b, by threads tid, tid + nthr, ...
MAR_DEVINL void load_row_stats(RowStat *rstat, const float2 *gen_ml, const int32_t *gen, int b, int H, int G,
                               int N, int tid, int nthr) {
    const int rows = H * G;
    const int32_t *gb = gen + (int64_t)b * G;
    for (int r = tid; r < rows; r += nthr) {
        const int g = r % G, pos = gb[g];
        RowStat st{0.f, 0.f, 0, 0};
        if ((unsigned)pos < (unsigned)N) {
            int first = g;
            for (int q = g - 1; q >= 0; --q)
                if (gb[q] == pos) first = q;
            st.src = r - g + first;
            const float2 ml = gen_ml[(int64_t)b * rows + st.src];
            st.m = ml.x;
            st.rl = __frcp_rn(ml.y);
        }
        rstat[r] = st;
    }
}

MAR_DEVINL int score_group_rows(int rows) { return (rows + kScoreGroups - 1) / kScoreGroups; }

// (hi, lo) of group q for the key whose column of gen_s (batch row b) starts at sj, with
// kBatch (even) loads in flight; the sums do not depend on kBatch.
template <int kBatch>
MAR_DEVINL void score_group_sum(const float *__restrict__ sj, const RowStat *rstat, int rows, int q, int N,
                                float sl2, float sl2_lo, float &hi, float &lo) {
    static_assert(kBatch % 2 == 0, "alternate rows must keep their accumulator across batches");
    const int per = score_group_rows(rows);
    const int r_lo = q * per, r_hi = min(rows, r_lo + per);
    float h0 = 0.f, l0 = 0.f, h1 = 0.f, l1 = 0.f;
    for (int r0 = r_lo; r0 < r_hi; r0 += kBatch) {
        float x[kBatch];
        RowStat st[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            st[k] = r0 + k < r_hi ? rstat[r0 + k] : RowStat{0.f, 0.f, 0, 0};
            x[k] = st[k].rl != 0.f ? sj[(int64_t)st[k].src * N] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kBatch; k += 2) {
            if (st[k].rl != 0.f) df_add(h0, l0, exp2_fma_acc(x[k], sl2, sl2_lo, st[k].m) * st[k].rl);
            if (st[k + 1].rl != 0.f) df_add(h1, l1, exp2_fma_acc(x[k + 1], sl2, sl2_lo, st[k + 1].m) * st[k + 1].rl);
        }
    }
    df_merge(h0, l0, h1, l1);
    hi = h0;
    lo = l0;
}

}  // namespace mar
