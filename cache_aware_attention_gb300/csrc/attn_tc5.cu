// bf16 attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), d = 64.
//
// Serves full attention (key list = all N rows of K/V) and cache-aware attention
// (key list = the fresh active rows K_A/V_A followed by the cache rows of the cached
// set), see attn.h.
//
// MARché notes, Key Design 2: each active query attends over fresh K_A/V_A and stored
// cached K/V as two partial softmax sums merged by the safe online-softmax rule
// (running max m, running sum l), with no concatenated key buffer in memory. Here the
// key list is streamed in blocks of 128 slots straight from the two sources into
// shared memory: TMA tile loads for contiguous rows (full attention), and TMA gather4
// loads (four rows per instruction) of the active rows and of the cached rows named by
// an in-CTA list built from the active indices (cache rows of active positions are
// never read). Each block updates (m, l, O) of all 128 query rows of the CTA.
//
// CTA = one (b, h) and 128 query rows; 6 warps:
//   warps 0-3  softmax + epilogue; thread t owns query row t (tensor-memory lane t)
//   warp 4     TMA producer (Q once, K/V blocks double-buffered)
//   warp 5     MMA issuer (one lane):  S = Q K^T  (M=128, N=128, K=64, both K-major)
//                                       O = P V   (M=128, N=64, K=128, P from TMEM,
//                                                  V MN-major)
// Tensor memory (256 columns): S at [0,128), overwritten in place by P as packed bf16
// pairs (64 columns), O at [128,192). Per block the softmax threads read S, compute the
// new running max, write P, fold the previous block's O into registers
// (o <- o 2^(m_old - m_new) + O_prev) and hand P to the MMA warp.
// Every wait is bounded (tc5.cuh) and sets a status bit instead of hanging.
#include <cmath>

#include "attn.h"
#include "common.cuh"
#include "tc5.cuh"
#include "tma_host.h"

namespace mar {
namespace {

using namespace tc5;

constexpr int D = 64;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTileBytes = BM * D * 2;  // 16 KB: one 128 x 64 bf16 tile
constexpr size_t kTilesBytes = 5 * kTileBytes;

enum Bar { Q_FULL = 0, KV_FULL = 1, KV_EMPTY = 3, S_FULL = 5, P_FULL = 6, O_FULL = 7, N_BARS = 8 };

struct Tc5Params {
    CUtensorMap mQ;   // 3-D [BH, nq, D], box {64, 128, 1}
    CUtensorMap mKd;  // full: 3-D [BH, n_dense, D] box {64,128,1}; cache-aware: 2-D [BH*A, D] box {64,1}
    CUtensorMap mVd;
    CUtensorMap mKc;  // cache-aware: 2-D [BH*N, D], box {64, 1}
    CUtensorMap mVc;
    AttnParams a;
    int gather;       // 1: cache-aware key list (gather4), 0: full attention (tile loads)
};

MAR_DEVINL uint32_t lane_addr(uint32_t tm, int warp, int col) {
    return tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)col;
}

__global__ void __launch_bounds__(kThreads, 2) attn_tc5_kernel(const __grid_constant__ Tc5Params P) {
    const AttnParams &p = P.a;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    bf16 *sQ = reinterpret_cast<bf16 *>(base);
    bf16 *sK0 = reinterpret_cast<bf16 *>(base + kTileBytes);
    bf16 *sV0 = reinterpret_cast<bf16 *>(base + 3 * kTileBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kTilesBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + N_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int32_t *sList = reinterpret_cast<int32_t *>(tmem_slot + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nqt = (p.nq + BM - 1) / BM;
    const int qt = blockIdx.x % nqt, bh = blockIdx.x / nqt, b = bh / p.H;
    const int q0 = qt * BM;

    if (warp == 4) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(&bars[Q_FULL], 1);
        mbar_init(&bars[KV_FULL], 1);
        mbar_init(&bars[KV_FULL + 1], 1);
        mbar_init(&bars[KV_EMPTY], 1);
        mbar_init(&bars[KV_EMPTY + 1], 1);
        mbar_init(&bars[S_FULL], 1);
        mbar_init(&bars[P_FULL], 4);
        mbar_init(&bars[O_FULL], 1);
        mbar_fence_init();
    }
    int C = 0;
    if (P.gather) {
        uint32_t *bitmap = reinterpret_cast<uint32_t *>(sList + p.N);
        int32_t *wt = reinterpret_cast<int32_t *>(bitmap + ((p.N + 31) >> 5));
        C = build_cached_list(p.idx + (int64_t)b * p.A, p.A, p.N, bitmap, sList, wt, p.status);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;
    const uint32_t tmS = tm, tmO = tm + 128;

    // key slots: full -> rows [0, n_dense); cache-aware -> A active rows (padded to a
    // multiple of 4 for gather4), then the C cached rows
    const int dense_slots = P.gather ? ((p.A + 3) & ~3) : p.n_dense;
    const int n_slots = P.gather ? dense_slots + C : p.n_dense;
    const int nblk = (n_slots + BN - 1) / BN;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&P.mQ);
            tma_prefetch_desc(&P.mKd);
            tma_prefetch_desc(&P.mVd);
            mbar_arrive_expect_tx(&bars[Q_FULL], kTileBytes);
            tma_load_3d(sQ, &P.mQ, 0, q0, bh, &bars[Q_FULL]);
        }
        for (int j = 0; j < nblk; ++j) {
            const int st = j & 1;
            if (!mbar_wait(&bars[KV_EMPTY + st], ((j >> 1) & 1) ^ 1, p.status, abort_flag)) break;
            bf16 *dK = sK0 + st * (kTileBytes / 2);
            bf16 *dV = sV0 + st * (kTileBytes / 2);
            if (lane == 0) mbar_arrive_expect_tx(&bars[KV_FULL + st], 2 * kTileBytes);
            __syncwarp();
            if (!P.gather) {
                if (lane == 0) {
                    tma_load_3d(dK, &P.mKd, 0, j * BN, bh, &bars[KV_FULL + st]);
                    tma_load_3d(dV, &P.mVd, 0, j * BN, bh, &bars[KV_FULL + st]);
                }
            } else {
                // lane l fetches slots 4l .. 4l+3 of the block
                const int s0 = j * BN + 4 * lane;
                int r[4];
                const CUtensorMap *mk, *mv;
                if (s0 < dense_slots || C == 0) {
                    mk = &P.mKd;
                    mv = &P.mVd;
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[i] = bh * p.A + min(s0 + i, p.A - 1);
                } else {
                    mk = &P.mKc;
                    mv = &P.mVc;
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[i] = bh * p.N + sList[min(s0 + i - dense_slots, C - 1)];
                }
                tma_gather4(reinterpret_cast<char *>(dK) + 512 * lane, mk, 0, r[0], r[1], r[2], r[3],
                            &bars[KV_FULL + st]);
                tma_gather4(reinterpret_cast<char *>(dV) + 512 * lane, mv, 0, r[0], r[1], r[2], r[3],
                            &bars[KV_FULL + st]);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(BM, BN, 0, 0);
            const uint32_t idO = idesc_bf16(BM, D, 0, 1);
            const uint64_t dQ = smem_desc(sQ, 16, 1024, Swz::B128);
            bool ok = mbar_wait(&bars[Q_FULL], 0, p.status, abort_flag);
            for (int j = 0; ok && j < nblk; ++j) {
                const int st = j & 1;
                ok = mbar_wait(&bars[KV_FULL + st], (j >> 1) & 1, p.status, abort_flag);
                if (ok && j > 0) ok = mbar_wait(&bars[O_FULL], (j - 1) & 1, p.status, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dK = smem_desc(sK0 + st * (kTileBytes / 2), 16, 1024, Swz::B128);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss(tmS, desc_advance(dQ, 32 * k), desc_advance(dK, 32 * k), idS, k > 0);
                mma_commit(&bars[S_FULL]);
                ok = mbar_wait(&bars[P_FULL], j & 1, p.status, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dV = smem_desc(sV0 + st * (kTileBytes / 2), 1024, 1024, Swz::B128);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) mma_ts(tmO, tmS + 8 * k, desc_advance(dV, 2048 * k), idO, k > 0);
                mma_commit(&bars[O_FULL]);
                mma_commit(&bars[KV_EMPTY + st]);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        if (P.gather && p.fuse_scatter && qt == 0) {
            // Fresh K_A/V_A rows -> cache rows of the active positions (never read here).
            const bf16 *Kd = static_cast<const bf16 *>(p.Kd);
            const bf16 *Vd = static_cast<const bf16 *>(p.Vd);
            bf16 *Kc = static_cast<bf16 *>(p.Kc);
            bf16 *Vc = static_cast<bf16 *>(p.Vc);
            for (int t = tid; t < p.A * (D / 8); t += 128) {
                const int a = t / (D / 8), c = t % (D / 8);
                const int pos = p.idx[(int64_t)b * p.A + a];
                if (pos < 0 || pos >= p.N) continue;
                const int64_t src = ((int64_t)bh * p.A + a) * D + 8 * c;
                const int64_t dst = ((int64_t)bh * p.N + pos) * D + 8 * c;
                *reinterpret_cast<uint4 *>(Kc + dst) = *reinterpret_cast<const uint4 *>(Kd + src);
                *reinterpret_cast<uint4 *>(Vc + dst) = *reinterpret_cast<const uint4 *>(Vd + src);
            }
        }
        const float sl2 = p.scale * kLog2e;
        const int A = p.A;
        auto valid = [&](int slot) -> bool {
            return P.gather ? (slot < A || (slot >= dense_slots && slot < n_slots)) : (slot < n_slots);
        };
        float o[D];
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] = 0.f;
        float m_run = 0.f, l_run = 0.f;
        bool have_o = false, ok = true;
        for (int j = 0; j < nblk; ++j) {
            if (!mbar_wait(&bars[S_FULL], j & 1, p.status, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                const int s0 = j * BN + 32 * c;
                if (s0 < n_slots) {
                    float v[32];
                    tmem_ld32(lane_addr(tmS, warp, 32 * c), v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (valid(s0 + i)) mx = fmaxf(mx, v[i] * sl2);
                }
            }
            const float m_new = (j == 0) ? mx : fmaxf(m_run, mx);
            const float mu = (m_new == -INFINITY) ? 0.f : m_new;
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                const int s0 = j * BN + 32 * c;
                uint32_t w[16];
                if (s0 < n_slots) {
                    float v[32];
                    tmem_ld32(lane_addr(tmS, warp, 32 * c), v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float p0 = valid(s0 + 2 * i) ? fast_exp2(v[2 * i] * sl2 - mu) : 0.f;
                        const float p1 = valid(s0 + 2 * i + 1) ? fast_exp2(v[2 * i + 1] * sl2 - mu) : 0.f;
                        rs += p0 + p1;
                        w[i] = pack_bf16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = 0u;
                }
                tmem_st16(lane_addr(tmS, warp, 16 * c), w);
            }
            tmem_wait_st();
            if (j == 0) {
                l_run = rs;
            } else {
                const float alpha = fast_exp2(m_run - mu);
                l_run = l_run * alpha + rs;
                // fold the previous block's O (relative to m_run) before PV_j overwrites it
                if (!mbar_wait(&bars[O_FULL], (j - 1) & 1, p.status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    tmem_ld32(lane_addr(tmO, warp, 32 * c), v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[32 * c + i] = have_o ? fmaf(o[32 * c + i], 1.f, v[i]) : v[i];
                }
                have_o = true;
                // o now holds sum_{i<j} P_i V_i relative to m_run; rescale to mu
#pragma unroll
                for (int c = 0; c < D; ++c) o[c] *= alpha;
            }
            m_run = mu;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[P_FULL]);
        }
        if (ok && mbar_wait(&bars[O_FULL], (nblk - 1) & 1, p.status, abort_flag)) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                tmem_ld32(lane_addr(tmO, warp, 32 * c), v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[32 * c + i] += v[i];
            }
            const int row = q0 + tid;
            if (row < p.nq) {
                const float inv = 1.f / l_run;
                bf16 *Og = static_cast<bf16 *>(p.O) + ((int64_t)bh * p.nq + row) * D;
#pragma unroll
                for (int c = 0; c < D; c += 8) {
                    uint4 u;
                    u.x = pack_bf16x2(o[c] * inv, o[c + 1] * inv);
                    u.y = pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
                    u.z = pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
                    u.w = pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
                    *reinterpret_cast<uint4 *>(Og + c) = u;
                }
                if (p.lse) p.lse[(int64_t)bh * p.nq + row] = (m_run + log2f(l_run)) * kLn2;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tm, kTmemCols);
}

bool map3(CUtensorMap *m, const void *ptr, int rows, int bh) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)rows, (uint64_t)bh};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)rows * D * 2};
    const uint32_t box[3] = {64, 128, 1};
    return make_map_bf16(m, ptr, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool map_rows(CUtensorMap *m, const void *ptr, int64_t rows) {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, 1};
    return make_map_bf16(m, ptr, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool attn_tc5_supported(const AttnParams &p) { return p.d == D; }

cudaError_t launch_attn_bf16_tc5(const AttnParams &p, cudaStream_t s) {
    if (p.d != D) return cudaErrorInvalidValue;
    static int configured[64] = {0};
    Tc5Params P;
    P.a = p;
    P.gather = p.idx ? 1 : 0;
    const int bh = p.B * p.H;
    bool ok = map3(&P.mQ, p.Q, p.nq, bh);
    if (P.gather) {
        ok = ok && map_rows(&P.mKd, p.Kd, (int64_t)bh * p.A) && map_rows(&P.mVd, p.Vd, (int64_t)bh * p.A);
        ok = ok && map_rows(&P.mKc, p.Kc, (int64_t)bh * p.N) && map_rows(&P.mVc, p.Vc, (int64_t)bh * p.N);
    } else {
        ok = ok && map3(&P.mKd, p.Kd, p.n_dense, bh) && map3(&P.mVd, p.Vd, p.n_dense, bh);
        P.mKc = P.mKd;
        P.mVc = P.mVd;
    }
    if (!ok) return cudaErrorInvalidValue;
    size_t smem = 1024 + kTilesBytes + N_BARS * 8 + 16;
    if (P.gather) smem += sizeof(int32_t) * (p.N + (p.N + 31) / 32 + kThreads / 32);
    cudaError_t e = ensure_smem(attn_tc5_kernel, smem, configured);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)((p.nq + BM - 1) / BM) * bh;
    attn_tc5_kernel<<<(unsigned)blocks, kThreads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace mar
