// bf16 attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), d = 64 or 80.
//
// Serves full attention (key list = all N rows of K/V) and cache-aware attention (key
// list = the fresh active rows K_A/V_A followed by the cache rows of the cached set),
// see attn.h.
//
// MARché notes, Key Design 2: each active query attends over fresh K_A/V_A and stored
// cached K/V as two partial softmax sums merged by the safe online-softmax rule (running
// max, running sum), with no concatenated key buffer in memory. The key list is streamed
// in blocks of 64 slots straight from the two sources into shared memory: TMA tile loads
// for contiguous rows (full attention), TMA gather4 loads (four rows per instruction) of
// the active rows and of the cached rows named by an in-CTA list built from the active
// indices (cache rows of active positions are never read).
//
// CTA = one (b, h) and 128 query rows; 6 warps:
//   warps 0-3  softmax + epilogue; thread t owns query row t (tensor-memory lane t)
//   warp 4     TMA producer (Q once; K/V blocks through a ring of stages)
//   warp 5     MMA issuer (one lane):  S_j = Q K_j^T  (M=128, N=64, K=d, K-major operands)
//                                       O  += P_j V_j  (M=128, N=d, K=64, P from TMEM,
//                                                       V MN-major)
// Tensor memory (256 columns): two S buffers of 64 columns (S_j, S_{j+1}), each
// overwritten in place by P_j as packed bf16 pairs, and O (d columns) accumulated by the
// MMAs across all blocks. While the softmax warps turn S_j into P_j, the tensor core
// already computes S_{j+1}.
//
// Online softmax with a lazy rescale: each row keeps the max m it used for its P values;
// a block whose row max exceeds m by more than 8 (base-2 units) raises m and rescales
// O and l by 2^(m_old - m_new) in tensor memory; otherwise P = 2^(s - m) <= 2^8 and no
// rescale is needed. O / l at the end is the same softmax-weighted sum either way.
// d = 80 keeps columns 64..79 of every tile in a separate 32-byte-swizzled region:
// QK^T takes 4 k-steps on the 128-byte-swizzled part and 1 on the tail; PV issues an
// N=64 and an N=16 MMA per k-step. Every wait is bounded (tc5.cuh).
#include <cmath>

#include "attn.h"
#include "common.cuh"
#include "tc5.cuh"
#include "tma_host.h"

namespace mar {
namespace {

using namespace tc5;

constexpr int BM = 128;          // query rows per CTA
constexpr int BN = 64;           // key slots per block
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescale = 8.f;  // lazy-rescale threshold (base-2 units)

template <int D>
struct Cfg {
    static constexpr int DB = D - 64;                         // tail columns (0 or 16)
    static constexpr int kStages = (D == 64) ? 4 : 3;
    static constexpr uint32_t kQa = BM * 128, kQb = BM * DB * 2;            // Q tile parts
    static constexpr uint32_t kKa = BN * 128, kKb = BN * DB * 2;            // one K (or V) block
    static constexpr uint32_t kKV = 2 * (kKa + kKb);                        // K + V of one block
    // shared-memory offsets (1024-aligned pieces)
    static constexpr uint32_t oQa = 0, oQb = oQa + kQa;
    static constexpr uint32_t oStage = ((oQb + kQb + 1023) / 1024) * 1024;
    static constexpr uint32_t kStageBytes = ((kKV + 1023) / 1024) * 1024;
    static constexpr uint32_t oBars = oStage + kStages * kStageBytes;
    // stage layout: Ka | Va | Kb | Vb
    static constexpr uint32_t sKa = 0, sVa = kKa, sKb = 2 * kKa, sVb = 2 * kKa + kKb;
};

enum Bar { Q_FULL = 0, S_FULL = 1, P_FULL = 3, O_DONE = 5, KV_FULL = 6 };  // then KV_EMPTY

template <int D>
struct Tc5Params {
    CUtensorMap mQa, mQb;    // 3-D [BH, nq, D]: box {64,128,1} (SW128) / {16,128,1} (SW32)
    CUtensorMap mKa, mKb;    // full: 3-D [BH, n_dense, D] box {64|16, 64, 1};
    CUtensorMap mVa, mVb;    // cache-aware: 2-D [BH*A, D] box {64|16, 1}
    CUtensorMap mKca, mKcb;  // cache-aware: 2-D [BH*N, D] box {64|16, 1}
    CUtensorMap mVca, mVcb;
    AttnParams a;
    int gather;
};

MAR_DEVINL uint32_t lane_addr(uint32_t tm, int warp, int col) {
    return tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)col;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) attn_tc5_kernel(const __grid_constant__ Tc5Params<D> P) {
    using C = Cfg<D>;
    constexpr int S = C::kStages;
    const AttnParams &p = P.a;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    unsigned char *sm = reinterpret_cast<unsigned char *>(base);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::oBars);
    uint64_t *kv_empty = bars + KV_FULL + S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + KV_FULL + 2 * S);
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[S_FULL + i], 1);
            mbar_init(&bars[P_FULL + i], 4);
        }
        mbar_init(&bars[O_DONE], 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&bars[KV_FULL + i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4 && lane == 0) {  // Q does not depend on the cached list: start it now
        tma_prefetch_desc(&P.mQa);
        mbar_arrive_expect_tx(&bars[Q_FULL], C::kQa + C::kQb);
        tma_load_3d(sm + C::oQa, &P.mQa, 0, q0, bh, &bars[Q_FULL]);
        if constexpr (C::DB > 0) tma_load_3d(sm + C::oQb, &P.mQb, 64, q0, bh, &bars[Q_FULL]);
    }
    int Ccnt = 0;
    if (P.gather) {
        uint32_t *bitmap = reinterpret_cast<uint32_t *>(sList + p.N);
        int32_t *wt = reinterpret_cast<int32_t *>(bitmap + ((p.N + 31) >> 5));
        Ccnt = build_cached_list(p.idx + (int64_t)b * p.A, p.A, p.N, bitmap, sList, wt, p.status);
    } else {
        __syncthreads();
    }
    const uint32_t tm = *tmem_slot;
    const uint32_t tmS0 = tm, tmO = tm + 128;

    const int dense_slots = P.gather ? ((p.A + 3) & ~3) : p.n_dense;
    const int n_slots = P.gather ? dense_slots + Ccnt : p.n_dense;
    const int nblk = (n_slots + BN - 1) / BN;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        for (int j = 0; j < nblk; ++j) {
            const int st = j % S;
            if (!mbar_wait(&kv_empty[st], ((j / S) & 1) ^ 1, p.status, abort_flag)) break;
            unsigned char *stg = sm + C::oStage + st * C::kStageBytes;
            if (lane == 0) mbar_arrive_expect_tx(&bars[KV_FULL + st], C::kKV);
            __syncwarp();
            if (!P.gather) {
                if (lane == 0) {
                    tma_load_3d(stg + C::sKa, &P.mKa, 0, j * BN, bh, &bars[KV_FULL + st]);
                    tma_load_3d(stg + C::sVa, &P.mVa, 0, j * BN, bh, &bars[KV_FULL + st]);
                    if constexpr (C::DB > 0) {
                        tma_load_3d(stg + C::sKb, &P.mKb, 64, j * BN, bh, &bars[KV_FULL + st]);
                        tma_load_3d(stg + C::sVb, &P.mVb, 64, j * BN, bh, &bars[KV_FULL + st]);
                    }
                }
            } else {
                // lane l: group g = l & 15 (slots 4g..4g+3 of the block); lanes 0-15 -> K, 16-31 -> V
                const int g = lane & 15;
                const bool isV = lane >= 16;
                const int s0 = j * BN + 4 * g;
                int r[4];
                const bool dense = (s0 < dense_slots) || (Ccnt == 0);
                if (dense) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[i] = bh * p.A + min(s0 + i, p.A - 1);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[i] = bh * p.N + sList[min(s0 + i - dense_slots, Ccnt - 1)];
                }
                const CUtensorMap *ma = dense ? (isV ? &P.mVa : &P.mKa) : (isV ? &P.mVca : &P.mKca);
                tma_gather4(stg + (isV ? C::sVa : C::sKa) + 512 * g, ma, 0, r[0], r[1], r[2], r[3],
                            &bars[KV_FULL + st]);
                if constexpr (C::DB > 0) {
                    const CUtensorMap *mb = dense ? (isV ? &P.mVb : &P.mKb) : (isV ? &P.mVcb : &P.mKcb);
                    tma_gather4(stg + (isV ? C::sVb : C::sKb) + 128 * g, mb, 64, r[0], r[1], r[2], r[3],
                                &bars[KV_FULL + st]);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(BM, BN, 0, 0);
            const uint32_t idOa = idesc_bf16(BM, 64, 0, 1);
            const uint32_t idOb = idesc_bf16(BM, 16, 0, 1);
            const uint64_t dQa = smem_desc(sm + C::oQa, 16, 1024, Swz::B128);
            const uint64_t dQb = smem_desc(sm + C::oQb, 16, 256, Swz::B32);
            auto issue_S = [&](int j) {
                const int st = j % S;
                const unsigned char *stg = sm + C::oStage + st * C::kStageBytes;
                const uint64_t dKa = smem_desc(stg + C::sKa, 16, 1024, Swz::B128);
                const uint32_t dst = tmS0 + 64 * (j & 1);
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_ss(dst, desc_advance(dQa, 32 * k), desc_advance(dKa, 32 * k), idS, k > 0);
                if constexpr (C::DB > 0) mma_ss(dst, dQb, smem_desc(stg + C::sKb, 16, 256, Swz::B32), idS, 1);
                mma_commit(&bars[S_FULL + (j & 1)]);
            };
            bool ok = mbar_wait(&bars[Q_FULL], 0, p.status, abort_flag);
            for (int j = 0; ok && j < 2 && j < nblk; ++j) {
                ok = mbar_wait(&bars[KV_FULL + j % S], (j / S) & 1, p.status, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_S(j);
            }
            for (int j = 0; ok && j < nblk; ++j) {
                const int st = j % S;
                ok = mbar_wait(&bars[P_FULL + (j & 1)], (j >> 1) & 1, p.status, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const unsigned char *stg = sm + C::oStage + st * C::kStageBytes;
                const uint64_t dVa = smem_desc(stg + C::sVa, 1024, 1024, Swz::B128);
                const uint64_t dVb = smem_desc(stg + C::sVb, 256, 256, Swz::B32);
                const uint32_t pcol = tmS0 + 64 * (j & 1);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint32_t acc = (j > 0 || k > 0) ? 1u : 0u;
                    mma_ts(tmO, pcol + 8 * k, desc_advance(dVa, 2048 * k), idOa, acc);
                    if constexpr (C::DB > 0) mma_ts(tmO + 64, pcol + 8 * k, desc_advance(dVb, 512 * k), idOb, acc);
                }
                mma_commit(&bars[O_DONE]);
                mma_commit(&kv_empty[st]);
                if (j + 2 < nblk) {
                    // S_{j+2} reuses P_j's columns: wait until PV_j has consumed them
                    ok = mbar_wait(&bars[O_DONE], j & 1, p.status, abort_flag);
                    if (ok) ok = mbar_wait(&bars[KV_FULL + (j + 2) % S], ((j + 2) / S) & 1, p.status, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_S(j + 2);
                }
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
        const bool live = (q0 + 32 * warp) < p.nq;  // warp-uniform: some row of this warp is real
        float m_use = 0.f, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            const int buf = j & 1;
            if (!mbar_wait(&bars[S_FULL + buf], (j >> 1) & 1, p.status, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (live) {
                float v[64];
                tmem_ld64(lane_addr(tmS0, warp, 64 * buf), v);
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] *= sl2;
                // mask slots that are not keys: past the list, or the gather4 padding
                const int s0 = j * BN;
                const bool all_valid = P.gather ? (s0 + BN <= n_slots && (s0 >= dense_slots || s0 + BN <= p.A))
                                                : (s0 + BN <= n_slots);
                if (!all_valid) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int s = s0 + i;
                        const bool ok_slot = P.gather ? (s < p.A || (s >= dense_slots && s < n_slots)) : (s < n_slots);
                        if (!ok_slot) v[i] = -INFINITY;
                    }
                }
                float mx = v[0];
#pragma unroll
                for (int i = 1; i < 64; ++i) mx = fmaxf(mx, v[i]);
                bool rescale = false;
                float factor = 1.f;
                if (j == 0) {
                    m_use = (mx == -INFINITY) ? 0.f : mx;
                } else if (mx > m_use + kRescale) {
                    factor = fast_exp2(m_use - mx);
                    m_use = mx;
                    rescale = true;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O holds sum_{i<j} P_i V_i; wait for it and scale rows that raised their max
                    if (!mbar_wait(&bars[O_DONE], (j - 1) & 1, p.status, abort_flag)) {
                        ok = false;
                    } else {
                        tc_fence_after();
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 16) {
                            float o[16];
                            tmem_ld16(lane_addr(tmO, warp, c0), o);
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(o[i] * factor);
                            tmem_st16(lane_addr(tmO, warp, c0), w);
                        }
                        l *= factor;
                    }
                }
                float rs = 0.f;
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = fast_exp2(v[2 * i] - m_use);
                    const float p1 = fast_exp2(v[2 * i + 1] - m_use);
                    rs += p0 + p1;
                    w[i] = pack_bf16x2(p0, p1);
                }
                l += rs;
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    w0[i] = w[i];
                    w1[i] = w[16 + i];
                }
                tmem_st16(lane_addr(tmS0, warp, 64 * buf), w0);
                tmem_st16(lane_addr(tmS0, warp, 64 * buf + 16), w1);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[P_FULL + buf]);
            if (!ok) break;
        }
        // A parity wait is only unambiguous when the phase before it is known complete:
        // the S of the last block was issued after PV of block nblk-3, so wait for PV of
        // block nblk-2 first, then for the last one.
        if (ok && nblk >= 2) ok = mbar_wait(&bars[O_DONE], (nblk - 2) & 1, p.status, abort_flag);
        if (ok && mbar_wait(&bars[O_DONE], (nblk - 1) & 1, p.status, abort_flag) && live) {
            tc_fence_after();
            const int row = q0 + tid;
            const float inv = 1.f / l;
            bf16 *Og = static_cast<bf16 *>(p.O) + ((int64_t)bh * p.nq + row) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                float o[16];
                tmem_ld16(lane_addr(tmO, warp, c0), o);
                if (row < p.nq) {
                    uint4 u0, u1;
                    u0.x = pack_bf16x2(o[0] * inv, o[1] * inv);
                    u0.y = pack_bf16x2(o[2] * inv, o[3] * inv);
                    u0.z = pack_bf16x2(o[4] * inv, o[5] * inv);
                    u0.w = pack_bf16x2(o[6] * inv, o[7] * inv);
                    u1.x = pack_bf16x2(o[8] * inv, o[9] * inv);
                    u1.y = pack_bf16x2(o[10] * inv, o[11] * inv);
                    u1.z = pack_bf16x2(o[12] * inv, o[13] * inv);
                    u1.w = pack_bf16x2(o[14] * inv, o[15] * inv);
                    *reinterpret_cast<uint4 *>(Og + c0) = u0;
                    *reinterpret_cast<uint4 *>(Og + c0 + 8) = u1;
                }
            }
            if (p.lse && row < p.nq) p.lse[(int64_t)bh * p.nq + row] = (m_use + log2f(l)) * kLn2;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tm, kTmemCols);
}

template <int D>
bool map3(CUtensorMap *m, const void *ptr, int rows, int bh, uint32_t boxw, uint32_t boxh) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)rows, (uint64_t)bh};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)rows * D * 2};
    const uint32_t box[3] = {boxw, boxh, 1};
    return make_map_bf16(m, ptr, 3, dims, strides, box,
                         boxw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B);
}

template <int D>
bool map_rows(CUtensorMap *m, const void *ptr, int64_t rows, uint32_t boxw) {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {boxw, 1};
    return make_map_bf16(m, ptr, 2, dims, strides, box,
                         boxw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B);
}

template <int D>
cudaError_t launch(const AttnParams &p, cudaStream_t s) {
    using C = Cfg<D>;
    static int configured[64] = {0};
    Tc5Params<D> P;
    P.a = p;
    P.gather = p.idx ? 1 : 0;
    const int bh = p.B * p.H;
    const uint32_t tw = D == 64 ? 64 : 16;  // tail box width (unused for d = 64)
    bool ok = map3<D>(&P.mQa, p.Q, p.nq, bh, 64, BM) && map3<D>(&P.mQb, p.Q, p.nq, bh, tw, BM);
    if (P.gather) {
        const int64_t ra = (int64_t)bh * p.A, rc = (int64_t)bh * p.N;
        ok = ok && map_rows<D>(&P.mKa, p.Kd, ra, 64) && map_rows<D>(&P.mKb, p.Kd, ra, tw);
        ok = ok && map_rows<D>(&P.mVa, p.Vd, ra, 64) && map_rows<D>(&P.mVb, p.Vd, ra, tw);
        ok = ok && map_rows<D>(&P.mKca, p.Kc, rc, 64) && map_rows<D>(&P.mKcb, p.Kc, rc, tw);
        ok = ok && map_rows<D>(&P.mVca, p.Vc, rc, 64) && map_rows<D>(&P.mVcb, p.Vc, rc, tw);
    } else {
        ok = ok && map3<D>(&P.mKa, p.Kd, p.n_dense, bh, 64, BN) && map3<D>(&P.mKb, p.Kd, p.n_dense, bh, tw, BN);
        ok = ok && map3<D>(&P.mVa, p.Vd, p.n_dense, bh, 64, BN) && map3<D>(&P.mVb, p.Vd, p.n_dense, bh, tw, BN);
        P.mKca = P.mKa; P.mKcb = P.mKb; P.mVca = P.mVa; P.mVcb = P.mVb;
    }
    if (!ok) return cudaErrorInvalidValue;
    size_t smem = 1024 + C::oBars + 8 * (KV_FULL + 2 * C::kStages) + 16;
    if (P.gather) smem += sizeof(int32_t) * (p.N + (p.N + 31) / 32 + kThreads / 32);
    cudaError_t e = ensure_smem(attn_tc5_kernel<D>, smem, configured);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)((p.nq + BM - 1) / BM) * bh;
    attn_tc5_kernel<D><<<(unsigned)blocks, kThreads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace

bool attn_tc5_supported(const AttnParams &p) { return p.d == 64 || p.d == 80; }

cudaError_t launch_attn_bf16_tc5(const AttnParams &p, cudaStream_t s) {
    if (p.d == 64) return launch<64>(p, s);
    if (p.d == 80) return launch<80>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace mar
