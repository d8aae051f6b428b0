// bf16 attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), d = 64 or 80.
//
// Serves full attention (key list = all N rows of K/V) and cache-aware attention (key
// list = the fresh active rows K_A/V_A followed by the cache rows of the cached set),
// see attn.h.
//
// MARché notes, Key Design 2: each active query attends over fresh K_A/V_A and stored
// cached K/V as two partial softmax sums merged by the safe online-softmax rule (running
// max, running sum), with no concatenated key buffer in memory. The key list is streamed
// in blocks of 64 rows straight from the two sources into shared memory with TMA tile
// loads: first the fresh active rows (cache-aware) or all rows (full attention), then,
// for cache-aware attention, the cache slab of the (b, h) in position order. Cache rows
// of active positions hold stale values: a bitmap of the active positions masks them out
// of the softmax and the S issuer clears their V rows in shared memory, so they never
// contribute (they are read, costing A/N extra bytes, because one tile load per 64 rows
// runs at the TMA unit's full rate while a per-row gather is bound by its request rate).
// The fresh active rows come either as dense [BH, A, d] blocks (TMA tile loads) or are read
// in place from the whole fresh tensors through the active index (the index warp copies
// them, 16 bytes per lane, into the same swizzled layouts).
//
// Persistent CTAs (two per SM; 8 warps x at most 128 registers, so that the two CTAs'
// 16 warps fill the four 16K-register sub-partitions of an SM): CTA c processes the
// tiles c, c + grid, ... where a tile is one (b, h) and 128 query rows. 8 warps:
//   warps 0-3  softmax + epilogue; thread t owns query row t (tensor-memory lane t)
//   warp 4     TMA producer: Q of each tile (double-buffered) and the K/V blocks of all
//              tiles through one ring of stages, running ahead across tile boundaries;
//              for full attention with the cache refresh it also stores the K/V blocks of
//              each (b, h)'s first query tile to the cache (TMA tile stores from the stages);
//              for full attention it stores each tile's O, which the epilogue stages in
//              the tile's Q buffer (cache-aware launches write O rows from the softmax
//              warps; in the gather form the index warp owns the Q buffers)
//   warp 5     S issuer (one elected lane):  S_g = Q K_g^T  (M=128, N=64, K=d, K-major
//              operands), once K_g has landed and PV_{g-SB} has released S/P buffer g % SB;
//              as soon as a cache block's stage has landed (before the wait for PV_{g-SB},
//              which this work then overlaps), the whole warp clears its stale V rows
//   warp 7     PV issuer (one elected lane): O += P_g V_g  (M=128, N=d, K=64, P from
//              TMEM, V MN-major), as soon as P_g is written; it releases the K/V stage
//   warp 6     index warp: bitmap of the active positions of each tile (double-
//              buffered), the fused cache scatter and, when the active rows are read in
//              place from the whole fresh tensors, the copies of those rows into the Q
//              buffer and the dense-block stages (which the producer hands over).
// g numbers the key blocks of a CTA across its tiles; every ring (stages, S/P buffers,
// Q buffers, bitmaps) is indexed by g or by the tile count, and every barrier is waited
// one phase at a time, in order, so parity waits are exact.
//
// Shared memory: two Q buffers and a ring of K/V stages, 3 for d = 80 and 4 for d = 64, one
// more when a cache-aware launch has at most 96 queries: its Q buffers then hold 64 or 96
// rows (the 96-row kernels are compiled in attn_tc5_q96.cu). A stage is reloaded only after the PV of the block it
// held, and a stage landing late delays the S of its block, on which the softmax warps
// wait: the extra stage took the MAR-H cache-aware launch from 295 to 270 us (d = 80) and
// the MAR-L one from 119 to 117 us (d = 64).
//
// Tensor memory (256 columns): two S buffers of 64 columns, each overwritten in place by
// P as packed bf16 pairs, and O (d columns) accumulated across the blocks of a tile. A
// third buffer (room for it at d = 64) measured no faster for full attention and 4%
// slower for the MAR-L cache-aware launch. The kGen instantiation (full attention with
// the layer-2 score) also stores the raw scores and (m, l) of the rows that are
// generating queries.
// Online softmax with a lazy rescale: a row keeps the max m used for its P values; a
// block whose row max exceeds m by more than 8 (base-2 units) raises m and rescales O
// and l by 2^(m_old - m_new); otherwise P = 2^(s - m) <= 2^8 and nothing is rescaled.
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

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 64;           // keys per block
constexpr int kThreads = 256;    // 8 warps
constexpr uint32_t kTmemCols = 256;
constexpr float kRescale = 8.f;  // lazy-rescale threshold (base-2 units)

// QR: query rows a Q buffer holds. 64 or 96 for cache-aware launches of at most that many
// queries (the MMAs still read 128 rows: the rows past QR fall on whatever follows in
// shared memory, and their S, P and O lanes belong to softmax warps that have no live row
// and never read them), else BM.
template <int D, int QR = BM>
struct Cfg {
    static constexpr int DB = D - 64;                                   // tail columns (0 or 16)
    // K/V stages: what shared memory holds next to two Q buffers of QR rows (two CTAs per SM)
    static constexpr int kStages = ((D == 64) ? 4 : 3) + (QR < BM ? 1 : 0);
    static_assert(kStages <= 5, "barrier slots hold at most five stages");
    // Waits spin at d = 64 (the softmax warps keep pace with the tensor pipe there, and a
    // warp resuming late from a suspended wait costs its block; measured 5-9% faster) and
    // suspend at d = 80 (where spinning warps take issue slots from the other CTA's softmax
    // warps on the same sub-partitions; measured 3% slower).
    static constexpr bool kSpin = (D == 64);
    // S/P buffers of 64 tensor-memory columns; O takes D columns after them (<= 256)
    static constexpr int kSB = 2;
    static_assert(64 * kSB + D <= 256, "tensor memory: S/P buffers + O exceed 256 columns");
    static constexpr uint32_t kQa = QR * 128, kQb = QR * DB * 2;        // Q tile parts
    static constexpr uint32_t kQBytes = ((kQa + kQb + 1023) / 1024) * 1024;
    static constexpr uint32_t kKa = BN * 128, kKb = BN * DB * 2;        // one K (or V) block
    static constexpr uint32_t kKV = 2 * (kKa + kKb);                    // K + V of one block
    static constexpr uint32_t kStageBytes = ((kKV + 1023) / 1024) * 1024;
    // shared memory: Q[2] | stages | barriers | bitmaps
    static constexpr uint32_t oQ = 0;
    static constexpr uint32_t oStage = 2 * kQBytes;
    static constexpr uint32_t oBars = oStage + kStages * kStageBytes;
    // Q buffer layout: Qa | Qb; stage layout: Ka | Va | Kb | Vb
    static constexpr uint32_t sKa = 0, sVa = kKa, sKb = 2 * kKa, sVb = 2 * kKa + kKb;
};

// barrier slots
enum Bar {
    Q_FULL = 0,      // [2]
    Q_EMPTY = 2,     // [2]
    S_FULL = 4,      // [kSB <= 3]
    P_FULL = 7,      // [kSB]
    O_DONE = 10,     // [kSB] PV of block g -> O_DONE[g % kSB]
    BM_FULL = 13,    // [2]
    BM_EMPTY = 15,   // [2]
    O_STAGED = 17,   // [2] the tile's normalised O is in its Q buffer (one arrival per softmax warp)
    DENSE_DONE = 19, // [S <= 5] fresh mode: the index warp is done with a dense-block stage
    DENSE_GO = 24,   // [S] fresh mode: the producer hands a free stage for a dense block to it
    KV_FULL = 29     // [S], then KV_EMPTY [S]
};

template <int D>
struct Tc5Params {
    CUtensorMap mQa, mQb;    // 3-D [BH, nq, D]: box {64,128,1} (SW128) / {16,128,1} (SW32)
    CUtensorMap mOa, mOb;    // O, the same layout and boxes (full attention: tile stores from the staged Q buffer)
    CUtensorMap mKa, mKb;    // 3-D [BH, n_dense, D], box {64|16, 64, 1}: all rows / active rows
    CUtensorMap mVa, mVb;
    CUtensorMap mKca, mKcb;  // cache [BH, N, D], box {64|16, 64, 1}: read (cache-aware) or
    CUtensorMap mVca, mVcb;  // written (full attention with the cache refresh)
    AttnParams a;
    int gather;
    int store;               // full attention: store every K/V block of query tile 0 to the cache
    int idle_scatter;        // the fused scatter is written by the softmax warps without a live row
    int n_tiles;
};

MAR_DEVINL uint32_t lane_addr(uint32_t tm, int warp, int col) {
    return tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)col;
}

// kGen: full attention that also leaves the generating rows' raw scores (a separate
// instantiation, so that the other launches keep the code they had without it).
MAR_DEVINL void st_global_v4_if(bool pred, float *ptr, float a, float b, float c, float d) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %0, 0;\n @p st.global.v4.f32 [%1], {%2, %3, %4, %5};\n}\n" ::"r"(
            (uint32_t)pred),
        "l"(ptr), "f"(a), "f"(b), "f"(c), "f"(d));
}
// 64 consecutive floats v[0..63] to ptr (16-byte aligned) when pred: one predicate, one base.
MAR_DEVINL void st_global_row64_if(bool pred, float *ptr, const float *v) {
#define MAR_ST4(o, i) "@p st.global.v4.f32 [%1+" #o "], {%" #i ", %" #i "+1, %" #i "+2, %" #i "+3};\n"
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %0, 0;\n"
        "@p st.global.v4.f32 [%1+0], {%2, %3, %4, %5};\n"
        "@p st.global.v4.f32 [%1+16], {%6, %7, %8, %9};\n"
        "@p st.global.v4.f32 [%1+32], {%10, %11, %12, %13};\n"
        "@p st.global.v4.f32 [%1+48], {%14, %15, %16, %17};\n"
        "@p st.global.v4.f32 [%1+64], {%18, %19, %20, %21};\n"
        "@p st.global.v4.f32 [%1+80], {%22, %23, %24, %25};\n"
        "@p st.global.v4.f32 [%1+96], {%26, %27, %28, %29};\n"
        "@p st.global.v4.f32 [%1+112], {%30, %31, %32, %33};\n"
        "@p st.global.v4.f32 [%1+128], {%34, %35, %36, %37};\n"
        "@p st.global.v4.f32 [%1+144], {%38, %39, %40, %41};\n"
        "@p st.global.v4.f32 [%1+160], {%42, %43, %44, %45};\n"
        "@p st.global.v4.f32 [%1+176], {%46, %47, %48, %49};\n"
        "@p st.global.v4.f32 [%1+192], {%50, %51, %52, %53};\n"
        "@p st.global.v4.f32 [%1+208], {%54, %55, %56, %57};\n"
        "@p st.global.v4.f32 [%1+224], {%58, %59, %60, %61};\n"
        "@p st.global.v4.f32 [%1+240], {%62, %63, %64, %65};\n"
        "}\n" ::"r"((uint32_t)pred),
        "l"(ptr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
        "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]),
        "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31]), "f"(v[32]), "f"(v[33]), "f"(v[34]),
        "f"(v[35]), "f"(v[36]), "f"(v[37]), "f"(v[38]), "f"(v[39]), "f"(v[40]), "f"(v[41]), "f"(v[42]), "f"(v[43]),
        "f"(v[44]), "f"(v[45]), "f"(v[46]), "f"(v[47]), "f"(v[48]), "f"(v[49]), "f"(v[50]), "f"(v[51]), "f"(v[52]),
        "f"(v[53]), "f"(v[54]), "f"(v[55]), "f"(v[56]), "f"(v[57]), "f"(v[58]), "f"(v[59]), "f"(v[60]), "f"(v[61]),
        "f"(v[62]), "f"(v[63]));
#undef MAR_ST4
}

// 64 consecutive floats v[0..63] to ptr (32-byte aligned) when pred: eight 256-bit stores.
MAR_DEVINL void st_global_row64_v8_if(bool pred, float *ptr, const float *v) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %0, 0;\n"
        "@p st.global.v8.f32 [%1+0], {%2, %3, %4, %5, %6, %7, %8, %9};\n"
        "@p st.global.v8.f32 [%1+32], {%10, %11, %12, %13, %14, %15, %16, %17};\n"
        "@p st.global.v8.f32 [%1+64], {%18, %19, %20, %21, %22, %23, %24, %25};\n"
        "@p st.global.v8.f32 [%1+96], {%26, %27, %28, %29, %30, %31, %32, %33};\n"
        "@p st.global.v8.f32 [%1+128], {%34, %35, %36, %37, %38, %39, %40, %41};\n"
        "@p st.global.v8.f32 [%1+160], {%42, %43, %44, %45, %46, %47, %48, %49};\n"
        "@p st.global.v8.f32 [%1+192], {%50, %51, %52, %53, %54, %55, %56, %57};\n"
        "@p st.global.v8.f32 [%1+224], {%58, %59, %60, %61, %62, %63, %64, %65};\n"
        "}\n" ::"r"((uint32_t)pred),
        "l"(ptr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
        "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]),
        "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31]), "f"(v[32]), "f"(v[33]), "f"(v[34]),
        "f"(v[35]), "f"(v[36]), "f"(v[37]), "f"(v[38]), "f"(v[39]), "f"(v[40]), "f"(v[41]), "f"(v[42]), "f"(v[43]),
        "f"(v[44]), "f"(v[45]), "f"(v[46]), "f"(v[47]), "f"(v[48]), "f"(v[49]), "f"(v[50]), "f"(v[51]), "f"(v[52]),
        "f"(v[53]), "f"(v[54]), "f"(v[55]), "f"(v[56]), "f"(v[57]), "f"(v[58]), "f"(v[59]), "f"(v[60]), "f"(v[61]),
        "f"(v[62]), "f"(v[63]));
}

// Warp-wide bounded wait of the attention kernel: suspending (try_wait) or spinning.
template <bool kSpin>
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity, uint32_t *status, volatile int *abort) {
    if constexpr (kSpin) return mbar_spin_all(bar, parity, status, abort);
    else return mbar_wait_all(bar, parity, status, abort);
}

// kGen: 0 = plain attention; 1 = with the generating rows' raw scores, 16-byte stores;
// 2 = the same with 32-byte stores (N % 8 == 0 and a 32-byte-aligned score buffer, so that
// every row and block starts on a 32-byte boundary).
// kDirectO: the softmax warps write O rows straight to global memory (cache-aware launches,
// whose O is A rows per (b, h)); else O is staged in the tile's Q buffer for a TMA store.
template <int D, int kGen, int QR, bool kDirectO>
__global__ void __maxnreg__(128) attn_tc5_kernel(const __grid_constant__ Tc5Params<D> P) {
    using C = Cfg<D, QR>;
    constexpr int S = C::kStages;
    constexpr int SB = C::kSB;
    const AttnParams &p = P.a;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    unsigned char *sm = reinterpret_cast<unsigned char *>(base);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::oBars);
    uint64_t *kv_empty = bars + KV_FULL + S;
    uint64_t *drain = bars + KV_FULL + 2 * S;  // [2] abort path: the S and the PV issuer's MMAs
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + KV_FULL + 2 * S + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int bm_words = 2 * ((p.N + BN - 1) / BN);  // one bitmap: whole 64-position blocks
    uint32_t *bitmaps = reinterpret_cast<uint32_t *>(tmem_slot + 4);  // [2][bm_words]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nqt = (p.nq + BM - 1) / BM;
    const int my_tiles = (P.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

    // key blocks per tile: nd blocks of dense rows (the fresh active rows, or all rows of
    // K/V), then for cache-aware attention nc blocks of the cache slab in position order
    const int nd = (p.n_dense + BN - 1) / BN;
    const int nc = (P.gather && p.A < p.N) ? (p.N + BN - 1) / BN : 0;
    const int nblk = nd + nc;

    if (warp == 4) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[Q_FULL + i], 1);
            mbar_init(&bars[Q_EMPTY + i], 1);
            mbar_init(&bars[BM_FULL + i], 1);
            mbar_init(&bars[BM_EMPTY + i], 4);
            mbar_init(&bars[O_STAGED + i], 4);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&bars[S_FULL + i], 1);
            mbar_init(&bars[P_FULL + i], 4);
            mbar_init(&bars[O_DONE + i], 1);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&bars[DENSE_GO + i], 1);
            mbar_init(&bars[DENSE_DONE + i], 1);
            mbar_init(&bars[KV_FULL + i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;
    const uint32_t tmS0 = tm, tmO = tm + 64 * SB;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&P.mQa);
            tma_prefetch_desc(&P.mKa);
            tma_prefetch_desc(&P.mVa);
            // Cache refresh (full attention, P.store): the query tile 0 of every (b, h) visits
            // all of its key blocks, and each staged block is stored to the cache by TMA once it
            // has landed. The store of block g is issued after the loads of block g + 1; a stage
            // is refilled only after its store has finished reading it (bulk groups, one per
            // block, possibly empty, so the count to wait for is fixed).
            int pend_g = -1, pend_bh = 0, pend_row = 0;  // block whose store is due next
            auto store_pending = [&]() -> bool {
                if (pend_g < 0) return true;
                const int pst = pend_g % S;
                if (!mbar_wait(&bars[KV_FULL + pst], (pend_g / S) & 1, p.status, abort_flag)) return false;
                const unsigned char *stg = sm + C::oStage + pst * C::kStageBytes;
                tma_store_3d(&P.mKca, 0, pend_row, pend_bh, stg + C::sKa);
                tma_store_3d(&P.mVca, 0, pend_row, pend_bh, stg + C::sVa);
                if constexpr (C::DB > 0) {
                    tma_store_3d(&P.mKcb, 64, pend_row, pend_bh, stg + C::sKb);
                    tma_store_3d(&P.mVcb, 64, pend_row, pend_bh, stg + C::sVb);
                }
                pend_g = -1;
                return true;
            };
            // O of tile t is staged by the softmax warps in Q buffer t & 1; it is stored to
            // global memory by TMA from there before that buffer takes the Q of tile t + 2 (or
            // after the last tile), and the buffer is reloaded only once the store has read it.
            // (In fresh mode the index warp owns the Q buffers and does this.)
            auto store_o = [&](int t) -> bool {
                if (!mbar_wait(&bars[O_STAGED + (t & 1)], (t >> 1) & 1, p.status, abort_flag)) return false;
                if constexpr (kDirectO) return true;  // the softmax warps wrote O themselves
                const int tt = (int)blockIdx.x + t * (int)gridDim.x;
                const int tbh = tt / nqt, tq0 = (tt % nqt) * BM;
                const unsigned char *src = sm + C::oQ + (t & 1) * C::kQBytes;
                tma_store_3d(&P.mOa, 0, tq0, tbh, src);
                if constexpr (C::DB > 0) tma_store_3d(&P.mOb, 64, tq0, tbh, src + C::kQa);
                bulk_commit_group();
                bulk_wait_group_read<0>();
                return true;
            };
            bool ok = true;
            uint32_t done_phase = 0;  // fresh mode: bit st = parity of the next DENSE_DONE[st] phase
            // abort path: per stage (bits 2st, 2st+1) and per Q buffer whether a TMA load was
            // issued into it and the barrier parity of the latest one (bit 1: issued, bit 0: parity)
            uint32_t kv_issued = 0, q_issued = 0;
            for (int it = 0; ok && it < my_tiles; ++it) {
                const int tile = (int)blockIdx.x + it * (int)gridDim.x;
                const int bh = tile / nqt, q0 = (tile % nqt) * BM;
                const bool store_tile = P.store && q0 == 0;
                const int qb = it & 1;
                unsigned char *sq = sm + C::oQ + qb * C::kQBytes;
                if (!p.fresh) {
                    if (it >= 2 && !(ok = store_o(it - 2))) break;  // the buffer still holds O of tile it - 2
                    if (!(ok = mbar_wait(&bars[Q_EMPTY + qb], ((it >> 1) & 1) ^ 1, p.status, abort_flag))) break;
                    mbar_arrive_expect_tx(&bars[Q_FULL + qb], C::kQa + C::kQb);
                    tma_load_3d(sq, &P.mQa, 0, q0, bh, &bars[Q_FULL + qb]);
                    if constexpr (C::DB > 0) tma_load_3d(sq + C::kQa, &P.mQb, 64, q0, bh, &bars[Q_FULL + qb]);
                    q_issued = (q_issued & ~(3u << (2 * qb))) | ((2u | ((it >> 1) & 1)) << (2 * qb));
                }
                for (int j = 0; j < nblk; ++j) {
                    const int g = it * nblk + j, st = g % S;
                    if (!(ok = mbar_wait(&kv_empty[st], ((g / S) & 1) ^ 1, p.status, abort_flag))) break;
                    if (p.fresh && g >= S && (g - S) % nblk < nd) {
                        // fresh mode: a stage last used by a dense block is free once the index
                        // warp has also finished with it (it fills the stage and writes the
                        // fused scatter from it)
                        if (!(ok = mbar_wait(&bars[DENSE_DONE + st], (done_phase >> st) & 1, p.status, abort_flag)))
                            break;
                        done_phase ^= 1u << st;
                    }
                    if (p.fresh && j < nd) {  // the index warp fills this stage and signals it
                        mbar_arrive(&bars[DENSE_GO + st]);
                        continue;
                    }
                    if (P.store) bulk_wait_group_read<S - 2>();  // the store of block g - S is done reading
                    unsigned char *stg = sm + C::oStage + st * C::kStageBytes;
                    uint64_t *fb = &bars[KV_FULL + st];
                    mbar_arrive_expect_tx(fb, C::kKV);
                    const bool dense = j < nd;
                    const int row = (dense ? j : j - nd) * BN;
                    tma_load_3d(stg + C::sKa, dense ? &P.mKa : &P.mKca, 0, row, bh, fb);
                    tma_load_3d(stg + C::sVa, dense ? &P.mVa : &P.mVca, 0, row, bh, fb);
                    if constexpr (C::DB > 0) {
                        tma_load_3d(stg + C::sKb, dense ? &P.mKb : &P.mKcb, 64, row, bh, fb);
                        tma_load_3d(stg + C::sVb, dense ? &P.mVb : &P.mVcb, 64, row, bh, fb);
                    }
                    kv_issued = (kv_issued & ~(3u << (2 * st))) | ((2u | ((g / S) & 1)) << (2 * st));
                    if (P.store) {
                        if (!(ok = store_pending())) break;
                        bulk_commit_group();
                        if (store_tile) {
                            pend_g = g;
                            pend_bh = bh;
                            pend_row = row;
                        }
                    }
                }
            }
            if (P.store) {
                if (ok) store_pending();
                bulk_commit_group();
            }
            for (int t = my_tiles - 2; ok && !p.fresh && t < my_tiles; ++t)
                if (t >= 0) ok = store_o(t);
            // every store has read its shared-memory source before the CTA exits (the writes
            // themselves are visible to later launches at grid completion)
            bulk_wait_group_read<0>();
            if (*abort_flag) {
                // Abort path: the loads already issued still write into the stages and Q
                // buffers; wait (bounded) until each has landed before the CTA releases its
                // shared memory. A load's phase is the latest one of its barrier, so the
                // parity wait is exact.
                for (int i = 0; i < S; ++i)
                    if ((kv_issued >> (2 * i)) & 2u) mbar_wait_drain(&bars[KV_FULL + i], (kv_issued >> (2 * i)) & 1u);
                for (int i = 0; i < 2; ++i)
                    if ((q_issued >> (2 * i)) & 2u) mbar_wait_drain(&bars[Q_FULL + i], (q_issued >> (2 * i)) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ S issuer
        // S_g = Q K_g^T once K_g has landed, Q of its tile has landed and PV_{g-SB} has
        // released S/P buffer g % SB. The whole warp runs the loop so that every descriptor
        // is warp-uniform; one elected lane issues each tcgen05 instruction.
        const uint32_t idS = idesc_bf16(BM, BN, 0, 0);
        const int total = my_tiles * nblk;
        for (int g = 0; g < total; ++g) {
            const int it = g / nblk, j = g - it * nblk;
            if (!wait_all<C::kSpin>(&bars[KV_FULL + g % S], (g / S) & 1, p.status, abort_flag)) break;
            if (j == 0 && !wait_all<C::kSpin>(&bars[Q_FULL + (it & 1)], (it >> 1) & 1, p.status, abort_flag)) break;
            if (j >= nd) {
                // A cache block: its rows at active positions are stale. Their P will be 0, but
                // 0 x NaN is NaN, so their V rows are cleared in shared memory here, before S
                // is issued (PV_g, which reads them, follows S_g through the softmax warps'
                // hand-over), unless the caller guarantees finite values there (a finite row
                // times P = 0 adds exactly 0). Whole rows are cleared, so the swizzle inside a
                // row does not matter.
                // After the clear (stores and proxy fence) this warp's next barrier test took
                // 700-1000 cycles even on a completed phase (measured); the wait for PV_{g-SB}
                // below comes after the clear and hides that.
                if (j == nd && !wait_all<C::kSpin>(&bars[BM_FULL + (it & 1)], (it >> 1) & 1, p.status, abort_flag)) break;
                const uint32_t *bm = bitmaps + (it & 1) * bm_words;
                const int pos0 = (j - nd) * BN;
                uint64_t stale = (uint64_t)bm[pos0 >> 5] | ((uint64_t)bm[(pos0 >> 5) + 1] << 32);
                if (p.N - pos0 < 64) stale &= (1ull << (p.N - pos0)) - 1ull;
                if (stale && !p.stale_finite) {
                    unsigned char *stw = sm + C::oStage + (g % S) * C::kStageBytes;
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    if constexpr (C::DB > 0) {
                        // d = 80 (two S/P buffers: the clear can delay S_g). Lane: 16-byte chunk
                        // (lane & 7) of rows (lane >> 3) + 4k of part a, chunk (lane & 1) of rows
                        // (lane >> 1) + 16k of the tail. The tests are shifts and masks of the
                        // lane's copy of the bits, every store is predicated at a constant offset
                        // from the lane's base: 20 stores and no loop or bit counts (which would
                        // take the XU pipe from the softmax's exponentials). Measured with three
                        // stages: 4% faster on the MAR-H shape than the loop below, which is 2%
                        // faster at d = 64.
                        const uint64_t sa = stale >> (lane >> 3);
                        const uint32_t alo = (uint32_t)sa, ahi = (uint32_t)(sa >> 32);
                        uint4 *va = reinterpret_cast<uint4 *>(stw + C::sVa) + 8 * (lane >> 3) + (lane & 7);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (alo & (1u << (4 * k))) va[32 * k] = z;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (ahi & (1u << (4 * k))) va[256 + 32 * k] = z;
                        const uint64_t sb = stale >> (lane >> 1);
                        const uint32_t blo = (uint32_t)sb, bhi = (uint32_t)(sb >> 32);
                        uint4 *vb = reinterpret_cast<uint4 *>(stw + C::sVb) + 2 * (lane >> 1) + (lane & 1);
                        if (blo & 1u) vb[0] = z;
                        if (blo & (1u << 16)) vb[32] = z;
                        if (bhi & 1u) vb[64] = z;
                        if (bhi & (1u << 16)) vb[96] = z;
                    } else {
                        for (int t = lane; t < BN * 8; t += 32)
                            if ((stale >> (t >> 3)) & 1ull) *reinterpret_cast<uint4 *>(stw + C::sVa + 16 * t) = z;
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
            }
            // PV_{g-SB} reads the S/P buffer that S_g overwrites (its stage is not g's: the ring
            // has more stages than S/P buffers), so the clear above need not wait for it
            if (g >= SB && !wait_all<C::kSpin>(&bars[O_DONE + g % SB], (g / SB - 1) & 1, p.status, abort_flag)) break;
            tc_fence_after();
            const unsigned char *sq = sm + C::oQ + (it & 1) * C::kQBytes;
            const unsigned char *stg = sm + C::oStage + (g % S) * C::kStageBytes;
            const uint64_t dQa = smem_desc(sq, 16, 1024, Swz::B128);
            const uint64_t dKa = smem_desc(stg + C::sKa, 16, 1024, Swz::B128);
            const uint32_t dst = tmS0 + 64 * (g % SB);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss(dst, desc_advance(dQa, 32 * k), desc_advance(dKa, 32 * k), idS, k > 0);
                if constexpr (C::DB > 0)
                    mma_ss(dst, smem_desc(sq + C::kQa, 16, 256, Swz::B32), smem_desc(stg + C::sKb, 16, 256, Swz::B32),
                           idS, 1);
                mma_commit(&bars[S_FULL + g % SB]);
                if (j == nblk - 1) mma_commit(&bars[Q_EMPTY + (it & 1)]);  // Q buffer reusable
            }
            __syncwarp();
        }
        __syncwarp();
        if (*abort_flag) {  // abort path: this warp's MMAs still write tensor memory; wait for them
            if (elect_one()) {
                mma_commit(&drain[0]);
                mbar_wait_drain(&drain[0], 0);
            }
            __syncwarp();
        }
    } else if (warp == 7) {
        // ------------------------------------------------------------ PV issuer
        // O += P_g V_g as soon as the softmax warps have written P_g; its commits release
        // the S/P buffer (O_DONE) and the K/V stage. tcgen05 operations complete in issue
        // order per issuing thread, and the S issuer orders itself after PV through O_DONE.
        const uint32_t idOa = idesc_bf16(BM, 64, 0, 1);
        const uint32_t idOb = idesc_bf16(BM, 16, 0, 1);
        const int total = my_tiles * nblk;
        for (int g = 0; g < total; ++g) {
            // V_g has landed (or lands before P_g exists: S_g needs the same stage); waiting on
            // its barrier phase orders this thread's reads after the TMA write. It comes first,
            // so that only the P_FULL wait (each wait and its vote take a few hundred cycles even
            // on a completed phase) sits between the softmax's hand-over and PV_g. The stage
            // cannot have been refilled: that needs this warp's commit below.
            if (!wait_all<C::kSpin>(&bars[KV_FULL + g % S], (g / S) & 1, p.status, abort_flag)) break;
            if (!wait_all<C::kSpin>(&bars[P_FULL + g % SB], (g / SB) & 1, p.status, abort_flag)) break;
            tc_fence_after();
            const int j = g % nblk;
            const unsigned char *stg = sm + C::oStage + (g % S) * C::kStageBytes;
            const uint64_t dVa = smem_desc(stg + C::sVa, 1024, 1024, Swz::B128);
            const uint64_t dVb = smem_desc(stg + C::sVb, 256, 256, Swz::B32);
            const uint32_t pcol = tmS0 + 64 * (g % SB);
            if (elect_one()) {
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint32_t acc = (j > 0 || k > 0) ? 1u : 0u;
                    mma_ts(tmO, pcol + 8 * k, desc_advance(dVa, 2048 * k), idOa, acc);
                    if constexpr (C::DB > 0) mma_ts(tmO + 64, pcol + 8 * k, desc_advance(dVb, 512 * k), idOb, acc);
                }
                mma_commit(&bars[O_DONE + g % SB]);
                mma_commit(&kv_empty[g % S]);
            }
            __syncwarp();
        }
        __syncwarp();
        if (*abort_flag) {  // abort path, as for the S issuer
            if (elect_one()) {
                mma_commit(&drain[1]);
                mbar_wait_drain(&drain[1], 0);
            }
            __syncwarp();
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ index warp
        // Fresh mode: the active rows of the tile's queries and of its dense key blocks are
        // copied here from the whole fresh tensors (rows bh * N + idx[b, a]), 16 bytes per
        // lane per copy, into the same swizzled layouts the TMA boxes produce: row r of a
        // 64-column part at r * 128 with its chunk c at (c ^ (r & 7)) * 16, the 16 tail
        // columns of d = 80 at r * 32 with chunk c at (c ^ ((r >> 2) & 1)) * 16. Rows past the
        // active set (and rows at out-of-range positions) are zero-filled. Each lane waits for
        // its own copies and fences them for the tensor cores before lane 0 signals the barrier.
        const bf16 *gQ = static_cast<const bf16 *>(p.Q);
        const bf16 *gK = static_cast<const bf16 *>(p.Kd);
        const bf16 *gV = static_cast<const bf16 *>(p.Vd);
        // positions of the active rows a0 + 32 k + lane (k < 4) of the rows a0 .. a0 + rows - 1
        // (rows <= 128), -1 past the active set or out of range: loaded once, then passed to
        // the copies and the scatter by shuffles (a position load inside their loops would
        // put one global-memory latency on every pass)
        auto load_pos = [&](const int32_t *ix, int a0, int rows, int (&pr)[4]) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int a = a0 + 32 * k + lane;
                const int pos = (32 * k < rows && a < p.A) ? __ldg(ix + a) : -1;
                pr[k] = (pos >= 0 && pos < p.N) ? pos : -1;
            }
        };
        // rows a0 .. a0 + rows - 1 of the active set (rows <= 128, a multiple of 32; positions
        // pr from load_pos) of one or two tensors into part a at da[n] and tail part at db[n]
        auto copy_rows = [&](const bf16 *const *src, unsigned char *const *da, unsigned char *const *db, int n,
                             const int (&pr)[4], int rows, int64_t slab) {
            for (int i = 0; i < rows / 4; ++i) {  // four rows per pass: 8 lanes per row
                const int r = 4 * i + (lane >> 3), c = lane & 7, sel = i >> 3;
                const int pos = __shfl_sync(0xffffffffu, sel == 0 ? pr[0] : sel == 1 ? pr[1] : sel == 2 ? pr[2] : pr[3],
                                            r & 31);
                const int64_t off = (slab + (pos < 0 ? 0 : pos)) * D + 8 * c;
                const uint32_t so = (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
                for (int t = 0; t < n; ++t) cp_async16(da[t] + so, src[t] + off, pos < 0 ? 0 : 16);
            }
            if constexpr (C::DB > 0) {
                for (int i = 0; i < rows / 16; ++i) {  // sixteen rows per pass: 2 lanes per row
                    const int r = 16 * i + (lane >> 1), c = lane & 1, sel = i >> 1;
                    const int pos = __shfl_sync(0xffffffffu,
                                                sel == 0 ? pr[0] : sel == 1 ? pr[1] : sel == 2 ? pr[2] : pr[3], r & 31);
                    const int64_t off = (slab + (pos < 0 ? 0 : pos)) * D + 64 + 8 * c;
                    const uint32_t so = (uint32_t)(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
                    for (int t = 0; t < n; ++t) cp_async16(db[t] + so, src[t] + off, pos < 0 ? 0 : 16);
                }
            }
        };
        // Fused scatter from a stage holding dense block a0 .. a0 + 63 (positions pr from
        // load_pos): its real rows go to the cache rows at their positions (K and V). The
        // producer refills the stage only after DENSE_DONE, which follows these reads.
        bf16 *gKc = static_cast<bf16 *>(p.Kc);
        bf16 *gVc = static_cast<bf16 *>(p.Vc);
        auto scatter_stage = [&](const unsigned char *stg, int a0, int64_t slab, const int (&pr)[4]) {
            const int nr = min(BN, p.A - a0);
            for (int i = 0; i < (nr + 3) / 4; ++i) {
                const int r = 4 * i + (lane >> 3), c = lane & 7;
                const int pos = __shfl_sync(0xffffffffu, i < 8 ? pr[0] : pr[1], r & 31);
                if (pos < 0) continue;  // past the active set (r >= nr) or out of range
                const uint32_t so = (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
                const int64_t off = (slab + pos) * D + 8 * c;
                *reinterpret_cast<uint4 *>(gKc + off) = *reinterpret_cast<const uint4 *>(stg + C::sKa + so);
                *reinterpret_cast<uint4 *>(gVc + off) = *reinterpret_cast<const uint4 *>(stg + C::sVa + so);
            }
            if constexpr (C::DB > 0) {
                for (int i = 0; i < (nr + 15) / 16; ++i) {
                    const int r = 16 * i + (lane >> 1), c = lane & 1;
                    const int pos = __shfl_sync(0xffffffffu, i < 2 ? pr[0] : pr[1], r & 31);
                    if (pos < 0) continue;
                    const uint32_t so = (uint32_t)(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
                    const int64_t off = (slab + pos) * D + 64 + 8 * c;
                    *reinterpret_cast<uint4 *>(gKc + off) = *reinterpret_cast<const uint4 *>(stg + C::sKb + so);
                    *reinterpret_cast<uint4 *>(gVc + off) = *reinterpret_cast<const uint4 *>(stg + C::sVb + so);
                }
            }
        };
        auto land = [&]() {  // this lane's copies complete and visible to the tensor cores
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
        };
        // the bitmap of tile it's active positions (double-buffered; handed to the softmax
        // warps when the tile has cache blocks), with the positions checked
        auto build_bitmap = [&](int it, int b) -> bool {
            const int bb = it & 1;
            uint32_t *bm = bitmaps + bb * bm_words;
            if (nc > 0 && !wait_all<C::kSpin>(&bars[BM_EMPTY + bb], ((it >> 1) & 1) ^ 1, p.status, abort_flag)) return false;
            for (int w = lane; w < bm_words; w += 32) bm[w] = 0u;
            __syncwarp();
            uint32_t bad = 0;
            for (int a = lane; a < p.A; a += 32) {
                const int pos = p.idx[(int64_t)b * p.A + a];
                if (pos < 0 || pos >= p.N) {
                    bad |= MAR_STATUS_INDEX_RANGE;
                    continue;
                }
                const uint32_t old = atomicOr(&bm[pos >> 5], 1u << (pos & 31));
                if (old & (1u << (pos & 31))) bad |= MAR_STATUS_INDEX_DUP;
            }
            if (bad) report(p.status, bad);
            __syncwarp();
            if (nc > 0 && lane == 0) mbar_arrive(&bars[BM_FULL + bb]);
            return true;
        };
        // fresh mode: this warp owns the Q buffers, so it also stores each tile's staged O
        auto store_o6 = [&](int t) -> bool {
            if (!wait_all<C::kSpin>(&bars[O_STAGED + (t & 1)], (t >> 1) & 1, p.status, abort_flag)) return false;
            if (!kDirectO && lane == 0) {
                const int tt = (int)blockIdx.x + t * (int)gridDim.x;
                const int tbh = tt / nqt, tq0 = (tt % nqt) * BM;
                const unsigned char *src = sm + C::oQ + (t & 1) * C::kQBytes;
                tma_store_3d(&P.mOa, 0, tq0, tbh, src);
                if constexpr (C::DB > 0) tma_store_3d(&P.mOb, 64, tq0, tbh, src + C::kQa);
                bulk_commit_group();
                bulk_wait_group_read<0>();
            }
            __syncwarp();
            return true;
        };
        if (kGen) {
            // generating positions out of range: reported once per batch row (its first tile
            // of head 0); such a slot has no row and adds nothing to the score
            for (int it = 0; it < my_tiles; ++it) {
                const int tile = (int)blockIdx.x + it * (int)gridDim.x;
                const int bh = tile / nqt, q0 = (tile % nqt) * BM;
                if (q0 != 0 || bh % p.H != 0) continue;
                bool bad = false;
                for (int gg = lane; gg < p.G; gg += 32)
                    bad |= (unsigned)__ldg(p.gen + (int64_t)(bh / p.H) * p.G + gg) >= (unsigned)p.N;
                if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.status, MAR_STATUS_INDEX_RANGE);
            }
        } else if (P.gather && p.fresh) {
            bool ok = true;
            uint32_t go_phase = 0;  // bit st: parity of the next DENSE_GO[st] phase
            for (int it = 0; ok && it < my_tiles; ++it) {
                const int tile = (int)blockIdx.x + it * (int)gridDim.x;
                const int bh = tile / nqt, qt = tile % nqt, b = bh / p.H;
                const int qb = it & 1, q0 = qt * BM;
                const int32_t *ix = p.idx + (int64_t)b * p.A;
                const int64_t slab = (int64_t)bh * p.N;
                // the buffer holds O of tile it - 2 (all of that tile's MMAs are complete)
                if (it >= 2 && !(ok = store_o6(it - 2))) break;
                {
                    unsigned char *sq = sm + C::oQ + qb * C::kQBytes;
                    unsigned char *sqb = sq + C::kQa;
                    // whole warps of query rows (those of a warp with no real row are never read)
                    const int rows = min(BM, (p.nq - q0 + 31) & ~31);
                    int pq[4];
                    load_pos(ix, q0, rows, pq);
                    copy_rows(&gQ, &sq, &sqb, 1, pq, rows, slab);
                }
                for (int j = 0; j < nd; ++j) {
                    const int g = it * nblk + j, st = g % S;
                    if (!(ok = wait_all<C::kSpin>(&bars[DENSE_GO + st], (go_phase >> st) & 1, p.status, abort_flag))) break;
                    go_phase ^= 1u << st;
                    unsigned char *stg = sm + C::oStage + st * C::kStageBytes;
                    const bf16 *src[2] = {gK, gV};
                    unsigned char *da[2] = {stg + C::sKa, stg + C::sVa};
                    unsigned char *db[2] = {stg + C::sKb, stg + C::sVb};
                    int pk[4];
                    load_pos(ix, j * BN, BN, pk);
                    copy_rows(src, da, db, 2, pk, BN, slab);
                    land();
                    if (lane == 0) {
                        if (j == 0) mbar_arrive(&bars[Q_FULL + qb]);
                        mbar_arrive(&bars[KV_FULL + st]);
                    }
                    // the bitmap is read from the first cache block on; the positions are
                    // checked even when there is none (A == N)
                    if (j == 0 && !(ok = build_bitmap(it, b))) break;
                    if (p.fuse_scatter && qt == 0 && !P.idle_scatter) scatter_stage(stg, j * BN, slab, pk);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[DENSE_DONE + st]);
                }
            }
            for (int t = my_tiles - 2; ok && t < my_tiles; ++t)
                if (t >= 0) ok = store_o6(t);
            if (lane == 0) bulk_wait_group_read<0>();
        } else if (P.gather) {
            bool ok = true;
            for (int it = 0; ok && it < my_tiles; ++it) {
                const int tile = (int)blockIdx.x + it * (int)gridDim.x;
                const int bh = tile / nqt, qt = tile % nqt, b = bh / p.H;
                // with no cache blocks (A == N) nothing reads the bitmap
                if (nc > 0 && !(ok = build_bitmap(it, b))) break;
                if (!p.fuse_scatter || qt != 0 || P.idle_scatter) continue;
                // Fresh K_A/V_A rows -> cache rows of the active positions. No query of this
                // launch uses those rows (they are masked as stale). The rows are copied 32 at a
                // time: each lane loads one row's position, which the copies take by shuffles;
                // eight 16-byte chunks per lane and pass, all loads before the stores, so that
                // the passes are not serialised on the load latency.
                const bf16 *Kd = static_cast<const bf16 *>(p.Kd);
                const bf16 *Vd = static_cast<const bf16 *>(p.Vd);
                constexpr int CH = D / 8;  // 16-byte chunks per row
                constexpr int kU = 8;
                for (int a0 = 0; a0 < p.A; a0 += 32) {
                    const int nr = min(32, p.A - a0);
                    int posl = lane < nr ? __ldg(p.idx + (int64_t)b * p.A + a0 + lane) : -1;
                    if (posl >= p.N) posl = -1;
                    for (int t0 = 0; t0 < nr * CH; t0 += 32 * kU) {
                        uint4 kv[kU], vv[kU];
                        int64_t dst[kU];
#pragma unroll
                        for (int u = 0; u < kU; ++u) {
                            const int t = t0 + 32 * u + lane;
                            const int r = t / CH, c = t % CH;
                            const int pos = __shfl_sync(0xffffffffu, posl, r & 31);
                            dst[u] = -1;
                            if (t < nr * CH && pos >= 0) {
                                const int64_t src = ((int64_t)bh * p.A + a0 + r) * D + 8 * c;
                                kv[u] = __ldg(reinterpret_cast<const uint4 *>(Kd + src));
                                vv[u] = __ldg(reinterpret_cast<const uint4 *>(Vd + src));
                                dst[u] = ((int64_t)bh * p.N + pos) * D + 8 * c;
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kU; ++u)
                            if (dst[u] >= 0) {
                                *reinterpret_cast<uint4 *>(gKc + dst[u]) = kv[u];
                                *reinterpret_cast<uint4 *>(gVc + dst[u]) = vv[u];
                            }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const float sl2 = p.scale * kLog2e;
        bool ok = true;
        // The fused scatter of dense block a0 .. a0 + 63 from its stage by the warps without a
        // live row (warps first_idle .. 3, T threads): each thread takes every T-th of the
        // block's (row, 16-byte chunk) pieces, eight at a time, positions loaded first.
        auto scatter_idle = [&](const unsigned char *stg, int bh, int a0) {
            constexpr int CH = D / 8;  // 16-byte chunks per row: 8 in part a, then the tail's
            constexpr int kU = 8;
            const int first_idle = (p.nq + 31) >> 5;
            const int t0 = (warp - first_idle) * 32 + lane, T = (4 - first_idle) * 32;
            const int nr = min(BN, p.A - a0), b = bh / p.H;
            const int32_t *ix = p.idx + (int64_t)b * p.A + a0;
            bf16 *Kc = static_cast<bf16 *>(p.Kc);
            bf16 *Vc = static_cast<bf16 *>(p.Vc);
            for (int u0 = t0; u0 < nr * CH; u0 += kU * T) {
                int pos[kU];
#pragma unroll
                for (int k = 0; k < kU; ++k) {
                    const int u = u0 + k * T;
                    pos[k] = u < nr * CH ? __ldg(ix + u / CH) : -1;
                }
#pragma unroll
                for (int k = 0; k < kU; ++k) {
                    const int u = u0 + k * T;
                    if (pos[k] < 0 || pos[k] >= p.N) continue;
                    const int r = u / CH, c = u - r * CH;
                    uint32_t sa, sv;
                    int64_t off;
                    if (c < 8) {
                        const uint32_t so = (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
                        sa = C::sKa + so;
                        sv = C::sVa + so;
                        off = ((int64_t)bh * p.N + pos[k]) * D + 8 * c;
                    } else {
                        const int cb = c - 8;
                        const uint32_t so = (uint32_t)(r * 32 + ((cb ^ ((r >> 2) & 1)) << 4));
                        sa = C::sKb + so;
                        sv = C::sVb + so;
                        off = ((int64_t)bh * p.N + pos[k]) * D + 64 + 8 * cb;
                    }
                    *reinterpret_cast<uint4 *>(Kc + off) = *reinterpret_cast<const uint4 *>(stg + sa);
                    *reinterpret_cast<uint4 *>(Vc + off) = *reinterpret_cast<const uint4 *>(stg + sv);
                }
            }
        };
        int gpos_next = -1;  // full attention with the score: gen[b, lane] of the next tile
        if constexpr (kGen)
            if (my_tiles > 0)
                gpos_next = lane < p.G ? __ldg(p.gen + (int64_t)((int)blockIdx.x / nqt / p.H) * p.G + lane) : -1;
        for (int it = 0; ok && it < my_tiles; ++it) {
            const int tile = (int)blockIdx.x + it * (int)gridDim.x;
            const int bh = tile / nqt, q0 = (tile % nqt) * BM;
            const bool live = (q0 + 32 * warp) < p.nq;  // warp-uniform: some row of this warp is real
            const uint32_t *bm = bitmaps + (it & 1) * bm_words;
            float m_use = 0.f, l = 0.f;
            // full attention with the layer-2 score: the generating slots g this row serves
            // full attention with the layer-2 score: the first generating slot this row serves
            // (a position listed twice is stored once; the reduction reads it for both slots).
            // Its raw scores go to gen_s row (bh, slot) by predicated stores, so that the other
            // threads run the same instructions and the block loop keeps one shape.
            float *gdst = nullptr;
            uint32_t is_gen = 0, gslot = 0;
            if constexpr (kGen) {
                // lane l holds gen[b, l] of this tile's batch row (loaded one tile ahead); the
                // row's slot is the lowest l whose position is the row
                const int pos_cur = gpos_next;
                if (it + 1 < my_tiles) {
                    const int nb = ((int)blockIdx.x + (it + 1) * (int)gridDim.x) / nqt / p.H;
                    gpos_next = lane < p.G ? __ldg(p.gen + (int64_t)nb * p.G + lane) : -1;
                }
                int slot = -1;
                for (int gg = p.G - 1; gg >= 0; --gg)
                    if (__shfl_sync(0xffffffffu, pos_cur, gg) == q0 + tid) slot = gg;
                is_gen = slot >= 0;
                gslot = is_gen ? (uint32_t)slot : 0u;
                gdst = p.gen_s + ((int64_t)bh * p.G + gslot) * p.N;
            }
            for (int j = 0; j < nblk; ++j) {
                const int g = it * nblk + j, buf = g % SB;
                if (j == nd && nc > 0 &&
                    !(ok = wait_all<C::kSpin>(&bars[BM_FULL + (it & 1)], (it >> 1) & 1, p.status, abort_flag)))
                    break;
                if (!(ok = wait_all<C::kSpin>(&bars[S_FULL + buf], (g / SB) & 1, p.status, abort_flag))) break;
                tc_fence_after();
                // slots of this block that are keys: dense rows below n_dense; cache rows below
                // N whose position is not active (active positions hold stale cache rows, whose
                // V rows the S issuer has cleared)
                uint64_t valid;
                if (j < nd) {
                    const int r = p.n_dense - j * BN;
                    valid = r >= 64 ? ~0ull : ((1ull << r) - 1ull);
                } else {
                    const int pos0 = (j - nd) * BN;
                    valid = ~((uint64_t)bm[pos0 >> 5] | ((uint64_t)bm[(pos0 >> 5) + 1] << 32));
                    const int r = p.N - pos0;
                    if (r < 64) valid &= (1ull << r) - 1ull;
                }
                if (live) {
                    float v[64];
                    tmem_ld64(lane_addr(tmS0, warp, 64 * buf), v);
                    if constexpr (kGen) {  // N % 4 == 0: the block's columns in whole float4s
                        const int ncol = p.N - j * BN;
                        if (ncol >= 64) {
                            if constexpr (kGen == 2)
                                st_global_row64_v8_if(is_gen, gdst + j * BN, v);
                            else
                                st_global_row64_if(is_gen, gdst + j * BN, v);
                        } else {  // the ragged last block (the same branch for every thread)
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                st_global_v4_if(is_gen && 4 * i < ncol, gdst + j * BN + 4 * i, v[4 * i],
                                                v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        }
                    }
                    if (valid != ~0ull) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] = ((valid >> i) & 1ull) ? v[i] : -INFINITY;
                    }
                    // row max of the raw scores (the scale is positive), four independent chains
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < 32; ++i) m4[i & 3] = max3f(m4[i & 3], v[2 * i], v[2 * i + 1]);
                    const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
                    bool rescale = false;
                    float factor = 1.f;
                    if (j == 0) {
                        m_use = (mx == -INFINITY) ? 0.f : mx;
                    } else if (mx > m_use + kRescale) {
                        factor = fast_exp2(m_use - mx);
                        m_use = mx;
                        rescale = true;
                    }
                    // P = 2^(s * scale * log2(e) - m) as bf16 pairs over S, one half at a time;
                    // one packed FMA forms both exponents of a pair
                    const f32x2 sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
                    f32x2 rsa = f2_pack(0.f, 0.f), rsb = rsa;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(v[32 * h + 2 * i], v[32 * h + 2 * i + 1]), sc2, nm2), x0, x1);
                            const f32x2 e = f2_pack(fast_exp2(x0), fast_exp2(x1));
                            if (i & 1) rsb = f2_add(rsb, e); else rsa = f2_add(rsa, e);
                            float p0, p1;
                            f2_unpack(e, p0, p1);
                            w[i] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16(lane_addr(tmS0, warp, 64 * buf + 16 * h), w);
                    }
                    float rs0, rs1;
                    f2_unpack(f2_add(rsa, rsb), rs0, rs1);
                    l = l * factor + (rs0 + rs1);
                    if (__any_sync(0xffffffffu, rescale)) {
                        // O holds the tile's sum over earlier blocks; wait for PV_{g-1} and
                        // scale the rows that raised their max (the others use factor 1).
                        // PV_g, which adds this block, is issued only after P_FULL below.
                        ok = wait_all<C::kSpin>(&bars[O_DONE + (g - 1) % SB], ((g - 1) / SB) & 1, p.status, abort_flag);
                        if (ok) {
                            tc_fence_after();
#pragma unroll
                            for (int c0 = 0; c0 < D; c0 += 16) {
                                float o[16];
                                tmem_ld16(lane_addr(tmO, warp, c0), o);
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] *= factor;
                                tmem_st16(lane_addr(tmO, warp, c0), o);
                            }
                        }
                    }
                    tmem_wait_st();
                } else if (P.idle_scatter && j < nd) {
                    // A warp with no live row (the tile has at most 96 queries, and it is the
                    // (b, h)'s only tile) writes the fused scatter of this dense block from its
                    // stage: the fresh K/V rows of the active positions to the cache. The stage
                    // stays put until the block's PV, which waits for this warp's arrival below.
                    if (!(ok = wait_all<C::kSpin>(&bars[KV_FULL + g % S], (g / S) & 1, p.status, abort_flag))) break;
                    scatter_idle(sm + C::oStage + (g % S) * C::kStageBytes, bh, j * BN);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // P (and a rescaled O) is in tensor memory, complete after tcgen05.wait::st and
                    // ordered by the tcgen05 fences: the arrival need not release this thread's
                    // global stores (the raw scores of a generating row), whose visibility a
                    // release arrival would wait for on every block
                    mbar_arrive_relaxed(&bars[P_FULL + buf]);
                    if (j == nblk - 1 && nc > 0) mbar_arrive(&bars[BM_EMPTY + (it & 1)]);
                }
                if (!ok) break;
            }
            if (!ok) break;
            // The previous phase of this barrier (PV_{gl-SB}) completed before S_gl was
            // issued, so the parity wait is exact; MMAs complete in order, so PV_gl's
            // completion covers all of the tile's PVs.
            const int gl = it * nblk + nblk - 1;
            if (!(ok = wait_all<C::kSpin>(&bars[O_DONE + gl % SB], (gl / SB) & 1, p.status, abort_flag))) break;
            tc_fence_after();
            if (live) {
                // normalised O, staged as bf16 in this tile's Q buffer (free: the tile's last S
                // has completed) in the layout of the TMA boxes: row r of the 64-column part at
                // r * 128 with its 16-byte chunk c at (c ^ (r & 7)) * 16 (128-byte swizzle); the
                // 16 tail columns of d = 80 at r * 32, chunk c at (c ^ ((r >> 2) & 1)) * 16
                // (32-byte swizzle). The producer stores the tile (rows past nq are clipped).
                const int row = q0 + tid, r = tid;
                const float inv = 1.f / l;
                unsigned char *stage = sm + C::oQ + (it & 1) * C::kQBytes;
                if constexpr (kDirectO) {
                    // a cache-aware launch: each thread writes its own row of O (160 bytes at
                    // d = 80) straight to global memory; no staging, proxy fence or TMA store
                    uint4 *orow = reinterpret_cast<uint4 *>(static_cast<bf16 *>(p.O) + ((int64_t)bh * p.nq + row) * D);
                    const bool w = row < p.nq;
                    {
                        float o[64];
                        tmem_ld64(lane_addr(tmO, warp, 0), o);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint4 u;
                            u.x = pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv);
                            u.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                            u.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                            u.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                            if (w) orow[c] = u;
                        }
                    }
                    if constexpr (C::DB > 0) {
                        float o[16];
                        tmem_ld16(lane_addr(tmO, warp, 64), o);
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint4 u;
                            u.x = pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv);
                            u.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                            u.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                            u.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                            if (w) orow[8 + c] = u;
                        }
                    }
                } else {
                {  // the 64-column part: one tensor-memory load, eight 16-byte chunks
                    float o[64];
                    tmem_ld64(lane_addr(tmO, warp, 0), o);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 u;
                        u.x = pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv);
                        u.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                        u.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                        u.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                        *reinterpret_cast<uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4)) = u;
                    }
                }
                if constexpr (C::DB > 0) {  // the 16 tail columns
                    float o[16];
                    tmem_ld16(lane_addr(tmO, warp, 64), o);
                    unsigned char *tail = stage + C::kQa;
                    const int sw = (r >> 2) & 1;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint4 u;
                        u.x = pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv);
                        u.y = pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                        u.z = pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                        u.w = pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                        *reinterpret_cast<uint4 *>(tail + r * 32 + ((c ^ sw) << 4)) = u;
                    }
                }
                }
                if (p.lse && row < p.nq) p.lse[(int64_t)bh * p.nq + row] = (m_use + log2f(l)) * kLn2;
                if constexpr (kGen)
                    if (is_gen) p.gen_ml[(int64_t)bh * p.G + gslot] = make_float2(m_use, l);
            }
            if constexpr (!kDirectO) fence_proxy_async_smem();  // the staged rows, for the TMA store
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[O_STAGED + (it & 1)]);
            // The next tile's first PV overwrites O only after P of its first block, which
            // this warp group writes after the reads above have completed.
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

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

template <int D, int QR>
cudaError_t launch(const AttnParams &p, cudaStream_t s) {
    using C = Cfg<D, QR>;
    static int configured[64] = {0}, configured_gen[64] = {0}, configured_gen8[64] = {0}, configured_ca[64] = {0};
    Tc5Params<D> P;
    P.a = p;
    P.gather = p.idx ? 1 : 0;
    const int bh = p.B * p.H;
    const uint32_t tw = D == 64 ? 64 : 16;  // tail box width (the tail maps are unused for d = 64)
    if (QR < BM && p.nq > QR) return cudaErrorInvalidValue;
    bool ok = map3<D>(&P.mOa, p.O, p.nq, bh, 64, QR) && map3<D>(&P.mOb, p.O, p.nq, bh, tw, QR);
    if (p.fresh) {
        // the index warp copies the active rows; these maps over the whole fresh tensors are
        // only prefetched, never loaded from
        if (!p.idx || p.nq != p.A || p.n_dense != p.A) return cudaErrorInvalidValue;
        ok = ok && map3<D>(&P.mQa, p.Q, p.N, bh, 64, QR) && map3<D>(&P.mQb, p.Q, p.N, bh, tw, QR);
        ok = ok && map3<D>(&P.mKa, p.Kd, p.N, bh, 64, BN) && map3<D>(&P.mKb, p.Kd, p.N, bh, tw, BN);
        ok = ok && map3<D>(&P.mVa, p.Vd, p.N, bh, 64, BN) && map3<D>(&P.mVb, p.Vd, p.N, bh, tw, BN);
    } else {
        ok = ok && map3<D>(&P.mQa, p.Q, p.nq, bh, 64, QR) && map3<D>(&P.mQb, p.Q, p.nq, bh, tw, QR);
        ok = ok && map3<D>(&P.mKa, p.Kd, p.n_dense, bh, 64, BN) && map3<D>(&P.mKb, p.Kd, p.n_dense, bh, tw, BN);
        ok = ok && map3<D>(&P.mVa, p.Vd, p.n_dense, bh, 64, BN) && map3<D>(&P.mVb, p.Vd, p.n_dense, bh, tw, BN);
    }
    P.store = (!P.gather && p.store_kv) ? 1 : 0;
    if (P.gather || P.store) {
        ok = ok && map3<D>(&P.mKca, p.Kc, p.N, bh, 64, BN) && map3<D>(&P.mKcb, p.Kc, p.N, bh, tw, BN);
        ok = ok && map3<D>(&P.mVca, p.Vc, p.N, bh, 64, BN) && map3<D>(&P.mVcb, p.Vc, p.N, bh, tw, BN);
    } else {
        P.mKca = P.mKa; P.mKcb = P.mKb; P.mVca = P.mVa; P.mVcb = P.mVb;
    }
    if (!ok) return cudaErrorInvalidValue;
    const long long tiles = (long long)((p.nq + BM - 1) / BM) * bh;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    P.n_tiles = (int)tiles;
    // A single query tile per (b, h) with at most 96 queries leaves softmax warps without a
    // live row; they write the fused scatter in place of the index warp where that warp's
    // per-tile work (the bitmap, in-launch copies and the scatter) is a large share of a
    // tile: short tiles (at most 8 key blocks) and a steady state (at least 4 tiles per CTA).
    // Measured per call: MAR-H (6 blocks, 27 tiles per CTA) 336 -> 318 us, MAR-L shape
    // 152 -> 144 us; slower with 18 blocks per tile (512 px, A = 66: 232 -> 243 us) and with
    // 2.5 tiles per CTA (MAR-B: 33.0 -> 34.9 us). The idle warps' share is A x d / 8 16-byte
    // chunks of each of K and V per tile, written in batches behind dependent position loads,
    // and it delays their hand-over of each dense block: with one idle warp, 20 chunks per lane
    // (MAR-L shape, A = 80) still measured faster there (167 against 193 us), 30 (MAR-H shape,
    // A = 96) slower (528 against 422 us), so the share is capped at 24 chunks per lane.
    {
        const int nblk = (p.n_dense + BN - 1) / BN + ((P.gather && p.A < p.N) ? (p.N + BN - 1) / BN : 0);
        const long long ctas = tiles < 2LL * sm_count() ? tiles : 2LL * sm_count();
        const int idle_warps = 4 - (p.nq + 31) / 32;
        const bool share_ok = idle_warps > 0 && (long long)p.A * (D / 8) <= 24LL * 32 * idle_warps;
        P.idle_scatter =
            (P.gather && p.fuse_scatter && p.nq <= 96 && share_ok && nblk <= 8 && tiles >= 4 * ctas) ? 1 : 0;
    }
    size_t smem = 1024 + C::oBars + 8 * (KV_FULL + 2 * C::kStages + 2) + 16;
    smem += sizeof(uint32_t) * 2 * 2 * ((p.N + BN - 1) / BN);  // two bitmaps
    const bool gen = p.gen != nullptr && !P.gather;
    if (gen && (p.G < 1 || p.G > 32)) return cudaErrorInvalidValue;  // one generating slot per lane
    if (QR < BM && gen) return cudaErrorInvalidValue;                 // (the score forms use BM rows)
    // 32-byte raw-score stores when every row and block of the score buffer starts on a
    // 32-byte boundary (row starts are multiples of 4 N bytes, block starts of 256 bytes)
    const bool gen8 = gen && (p.N % 8) == 0 && (reinterpret_cast<uintptr_t>(p.gen_s) % 32) == 0;
    const long long grid = tiles < 2LL * sm_count() ? tiles : 2LL * sm_count();
    if constexpr (QR == BM) {
        if (gen8 || gen) {
            cudaError_t e = gen8 ? ensure_smem(attn_tc5_kernel<D, 2, QR, false>, smem, configured_gen8, /*max_carveout=*/true)
                                 : ensure_smem(attn_tc5_kernel<D, 1, QR, false>, smem, configured_gen, /*max_carveout=*/true);
            if (e != cudaSuccess) return e;
            if (gen8)
                attn_tc5_kernel<D, 2, QR, false><<<(unsigned)grid, kThreads, smem, s>>>(P);
            else
                attn_tc5_kernel<D, 1, QR, false><<<(unsigned)grid, kThreads, smem, s>>>(P);
            return cudaGetLastError();
        }
        if (!p.idx) {  // full attention: O staged for a TMA store (direct stores measured slower)
            cudaError_t e = ensure_smem(attn_tc5_kernel<D, 0, QR, false>, smem, configured, /*max_carveout=*/true);
            if (e != cudaSuccess) return e;
            attn_tc5_kernel<D, 0, QR, false><<<(unsigned)grid, kThreads, smem, s>>>(P);
            return cudaGetLastError();
        }
    }
    // cache-aware attention (the only kind with QR < BM): O rows written by the softmax warps
    if (!p.idx) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem(attn_tc5_kernel<D, 0, QR, true>, smem, configured_ca, /*max_carveout=*/true);
    if (e != cudaSuccess) return e;
    attn_tc5_kernel<D, 0, QR, true><<<(unsigned)grid, kThreads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace

// attn_tc5_q96.cu includes this file for the kernel and launch templates only.
#ifndef MAR_TC5_EXTRA_TU
bool attn_tc5_supported(const AttnParams &p) { return p.d == 64 || p.d == 80; }

cudaError_t launch_attn_bf16_tc5(const AttnParams &p, cudaStream_t s) {
    // cache-aware launches of at most 64 (96) queries keep 64-row (96-row) Q buffers and one
    // more K/V stage
    const bool q64 = p.nq <= 64 && p.idx;
    if (!q64 && p.nq <= 96 && p.idx) return launch_attn_bf16_tc5_q96(p, s);  // 96-row Q buffers
    if (p.d == 64) return q64 ? launch<64, 64>(p, s) : launch<64, BM>(p, s);
    if (p.d == 80) return q64 ? launch<80, 64>(p, s) : launch<80, BM>(p, s);
    return cudaErrorInvalidValue;
}
#endif  // MAR_TC5_EXTRA_TU

}  // namespace mar
