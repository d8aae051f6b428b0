// bf16 attention with warp-level tensor-core MMA (mma.sync m16n8k16, fp32 accumulate).
//
// Serves both full attention and cache-aware attention (see attn.h for the key list).
// MARché notes, Key Design 2: the active queries' scores against the fresh K_A/V_A
// and against the stored cached K/V are two partial softmax sums merged on chip by
// the safe online-softmax rule (running max, running sum), without concatenating
// the two key sets in memory. Here the key list is streamed in blocks of 64 rows:
// dense rows first, then the cached rows named by the in-shared-memory list of
// cached positions (built from idx; cache rows of active positions are never read).
// Each block updates the running (m, l, O) of every query row: O <- O * 2^(m-m') +
// P V with P = 2^(s*scale*log2e - m').
//
// CTA = 4 warps x 16 query rows; K/V blocks double-buffered with cp.async.
#include <cmath>

#include "attn.h"
#include "common.cuh"

namespace mar {
namespace {

constexpr int BM = 64;   // query rows per CTA
constexpr int BN = 64;   // keys per block
constexpr int kThreads = 128;

template <int D>
struct Smem {
    static constexpr int LD = D + 8;  // padded row stride (elements): conflict-free ldmatrix
    static constexpr size_t q_elems = (size_t)BM * LD;
    static constexpr size_t kv_elems = (size_t)BN * LD;
    static constexpr size_t bytes_tiles = (q_elems + 4 * kv_elems) * sizeof(bf16);
};

template <int D>
__global__ void __launch_bounds__(kThreads) attn_mma_kernel(const AttnParams p) {
    constexpr int LD = Smem<D>::LD;
    constexpr int KCH = D / 8;   // 16-byte chunks per row
    constexpr int KS = D / 16;   // k-steps of QK^T
    constexpr int NT = D / 8;    // n-tiles of the output
    extern __shared__ __align__(128) unsigned char smem_raw[];
    bf16 *sQ = reinterpret_cast<bf16 *>(smem_raw);
    bf16 *sK = sQ + Smem<D>::q_elems;
    bf16 *sV = sK + 2 * Smem<D>::kv_elems;
    int32_t *sList = reinterpret_cast<int32_t *>(sV + 2 * Smem<D>::kv_elems);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nqt = (p.nq + BM - 1) / BM;
    const int qt = blockIdx.x % nqt, bh = blockIdx.x / nqt, b = bh / p.H;
    const int q0 = qt * BM;
    const bf16 *__restrict__ Q = static_cast<const bf16 *>(p.Q);
    const bf16 *__restrict__ Kd = static_cast<const bf16 *>(p.Kd);
    const bf16 *__restrict__ Vd = static_cast<const bf16 *>(p.Vd);
    bf16 *Kc = static_cast<bf16 *>(p.Kc);
    bf16 *Vc = static_cast<bf16 *>(p.Vc);

    int C = 0;
    if (p.idx) {
        uint32_t *bitmap = reinterpret_cast<uint32_t *>(sList + p.N);
        int32_t *wt = reinterpret_cast<int32_t *>(bitmap + ((p.N + 31) >> 5));
        C = build_cached_list(p.idx + (int64_t)b * p.A, p.A, p.N, bitmap, sList, wt, p.status);
        if (p.fuse_scatter && qt == 0) {
            // Fresh K_A/V_A rows -> cache rows of the active positions (never read here).
            for (int t = tid; t < p.A * KCH; t += kThreads) {
                int a = t / KCH, c = t % KCH;
                int pos = p.idx[(int64_t)b * p.A + a];
                if (pos < 0 || pos >= p.N) continue;
                const int64_t src = dense_row(p, bh, b, a, p.n_dense) * D + 8 * c;
                const int64_t dst = ((int64_t)bh * p.N + pos) * D + 8 * c;
                *reinterpret_cast<uint4 *>(Kc + dst) = *reinterpret_cast<const uint4 *>(Kd + src);
                *reinterpret_cast<uint4 *>(Vc + dst) = *reinterpret_cast<const uint4 *>(Vd + src);
            }
        }
    }
    const int n_keys = p.n_dense + C;
    const int nblk = (n_keys + BN - 1) / BN;

    // Query tile: rows past nq are zero-filled.
    for (int c = tid; c < BM * KCH; c += kThreads) {
        int r = c / KCH, ch = c % KCH, row = q0 + r;
        const bf16 *src = Q + dense_row(p, bh, b, row < p.nq ? row : 0, p.nq) * D + 8 * ch;
        cp_async16(sQ + r * LD + 8 * ch, src, row < p.nq ? 16 : 0);
    }
    auto load_kv = [&](int blk, int buf) {
        bf16 *dk = sK + buf * Smem<D>::kv_elems, *dv = sV + buf * Smem<D>::kv_elems;
        for (int c = tid; c < BN * KCH; c += kThreads) {
            int r = c / KCH, ch = c % KCH, t = blk * BN + r;
            const bf16 *ks = Kd, *vs = Vd;
            int bytes = 16;
            if (t < p.n_dense) {
                const int64_t r = dense_row(p, bh, b, t, p.n_dense);
                ks = Kd + r * D + 8 * ch;
                vs = Vd + r * D + 8 * ch;
            } else if (t < n_keys) {
                int pos = sList[t - p.n_dense];
                ks = Kc + ((int64_t)bh * p.N + pos) * D + 8 * ch;
                vs = Vc + ((int64_t)bh * p.N + pos) * D + 8 * ch;
            } else {
                bytes = 0;  // past the key list: zero-fill (finite), masked below
            }
            cp_async16(dk + r * LD + 8 * ch, ks, bytes);
            cp_async16(dv + r * LD + 8 * ch, vs, bytes);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    const bool warp_live = (q0 + warp * 16) < p.nq;
    const float sl2 = p.scale * kLog2e;
    uint32_t qf[KS][4];
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int blk = 0; blk < nblk; ++blk) {
        if (blk + 1 < nblk) load_kv(blk + 1, (blk + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (blk == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const bf16 *a = sQ + (warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LD +
                                ks * 16 + 8 * (lane >> 4);
                ldmatrix_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], a);
            }
        }
        if (warp_live) {
            const bf16 *ksm = sK + (blk & 1) * Smem<D>::kv_elems;
            const bf16 *vsm = sV + (blk & 1) * Smem<D>::kv_elems;
            float s[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const bf16 *kp = ksm + (np * 16 + (lane & 7) + 8 * (lane >> 4)) * LD + ks * 16 +
                                     8 * ((lane >> 3) & 1);
                    ldmatrix_x4(b0, b1, b2, b3, kp);
                    mma_bf16_16816(s[2 * np], qf[ks], b0, b1);
                    mma_bf16_16816(s[2 * np + 1], qf[ks], b2, b3);
                }
            }
            // scale into the log2 domain, mask keys past the list, block row max
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int key = blk * BN + n * 8 + 2 * (lane & 3) + (e & 1);
                    s[n][e] = (key < n_keys) ? s[n][e] * sl2 : -INFINITY;
                }
                mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
                mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
            const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                s[n][0] = fast_exp2(s[n][0] - mu0);
                s[n][1] = fast_exp2(s[n][1] - mu0);
                s[n][2] = fast_exp2(s[n][2] - mu1);
                s[n][3] = fast_exp2(s[n][3] - mu1);
                rs0 += s[n][0] + s[n][1];
                rs1 += s[n][2] + s[n][3];
            }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= al0; o[n][1] *= al0;
                o[n][2] *= al1; o[n][3] *= al1;
            }
            // O += P V  (P from registers as the A operand, V via transposed ldmatrix)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t a[4];
                a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
                a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
                a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
                for (int dp = 0; dp < NT / 2; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    const bf16 *vp = vsm + (kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LD +
                                     dp * 16 + 8 * (lane >> 4);
                    ldmatrix_x4_trans(b0, b1, b2, b3, vp);
                    mma_bf16_16816(o[2 * dp], a, b0, b1);
                    mma_bf16_16816(o[2 * dp + 1], a, b2, b3);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    if (!warp_live) return;
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const int r0 = q0 + warp * 16 + (lane >> 2), r1 = r0 + 8;
    bf16 *O = static_cast<bf16 *>(p.O);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int col = n * 8 + 2 * (lane & 3);
        if (r0 < p.nq)
            *reinterpret_cast<uint32_t *>(O + ((int64_t)bh * p.nq + r0) * D + col) =
                pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
        if (r1 < p.nq)
            *reinterpret_cast<uint32_t *>(O + ((int64_t)bh * p.nq + r1) * D + col) =
                pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
    }
    if (p.lse && (lane & 3) == 0) {
        if (r0 < p.nq) p.lse[(int64_t)bh * p.nq + r0] = (m0 + log2f(l0)) * kLn2;
        if (r1 < p.nq) p.lse[(int64_t)bh * p.nq + r1] = (m1 + log2f(l1)) * kLn2;
    }
}

template <int D>
cudaError_t launch(const AttnParams &p, cudaStream_t s) {
    static int configured[64] = {0};
    size_t smem = Smem<D>::bytes_tiles;
    if (p.idx) smem += sizeof(int32_t) * (p.N + (p.N + 31) / 32 + kThreads / 32);
    cudaError_t e = ensure_smem(attn_mma_kernel<D>, smem, configured);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)((p.nq + BM - 1) / BM) * p.B * p.H;
    attn_mma_kernel<D><<<(unsigned)blocks, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bf16_mma(const AttnParams &p, cudaStream_t s) {
    switch (p.d) {
        case 32: return launch<32>(p, s);
        case 64: return launch<64>(p, s);
        case 80: return launch<80>(p, s);
        case 128: return launch<128>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mar
