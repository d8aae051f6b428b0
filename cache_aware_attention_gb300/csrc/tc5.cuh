// Blackwell (sm_100/sm_103) building blocks: mbarriers with bounded waits, TMA tensor
// tile loads, tcgen05 tensor-memory allocation, UMMA shared-memory and
// instruction descriptors, tcgen05.mma / commit, and tensor-memory loads/stores.
//
// Every wait is bounded: after kSpinLimit polls the waiter records MAR_STATUS_TIMEOUT in
// the caller's status word and returns false, so a kernel can unwind instead of hanging.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace mar {
namespace tc5 {

constexpr uint32_t kSpinLimit = 1u << 20;  // polls before a wait gives up (about a second)

// ------------------------------------------------------------------------ mbarrier
MAR_DEVINL void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
MAR_DEVINL void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::); }

// The arrival's state token goes to the sink: no register waits on the arrive's latency.
MAR_DEVINL void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Arrival with relaxed memory semantics: it orders no earlier memory access of this thread.
// For hand-overs whose data is in tensor memory (ordered by tcgen05.wait and the tcgen05
// fences), where a release arrival would also wait for this thread's outstanding global
// stores to become visible.
MAR_DEVINL void mbar_arrive_relaxed(uint64_t *bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
MAR_DEVINL void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
MAR_DEVINL bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the same condition (never suspends the thread): for issuers that
// poll several barriers and act on whichever is ready.
MAR_DEVINL bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete. Returns false on timeout (and
// records it in *status); *abort (shared) is also raised so other roles can unwind.
// try_wait costs about 200 cycles even on a phase that has already completed, so a
// non-blocking test comes first: most waits of a well-fed pipeline find the phase done.
MAR_DEVINL bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status, volatile int *abort,
                          uint32_t limit = kSpinLimit) {
    if (mbar_test(bar, parity)) return true;
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
    }
    report(status, MAR_STATUS_TIMEOUT);
    if (abort) *abort = 1;
    return false;
}
// mbar_wait by every lane of a warp with one result for all of them: a warp that gives
// up (a lane timed out, or saw another role's abort) leaves its loop as a whole, so the
// warp-wide instructions after it (.sync.aligned tensor-memory accesses, elect,
// shuffles) always run converged. The vote is taken on every wait: a vote only after
// polling would leave out the lanes whose first test passed (a barrier test need not
// give every lane the same answer), and single-lane issuer loops, which need no vote,
// measured 15-35% slower.
MAR_DEVINL bool mbar_wait_all(uint64_t *bar, uint32_t parity, uint32_t *status, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort));
}
// Spin-wait: non-suspending tests (mbarrier.test_wait), bounded by time (about a second
// of SM clocks) rather than by a poll count. A warp suspended in try_wait can resume some
// hundreds of cycles after the phase completes; where the waiting warps' issue slots are
// not needed by others this polls instead (the d = 64 attention kernel: 5-9% faster).
constexpr long long kSpinCycles = 1ll << 31;
MAR_DEVINL bool mbar_spin(uint64_t *bar, uint32_t parity, uint32_t *status, volatile int *abort) {
    const long long t0 = clock64();
    for (;;) {
#pragma unroll 1
        for (int k = 0; k < 32; ++k)
            if (mbar_test(bar, parity)) return true;
        if (abort && *abort) return false;
        if (clock64() - t0 > kSpinCycles) break;
    }
    report(status, MAR_STATUS_TIMEOUT);
    if (abort) *abort = 1;
    return false;
}
// mbar_spin by every lane of a warp with one result for all of them (as mbar_wait_all).
MAR_DEVINL bool mbar_spin_all(uint64_t *bar, uint32_t parity, uint32_t *status, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_spin(bar, parity, status, abort));
}
// The same wait on the abort path: it ignores the abort flag (the CTA is unwinding and
// waits for its own asynchronous copies and MMAs still in flight before it releases the
// shared and tensor memory they write). Bounded as well; returns false if it gave up.
MAR_DEVINL bool mbar_wait_drain(uint64_t *bar, uint32_t parity, uint32_t limit = kSpinLimit) {
    if (mbar_test(bar, parity)) return true;
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ------------------------------------------------------------------------ TMA
MAR_DEVINL void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
MAR_DEVINL void tma_load_3d(void *dst, const CUtensorMap *m, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------------ tensor memory
// Whole warp. Writes the allocated TMEM base address to *dst_smem.
MAR_DEVINL void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
MAR_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (tensor core, TMA) accesses.
MAR_DEVINL void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
MAR_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
MAR_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Tensor-memory loads: 32 lanes x n consecutive 32-bit columns, thread t of the warp
// gets lane (base + t). The load and its tcgen05.wait::ld sit in one asm statement, so
// the compiler cannot schedule any use of the destination registers before the data
// has arrived (a separate wait statement would not order the register uses).
MAR_DEVINL void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "{\n tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        " tcgen05.wait::ld.sync.aligned;\n}\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
MAR_DEVINL void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "{\n tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        " tcgen05.wait::ld.sync.aligned;\n}\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

MAR_DEVINL void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
MAR_DEVINL void tmem_st16(uint32_t taddr, const float (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16};\n" ::"r"(taddr),
        "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]), "f"(r[8]),
        "f"(r[9]), "f"(r[10]), "f"(r[11]), "f"(r[12]), "f"(r[13]), "f"(r[14]), "f"(r[15])
        : "memory");
}
MAR_DEVINL void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// ------------------------------------------------------------------------ UMMA descriptors
// Shared-memory matrix descriptor (sm_100 format): start address, leading and stride
// byte offsets (16-byte units), version 1 at bit 46, layout (swizzle) at bits 61-63.
enum class Swz : uint64_t { None = 0, B128 = 2, B64 = 4, B32 = 6 };

MAR_DEVINL uint64_t smem_desc(const void *smem, uint32_t lbo_bytes, uint32_t sbo_bytes, Swz swz) {
    const uint64_t a = smem_u32(smem);
    uint64_t d = 0;
    d |= (a >> 4) & 0x3FFFull;
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;
    d |= (uint64_t)swz << 61;
    return d;
}
// Advances the start-address field of a descriptor by `bytes` (must stay in the same
// 256 KB window; used for k-steps inside a swizzle atom and for atom steps).
MAR_DEVINL uint64_t desc_advance(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
// a_mn / b_mn: 1 when the operand is MN-major (transposed), 0 when K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16)
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T-as-described; issued by one thread.
MAR_DEVINL void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same with the A operand read from tensor memory (M rows in lanes, 2 bf16 per column).
MAR_DEVINL void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every MMA issued so far by this thread has completed.
MAR_DEVINL void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

MAR_DEVINL bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// Tile store shared -> global by the TMA unit (bulk-group completion). Rows or columns of
// the box outside the tensor are not written.
MAR_DEVINL void tma_store_3d(const CUtensorMap *m, int c0, int c1, int c2, const void *src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}
MAR_DEVINL void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Waits until at most N committed bulk groups of this thread still read shared memory.
template <int N> MAR_DEVINL void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}
// Contiguous global -> shared copy by the TMA unit, completing `bytes` on `bar`. Both
// addresses 16-byte aligned, bytes a multiple of 16.
MAR_DEVINL void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
}  // namespace tc5
}  // namespace mar
