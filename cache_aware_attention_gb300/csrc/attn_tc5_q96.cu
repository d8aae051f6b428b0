// The tcgen05 attention kernel for cache-aware launches of 65 to 96 queries: 96-row Q
// buffers, which leave shared memory for one more K/V stage (4 at d = 80, 5 at d = 64; the
// MMAs still read 128 rows, and rows 96..127 belong to the softmax warp that has no live
// row). Measured: 512 px shape at A = 66 and 90, 225 -> 211 us; MAR-H shape at A = 96, 538
// -> 532 us. Its own translation unit: instantiated in attn_tc5.cu, these kernels shifted
// the code of the others there and the MAR-H cache-aware launch (A = 40) measured 1.6%
// slower.
#define MAR_TC5_EXTRA_TU
#include "attn_tc5.cu"

namespace mar {

cudaError_t launch_attn_bf16_tc5_q96(const AttnParams &p, cudaStream_t s) {
    if (p.nq > 96 || !p.idx) return cudaErrorInvalidValue;
    if (p.d == 64) return launch<64, 96>(p, s);
    if (p.d == 80) return launch<80, 96>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace mar
