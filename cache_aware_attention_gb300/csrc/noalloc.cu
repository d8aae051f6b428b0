// mar_attn_full_noalloc: full attention + layer-2 score with no caller workspace.
//
// Some callers cannot allocate device memory for the score's scratch buffer: plugins
// running inside a host framework whose allocator owns the whole device pool (a raw
// cudaMalloc there is forbidden or fragments the pool), decode loops that must not risk
// an allocation stalling or failing mid-step, and code that is handed only its input and
// output tensors. For them the per-head score partials live in a fixed buffer compiled
// into this library instead of in a caller-provided workspace.
//
// The buffer is a file-scope __device__ array, so every GPU that loads the library holds
// kScratchBytes of it until the process exits. Host code cannot use the array's name as
// a device address (it is a host-side stand-in); the address is obtained once per device
// with cudaGetSymbolAddress, with that device current, on the first call made on it.
#include <mutex>

#include "attn.h"
#include "marattn.h"
#include "score.h"

namespace mar {
int record_cuda_error(cudaError_t e);
}

namespace {

// 24 MiB: the raw-score rows of B*H*G*N <= 6,291,456 (b, h, generating query, token)
// entries (e.g. 64 rows x 12 heads x 4 queries x 320 tokens), or the per-head fp64
// partials of B*H*N <= 3,145,728 (b, h, token) entries that more than 16 heads need.
constexpr size_t kScratchBytes = size_t(24) << 20;

static __device__ __align__(256) unsigned char g_score_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up on first use).
cudaError_t scratch_ptr(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_score_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t mar_noalloc_scratch_bytes(void) { return kScratchBytes; }

int mar_attn_full_noalloc(const mar_shape *s, const void *Q, const void *K, const void *V, void *O,
                          float scale, const int32_t *gen_idx, int32_t G, float *score_out, float *lse_out,
                          uint32_t *d_status, mar_stream_t stream) {
    if (!s) return MAR_ERR_ARG;
    // full: the raw-score form's scratch where it applies; least: what the separate score
    // launch needs (0 up to 16 heads). mar_attn_full takes the raw-score form whenever the
    // workspace it is given holds `full`.
    const bool want = score_out != nullptr;
    const size_t full = mar_attn_full_workspace_bytes(s, G, want);
    const size_t least = mar_attn_full_min_workspace_bytes(s, G, want);
    if (least > kScratchBytes) return MAR_ERR_SCRATCH_LIMIT;
    void *ws = nullptr;
    if (full) {
        cudaError_t e = scratch_ptr(&ws);
        if (e != cudaSuccess) return mar::record_cuda_error(e);
    }
    return mar_attn_full(s, Q, K, V, O, scale, gen_idx, G, score_out, lse_out, ws, full ? kScratchBytes : 0,
                         d_status, stream);
}

}  // extern "C"
