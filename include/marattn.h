/*
 * marattn.h -- C ABI of the cache-aware attention library for masked-autoregressive
 * (MAR) image decoding on GB300 (sm_103a).
 *
 * The library implements the per-step hot path of MARché-style decoding:
 * full bidirectional attention with the layer-2 relevance score, top-K refresh
 * selection, split active/cached attention merged by online softmax, the KV-cache
 * gather/scatter, and LazyMAR's condition-cache guidance update.
 *
 * Sources, cited by page title and section:
 *  [M] "MARché: Fast Masked Autoregressive Image Generation with Cache-Aware
 *      Attention" (paper notes): Method / Overall Architecture; Key Designs 1-3.
 *  [R] "MARch'e: ... Cache-Aware Attention" (machine review): "What carries the
 *      argument"; "Assumptions & free parameters" (Appendix A equivalence).
 *  [L] "LazyMAR: Accelerating Masked Autoregressive Models via Feature Caching"
 *      (paper notes): Key Designs, Condition Cache.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers are caller-owned DEVICE pointers unless stated otherwise. The
 *    library allocates no device memory at run time and keeps no state between
 *    calls, except the fixed scratch buffer of mar_attn_full_noalloc (a static
 *    device array, see that call).
 *  - Tensors are dense and contiguous in the layouts given below:
 *      Q, K, V, O, cache           [B, H, N, d]   (token rows of d elements)
 *      Q_A, K_A, V_A, O_A          [B, H, A, d]   (active rows, in idx order)
 *      active_idx                  [B, A] int32   (token positions in [0, N))
 *    B counts rows after classifier-free-guidance doubling.
 *  - Element type: MAR_BF16 (bf16 storage, fp32 accumulation, bf16 output) or
 *    MAR_F32 (fp32 throughout). Supported head dims d: 32, 64, 80, 128.
 *  - Alignment: every Q/K/V/O/cache pointer must be 16-byte aligned
 *    (MAR_ERR_ALIGN); fp32 score/lse arrays need their natural 4-byte alignment.
 *  - Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream). Argument errors are detected on the host and
 *    returned before anything is launched.
 *  - Device-detected errors set bits in the caller's `d_status` word (a device
 *    uint32 that the caller zeroes; may be NULL to skip reporting): a position
 *    out of [0, N) (all calls that take positions) or repeated within one row
 *    (attention calls), and a bounded wait inside a kernel that gave up
 *    (MAR_STATUS_TIMEOUT). The offending access is skipped and the outputs that
 *    depend on it are unspecified. Kernels never trap.
 *  - Returns MAR_OK (0) or a negative mar_result.
 */
#ifndef MARATTN_H
#define MARATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *mar_stream_t; /* same object as cudaStream_t */

enum mar_dtype { MAR_F32 = 0, MAR_BF16 = 1 };

enum mar_result {
    MAR_OK = 0,
    MAR_ERR_ARG = -1,       /* NULL pointer, negative count, K > candidates, ... */
    MAR_ERR_SHAPE = -2,     /* unsupported head dim or size limit exceeded */
    MAR_ERR_DTYPE = -3,     /* unknown element type */
    MAR_ERR_ALIGN = -4,     /* pointer not 16-byte aligned */
    MAR_ERR_WORKSPACE = -5, /* workspace NULL, too small or misaligned */
    MAR_ERR_CUDA = -6,      /* a CUDA call failed; see mar_last_cuda_error() */
    MAR_ERR_NODEV = -7,     /* no usable sm_103 device */
    MAR_ERR_SCRATCH_LIMIT = -8 /* needs more scratch than the built-in no-allocation buffer */
};

/* Bits OR-ed into *d_status by the kernels. */
#define MAR_STATUS_INDEX_RANGE 0x1u /* a position outside [0, N) */
#define MAR_STATUS_INDEX_DUP 0x2u   /* a position repeated within one row */
/* A wait of the tensor-core attention kernel (on a copy, a tensor-core operation or
 * another role of the same thread block) ran past its limit of about a second. The
 * kernel then stops its work, waits (again bounded) for the copies and tensor-core
 * operations it has already issued, releases its tensor memory and returns: the
 * outputs of that call are unspecified, the CUDA context stays usable and later calls
 * are unaffected. It signals a fault of the device or of the library, never a
 * property of the inputs. */
#define MAR_STATUS_TIMEOUT 0x4u

/* Bits of the `fuse_scatter` argument of mar_attn_cache_aware and
 * mar_attn_cache_aware_gather (0 and 1 keep their plain meaning; any other bit returns
 * MAR_ERR_ARG). */
#define MAR_CA_FUSE_SCATTER 0x1 /* also write K_A/V_A into the cache rows at the active positions */
/* The caller guarantees that V_cache holds finite values at the active positions, as in a
 * decode loop, where those rows hold an earlier step's V (written by a refresh or a
 * scatter). Those rows get attention weight exactly 0 either way. Without this bit the
 * kernel also zeroes them in shared memory before the P.V product, so that whatever they
 * hold (NaN or infinity included) leaves the output unchanged; with it they are used as
 * loaded, and a finite row adds exactly 0. If the guarantee does not hold, the outputs of
 * the call are unspecified. */
#define MAR_CA_STALE_FINITE 0x2

enum mar_cfg_mode { MAR_CFG_APPLY = 0, MAR_CFG_UPDATE = 1 };

typedef struct mar_shape {
    int32_t B;     /* batch rows (after CFG doubling) */
    int32_t H;     /* heads */
    int32_t N;     /* tokens per row (buffer + image tokens) */
    int32_t d;     /* head dim: 32, 64, 80 or 128 (attention); see the row copies */
    int32_t dtype; /* enum mar_dtype */
} mar_shape;

/* Human-readable text for a mar_result (static storage). */
const char *mar_error_string(int code);
/* cudaError_t of the last failed CUDA call on this thread (0 if none). */
int mar_last_cuda_error(void);
/* ABI version of this header: major * 10000 + minor * 100 + patch. */
int mar_version(void);

/*
 * mar_attn_full -- full bidirectional softmax attention, optionally with the
 * layer-2 head-averaged relevance score.
 *
 * [M] Overall Architecture: layers 1-2 run standard full attention at every
 * step (and all layers on a full-refresh step, Key Design 3). For each (b, h, i):
 *   O[b,h,i,:] = sum_j softmax_j(scale * <Q[b,h,i,:], K[b,h,j,:]>) V[b,h,j,:]
 *   lse[b,h,i] = log sum_j exp(scale * <Q[b,h,i,:], K[b,h,j,:]>)   (natural log)
 * [M] Key Design 1: the weights from the G generating queries to every token,
 * averaged over heads (and over the generating queries):
 *   score[b,j] = 1/(H*G) * sum_h sum_g softmax_j(scale * <Q[b,h,gen[b,g],:], K[b,h,j,:]>)
 * The score is accurate to below 1e-6 relative (fp32 dot products and exponentials,
 * sums over keys and rows carried to fp64-grade accuracy), so that the top-K built on
 * it matches an exact evaluation except on near-ties. For bf16 with d = 64 or 80,
 * G <= 32 and N a multiple of 4 the attention launch itself leaves the raw scores of
 * the generating rows (its tensor-core dot products) and their softmax statistics for
 * a small reduction launch; other shapes compute the dot products again in a
 * separate score launch.
 *
 *  Q, K, V, O  [B,H,N,d] (dtype); O may not alias Q, K or V.
 *  scale       softmax scale; 0 selects 1/sqrt(d).
 *  gen_idx     [B,G] int32 generating positions, or NULL when score_out is NULL.
 *  score_out   [B,N] fp32 or NULL. Requires G >= 1.
 *  lse_out     [B,H,N] fp32 or NULL.
 *  workspace   device scratch of mar_attn_full_workspace_bytes() bytes (256-byte
 *              aligned), or NULL when that size is 0. Contents are overwritten;
 *              calls that overlap on the GPU must not share it. The size is
 *              4*B*H*G*N + 8*B*H*G bytes (each rounded up to 256) where the attention
 *              launch leaves the raw scores; otherwise the separate score launch
 *              computes the score and needs 8*B*H*N bytes when H > 16, none when
 *              H <= 16. A workspace of at least mar_attn_full_min_workspace_bytes()
 *              (possibly 0, i.e. NULL) but below the full size is also accepted: the
 *              score is then computed by the separate score launch.
 */
size_t mar_attn_full_workspace_bytes(const mar_shape *shape, int32_t G, int want_score);
size_t mar_attn_full_min_workspace_bytes(const mar_shape *shape, int32_t G, int want_score);
int mar_attn_full(const mar_shape *shape, const void *Q, const void *K, const void *V,
                  void *O, float scale, const int32_t *gen_idx, int32_t G,
                  float *score_out, float *lse_out, void *workspace,
                  size_t workspace_bytes, uint32_t *d_status, mar_stream_t stream);

/*
 * mar_attn_full_select -- the layer-2 call of a cached step: full attention, the
 * head-averaged score and, on it, the refresh set and the active set.
 *
 * [M] Key Design 1: exactly mar_attn_full (with score_out) followed by
 * mar_refresh_topk(score_out, exclude_idx, E, Ksel, out_idx, active_out), issued as
 * one call (the same launches and values).
 *  Arguments as for mar_attn_full and mar_refresh_topk; score_out is required.
 */
int mar_attn_full_select(const mar_shape *shape, const void *Q, const void *K, const void *V,
                         void *O, float scale, const int32_t *gen_idx, int32_t G,
                         const int32_t *exclude_idx, int32_t E, int32_t Ksel, float *score_out,
                         int32_t *out_idx, int32_t *active_out, float *lse_out, void *workspace,
                         size_t workspace_bytes, uint32_t *d_status, mar_stream_t stream);

/*
 * mar_attn_full_refresh -- full attention of a full-refresh step together with the
 * full cache overwrite of that layer.
 *
 * [M] Key Design 3: on a full-refresh step every token is recomputed at every
 * layer and the layer's cache is rebuilt from the fresh K/V (Key Design 2 keeps
 * the latest projection of every token). This call computes exactly the O (and
 * lse) of mar_attn_full for Q, K, V and leaves
 *   K_cache[b,h,j,:] = K[b,h,j,:],  V_cache[b,h,j,:] = V[b,h,j,:]   for all j
 * (bit copies), i.e. mar_attn_full followed by mar_kv_scatter with active_idx ==
 * NULL. For bf16 with d = 64 or 80 both happen in one launch: the attention kernel
 * stores the K/V tiles it has staged in shared memory, so K and V are read from
 * memory once; other shapes take two launches.
 *
 *  Q, K, V, O        [B,H,N,d] (dtype); O may not alias Q, K or V.
 *  K_cache, V_cache  [B,H,N,d] (dtype), overwritten; must not alias Q, K, V, O or
 *                    each other.
 *  scale, lse_out    as for mar_attn_full.
 */
int mar_attn_full_refresh(const mar_shape *shape, const void *Q, const void *K, const void *V,
                          void *O, void *K_cache, void *V_cache, float scale, float *lse_out,
                          uint32_t *d_status, mar_stream_t stream);

/*
 * mar_attn_full_noalloc -- mar_attn_full for callers that cannot allocate.
 *
 * The paper has no counterpart to this call; it exists for callers that must not
 * allocate device memory, such as plugins inside a host framework whose allocator
 * owns the device pool, or decode loops that cannot risk an allocation stalling or
 * failing mid-step. It computes exactly what mar_attn_full computes, with the same
 * arguments except the workspace: the score's scratch lives in a buffer compiled into
 * the library (mar_noalloc_scratch_bytes() bytes, 24 MiB, held on every GPU that loads
 * the library until the process exits).
 *  - Takes the raw-score form of the score when its scratch (see mar_attn_full) fits
 *    in the buffer, else the separate score launch. Returns MAR_ERR_SCRATCH_LIMIT when
 *    neither fits: H > 16 with 8*B*H*N bytes above 24 MiB (B*H*N above 3,145,728), and
 *    the raw-score form not applicable or above 24 MiB as well.
 *  - Allocates nothing. The first call made on a device looks up the buffer's device
 *    address; make that first call before any stream capture.
 *  - All calls share the one buffer: calls that can overlap on the GPU (different
 *    streams, or different host threads on one device) race and must be serialised
 *    by the caller. The buffer keeps the previous call's contents; nothing in it needs
 *    to start at zero.
 */
size_t mar_noalloc_scratch_bytes(void);
int mar_attn_full_noalloc(const mar_shape *shape, const void *Q, const void *K, const void *V,
                          void *O, float scale, const int32_t *gen_idx, int32_t G,
                          float *score_out, float *lse_out, uint32_t *d_status,
                          mar_stream_t stream);

/*
 * mar_attn_cache_aware -- split attention of the active queries over fresh
 * active K/V and stored cached K/V, merged with the safe online-softmax rule.
 *
 * [M] Key Design 2 and [R] "What carries the argument": with C(b) the positions
 * of row b that are NOT in active_idx[b] (the cached set; the two sets are
 * disjoint), each active query i attends over the key list
 *   K_A[b,h,0..A) followed by K_cache[b,h,p,:] for p in C(b)
 * (V likewise) as two partial softmax sums merged by running max and running
 * sum:  z_i = (alpha^(A) V_A + alpha^(C) V_C) / l_i. Cache rows at active
 * positions hold stale values and never contribute, whatever they hold (they may
 * be read and are then masked out). The result equals full attention over the
 * concatenated list ([R] Appendix A equivalence).
 *
 *  Q_A, K_A, V_A, O_A  [B,H,A,d]; active_idx [B,A] distinct positions in [0,N).
 *  K_cache, V_cache    [B,H,N,d]. Read at cached positions; with the
 *                      MAR_CA_FUSE_SCATTER bit of fuse_scatter the call also writes
 *                      K_A/V_A into the rows at the active positions (the
 *                      mar_kv_scatter update), which no query of the call reads.
 *  fuse_scatter        MAR_CA_FUSE_SCATTER | MAR_CA_STALE_FINITE bits (0 or 1 as a
 *                      plain flag).
 *  lse_out             [B,H,A] fp32 or NULL.
 *  workspace, workspace_bytes
 *                      reserved: the kernels of this call need no scratch memory
 *                      (mar_attn_cache_aware_workspace_bytes() returns 0 for every
 *                      shape); pass NULL and 0. Any value is accepted and ignored.
 *  A == 0 is a no-op. A == N (no cached tokens) is plain attention over K_A.
 *  Limit: N <= 16384.
 */
size_t mar_attn_cache_aware_workspace_bytes(const mar_shape *shape, int32_t A);
int mar_attn_cache_aware(const mar_shape *shape, int32_t A, const void *Q_A,
                         const void *K_A, const void *V_A, void *K_cache, void *V_cache,
                         const int32_t *active_idx, void *O_A, float scale,
                         float *lse_out, int32_t fuse_scatter, void *workspace,
                         size_t workspace_bytes, uint32_t *d_status,
                         mar_stream_t stream);

/*
 * mar_attn_cache_aware_gather -- mar_attn_cache_aware with the active gather
 * folded in: the gather of the active rows, the cache-aware attention and the
 * cache update of one cached layer in one launch.
 *
 * [M] Overall Architecture and Key Design 2: the cached layers compute fresh
 * Q/K/V only for the active tokens. Here the fresh tensors are whole [B,H,N,d]
 * tensors and the active rows are read from them in place:
 *   Q_A[b,h,a,:] = Q[b,h,active_idx[b,a],:]   (K_A, V_A likewise)
 * and the result is exactly mar_attn_cache_aware(Q_A, K_A, V_A, ...) (the same
 * kernels, reading the rows through active_idx instead of from dense copies).
 * With the MAR_CA_FUSE_SCATTER bit of fuse_scatter the cache rows at the active
 * positions receive the fresh rows:  K_cache[b,h,p,:] = K[b,h,p,:] for p in
 * active_idx[b] (V likewise); MAR_CA_STALE_FINITE as for mar_attn_cache_aware.
 *  Q, K, V             [B,H,N,d] fresh tensors (read only at active positions).
 *  K_cache, V_cache    [B,H,N,d]; must not be the same buffers as K, V or Q.
 *  O_A                 [B,H,A,d];  lse_out [B,H,A] fp32 or NULL.
 *  active_idx          [B,A] distinct positions in [0,N); an out-of-range or
 *                      repeated position sets MAR_STATUS_INDEX_RANGE / _DUP and
 *                      leaves the output unspecified (no fault).
 * A == 0 is a no-op. Limits: N <= 16384 and B*H*N < 2^31 (MAR_ERR_SHAPE).
 */
int mar_attn_cache_aware_gather(const mar_shape *shape, int32_t A, const void *Q, const void *K,
                                const void *V, void *K_cache, void *V_cache,
                                const int32_t *active_idx, void *O_A, float scale,
                                float *lse_out, int32_t fuse_scatter, uint32_t *d_status,
                                mar_stream_t stream);

/*
 * mar_kv_scatter -- write refreshed K/V rows into the per-layer cache.
 *
 * [M] Key Design 2: active tokens carry fresh K/V; the cache keeps every
 * token's latest projection. Key Design 3: a full-refresh step overwrites all.
 *   K_cache[b,h,active_idx[b,a],:] = K_A[b,h,a,:]   (V likewise; bit copies)
 * active_idx == NULL with A == N overwrites every row in order (full refresh).
 * Either the K pair or the V pair may be NULL to skip that tensor. Repeated
 * positions leave it unspecified which row lands. Row copies (this call and
 * mar_kv_gather) take any d whose row is whole 16-byte vectors, d <= 16384 (e.g. a
 * [B, 1, N, D] hidden state of a token cache). A position of -1 marks an unused slot
 * of a padded row of positions (mar_select_recompute pads its rows that way): the slot
 * is skipped silently. Any other position outside [0, N) sets MAR_STATUS_INDEX_RANGE
 * and is skipped.
 */
int mar_kv_scatter(const mar_shape *shape, int32_t A, const void *K_A, const void *V_A,
                   const int32_t *active_idx, void *K_cache, void *V_cache,
                   uint32_t *d_status, mar_stream_t stream);

/*
 * mar_kv_gather -- copy the active rows of up to 3 full tensors into dense
 * active blocks (the active-token gather that feeds the fresh projections).
 *   dst[t][b,h,a,:] = src[t][b,h,active_idx[b,a],:]   for t < n_tensors (bit copies)
 * src and dst are HOST arrays of n_tensors (1..3) device pointers. Positions as for
 * mar_kv_scatter: the dst rows of -1 slots are left as they were.
 */
int mar_kv_gather(const mar_shape *shape, int32_t A, int32_t n_tensors,
                  const void *const *src, void *const *dst, const int32_t *active_idx,
                  uint32_t *d_status, mar_stream_t stream);

/*
 * mar_refresh_topk -- choose the refreshing tokens and build the active set.
 *
 * [M] Key Design 1: the K tokens with the highest layer-2 relevance score,
 * excluding the generating and just-decoded tokens (exclude_idx, which are
 * active anyway), become the refreshing tokens. Equal scores go to the lower
 * position (scores are ordered by their fp32 bit pattern, so -0 < +0).
 *  score        [B,N] fp32.
 *  exclude_idx  [B,E] int32 (E may be 0, then NULL is allowed).
 *  out_idx      [B,K] int32: the chosen positions in ascending order (or NULL).
 *  active_out   [B,E+K] int32: exclude_idx[b] followed by out_idx[b] -- the
 *               active set [generating, just-decoded, refreshing] (or NULL).
 * Errors: K > N - E returns MAR_ERR_ARG. Limits: N <= 4096 (MAR_ERR_SHAPE beyond).
 */
int mar_refresh_topk(int32_t B, int32_t N, const float *score, const int32_t *exclude_idx,
                     int32_t E, int32_t K, int32_t *out_idx, int32_t *active_out,
                     uint32_t *d_status, mar_stream_t stream);

/*
 * mar_refresh_topk_pairs -- one refresh set per classifier-free-guidance pair.
 *
 * [M] Key Design 1 selects the refreshing tokens per batch row; the pages do not say
 * whether, with guidance, the conditional row b and the unconditional row
 * b + B_pairs select separately or share one set. This call is the shared reading
 * (mar_refresh_topk is the separate one): the pair's candidates are
 * ranked on the fp32 sum of the two rows' scores (one IEEE single addition per
 * position), with row b's exclusions, ties to the lower position, output ascending.
 * Both rows receive the same set; each row's active_out starts with its own exclusions.
 *  score        [2*B_pairs, N] fp32 (rows [0, B_pairs) conditional, then unconditional).
 *  exclude_idx  [2*B_pairs, E] int32; out_idx [2*B_pairs, K] and/or active_out
 *               [2*B_pairs, E + K]. Limits and errors as for mar_refresh_topk.
 */
int mar_refresh_topk_pairs(int32_t B_pairs, int32_t N, const float *score, const int32_t *exclude_idx,
                           int32_t E, int32_t K, int32_t *out_idx, int32_t *active_out,
                           uint32_t *d_status, mar_stream_t stream);

/*
 * mar_token_cosine -- per-token cosine similarity of two feature tensors.
 *
 * [L] Token Cache: deeper layers reuse a token's cached value when its current
 * feature is close, in cosine similarity, to the cached one. [M] Figure 1 and
 * Figures 10-11: the cosine of the key (value) projections between decoding steps,
 * which shows the drift that cached attention tolerates. A token's feature is its
 * values over all heads:
 *   cos[b,n] = <X[b,:,n,:], Y[b,:,n,:]> / (|X[b,:,n,:]| |Y[b,:,n,:]|)
 * both zero -> 1, one zero -> 0. Sums are carried to fp64-grade accuracy in a fixed
 * order (deterministic); the result is fp32.
 *  X, Y     [B,H,N,d] (dtype); any d with d * element size a multiple of 16 bytes,
 *           d <= 16384 (H = 1 with d = the model width for a [B,N,D] hidden state).
 *  cos_out  [B,N] fp32.
 */
int mar_token_cosine(const mar_shape *shape, const void *X, const void *Y, float *cos_out,
                     mar_stream_t stream);

/*
 * mar_select_recompute -- the token cache's recompute set.
 *
 * [L] Token Cache: tokens with a high similarity to the cached feature reuse the
 * cached value; the others are recomputed. Here position n of row b is recomputed
 * when it is in force_idx[b] or when not (cos[b,n] > tau) (a NaN similarity is
 * recomputed); the decision is taken on the given fp32 values.
 *  cos        [B,N] fp32 (e.g. from mar_token_cosine); N <= 16384.
 *  force_idx  [B,F] int32 or NULL when F == 0 (e.g. the tokens decoded this step);
 *             out-of-range entries set MAR_STATUS_INDEX_RANGE and are ignored.
 *  out_idx    [B,N] int32: the recomputed positions in ascending order, then -1.
 *  out_count  [B] int32: how many.
 */
int mar_select_recompute(int32_t B, int32_t N, const float *cos, float tau, const int32_t *force_idx,
                         int32_t F, int32_t *out_idx, int32_t *out_count, uint32_t *d_status,
                         mar_stream_t stream);

/*
 * mar_cfg_residual -- LazyMAR condition cache on fp32 outputs of n elements.
 *
 * [L] Condition Cache: a cached step runs only the conditional branch and
 * takes uncond = cond - residual (MAR_CFG_APPLY: writes uncond); a full step
 * runs both branches and refreshes residual = cond - uncond (MAR_CFG_UPDATE:
 * writes residual). If `guided` is non-NULL it also receives textbook guidance
 * uncond + w * (cond - uncond) (not printed on the pages). IEEE round-to-
 * nearest fp32 operations, no fused multiply-add.
 */
int mar_cfg_residual(int32_t mode, int64_t n, const float *cond, float *uncond,
                     float *residual, float w, float *guided, mar_stream_t stream);

/*
 * mar_status_read -- synchronise `stream` and copy *d_status to *h_status
 * (host pointer).
 */
int mar_status_read(const uint32_t *d_status, uint32_t *h_status, mar_stream_t stream);

/*
 * mar_selftest_wait_timeout -- exercises the bounded wait of the tensor-core kernels.
 *
 * Not part of the method (the pages have no counterpart): a diagnostic for the
 * status path. One thread block initialises a shared-memory barrier that nothing ever
 * completes and waits on it with the same bounded wait the attention kernel uses, but
 * with `spin_limit` polls instead of the kernel's limit of about a second. The wait
 * gives up, sets MAR_STATUS_TIMEOUT in *d_status and the kernel returns; no copy or
 * tensor-core operation is in flight. spin_limit must be in [1, 1<<20] (MAR_ERR_ARG
 * otherwise); d_status must not be NULL.
 */
int mar_selftest_wait_timeout(uint32_t spin_limit, uint32_t *d_status, mar_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MARATTN_H */
