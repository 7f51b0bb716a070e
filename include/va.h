/*
 * va.h - C ABI of the B300 (sm_103a) block-sparse video attention library.
 *
 * Operations (sources named by page and section):
 *   - static spatiotemporal block masks over a flattened (frame, height, width)
 *     latent token grid: the radial energy-decay mask (Radial Attention news
 *     page, hyper.ai) and the LVSA local-window + rotating periodic anchor
 *     mask (LVSA review, secrett2633 blog, sec. 3 and Fig. 2);
 *   - block-sparse softmax attention forward under such a mask (LVSA review
 *     sec. 1 "block-sparse attention"; LinVideo, gist.science 2510.08318,
 *     technical summary sec. 1 on the O(n^2) attention bottleneck);
 *   - k-means clustering of query/key tokens and centroid-compensated sparse
 *     attention with error-aware routing under a density budget (SVG-EAR,
 *     gist.science 2603.08982, technical summary sec. 2, ideas 1 and 2).
 *
 * Conventions shared by every call:
 *   - Token n of a T x H x W latent is n = t*H*W + h*W + w (t-major).
 *   - Tensors are DEVICE pointers owned by the caller, contiguous
 *     [B, heads, N, d] (d fastest), 16-byte aligned. dtype VA_BF16 means
 *     bfloat16 elements, VA_F32 means float32.
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL is the
 *     legacy default stream) unless documented otherwise, and run on the
 *     CUDA device current in the calling thread.
 *   - Scratch device memory comes, stream-ordered, from a memory pool the
 *     library keeps per device. Memory freed at the end of a call stays in
 *     the pool for the next call rather than returning to the driver, so a
 *     process holds the peak scratch of its largest call (about 1 GB for the
 *     compensated route at 32,760 tokens, 12 heads).
 *   - Every call returns VA_OK (0) or a negative VA_ERR_* code; on an error
 *     return nothing was launched unless stated. The library never aborts the
 *     process and never traps the GPU: a device-side wait that times out, or a
 *     device-side bounds check that fails, records a code that
 *     va_device_error() reports.
 */
#ifndef VA_H
#define VA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* va_stream_t; /* identical to cudaStream_t */
typedef struct va_mask va_mask;          /* opaque, library-owned */

/* status codes */
#define VA_OK 0
#define VA_ERR_INVALID (-1)     /* null pointer, bad size, misaligned, shape mismatch */
#define VA_ERR_UNSUPPORTED (-2) /* dtype / head_dim / block / device not supported */
#define VA_ERR_CUDA (-3)        /* a CUDA runtime call failed */
#define VA_ERR_OOM (-4)         /* device allocation failed */
#define VA_ERR_TIMEOUT (-5)     /* a device-side wait gave up (from va_device_error) */
#define VA_ERR_DEVICE (-6)      /* a device-side bounds check failed (from va_device_error) */

/* mask kinds */
#define VA_MASK_DENSE 0  /* every block pair live (dense attention on the same kernel) */
#define VA_MASK_RADIAL 1 /* radial energy-decay mask */
#define VA_MASK_LVSA 2   /* local frame window + rotating periodic anchor frames */

/* element types */
#define VA_F32 0
#define VA_BF16 1

/*
 * Mask parameters.
 *   block      tokens per block (query and key blocks are the same size); the
 *              last block holds N - (nqb-1)*block tokens. 1..4096.
 *   w0         radial: base half-width W0 of the in-frame window; token pair
 *              (i, j) is live iff |s_i - s_j| <= W0 >> octave(|t_i - t_j|)
 *              with s = in-frame index, octave(0)=0 and octave(dt) = bit
 *              length of dt. 0 selects W0 = H*W.
 *   local      LVSA: frames within +-local of the query frame are attended.
 *   period     LVSA: anchor period P; key frame t is an anchor at denoising
 *              step s iff (t - anchor0 - rot_stride*s) mod P == 0. P == 0
 *              means the single anchor frame anchor0 (no rotation).
 *   anchor0    LVSA: anchor offset.
 *   rot_stride LVSA: anchor shift per denoising step.
 * A (query block, key block) pair is live iff some real token pair in it is
 * live under the token rule; a live pair is computed in full.
 */
typedef struct va_mask_params {
  int32_t block;
  int32_t w0;
  int32_t local;
  int32_t period;
  int32_t anchor0;
  int32_t rot_stride;
} va_mask_params;

/*
 * Build the block mask of `kind` for a T x H x W grid at denoising `step` and
 * return it as a library-owned handle holding a device CSR:
 *   row_ptr[nqb + 1] (int32), col_idx[nnz] (int32, strictly ascending per row),
 *   nqb = ceil(T*H*W / block).
 * Sources: the radial rule follows the Radial Attention news page (hyper.ai:
 * static mask, window shrinking exponentially with temporal distance,
 * O(n log n)); the LVSA rule follows the LVSA review (secrett2633 blog,
 * sec. 3 and Fig. 2: local frame window plus periodic anchor frames that
 * rotate with the denoising step); block pooling follows its sec. 1
 * ("block-sparse attention"). The pages give no formulas: the token rules
 * above va_mask_params are readings of them.
 * The mask is identical for every batch element and head. The result is
 * bit-exact (integer arithmetic only). The handle's arrays live on the
 * device current at the call; the attention calls reject a mask from another
 * device. This call synchronises `stream` once (to size col_idx); the handle
 * is ready when it returns.
 * Errors: VA_ERR_INVALID (null out/params, non-positive sizes, N >= 2^30,
 * block outside 1..4096, negative local/period/w0), VA_ERR_UNSUPPORTED
 * (nqb > VA_MASK_MAX_BLOCKS, or more than 2^31 - 1 live block pairs, which
 * int32 row offsets cannot index), VA_ERR_OOM, VA_ERR_CUDA.
 */
#define VA_MASK_MAX_BLOCKS 65536
int va_mask_build(int kind, int T, int H, int W, const va_mask_params* params, int step,
                  va_mask** out, va_stream_t stream);

/* Device CSR arrays of a mask (owned by the handle) and its sizes. Any output
 * pointer may be NULL. Errors: VA_ERR_INVALID for a NULL mask. */
int va_mask_csr(const va_mask* mask, const int32_t** row_ptr_dev, const int32_t** col_idx_dev,
                int* nqb, int64_t* nnz);

/* Grid and accounting data of a mask: N = T*H*W, block, and live_pairs =
 * sum over live block pairs of |I|*|J| (real tokens only). Any output may be
 * NULL. Errors: VA_ERR_INVALID for a NULL mask. */
int va_mask_info(const va_mask* mask, int* N, int* block, int64_t* live_pairs);

/* Copy the CSR to caller-owned HOST arrays row_ptr[nqb+1] and col_idx[nnz]
 * (synchronous). Errors: VA_ERR_INVALID, VA_ERR_CUDA. */
int va_mask_to_host(const va_mask* mask, int32_t* row_ptr, int32_t* col_idx);

/* Release a mask (NULL is accepted). Synchronises the device work that may
 * still use it only through the caller: do not free a mask that a queued
 * kernel still reads. */
int va_mask_free(va_mask* mask);

/*
 * Allocation-free mask build (the paper has no counterpart: this is an
 * interface for callers, not part of the method).
 *
 * Builds the same CSR as va_mask_build, bit for bit, into caller-owned DEVICE
 * arrays row_ptr[nqb + 1] and col_idx[col_capacity] (int32), with
 * nqb = ceil(T*H*W / block), and writes the number of live block pairs to
 * *nnz (host). It is meant for callers that must not allocate device memory
 * on this path: code running under a caching or arena allocator that owns the
 * whole device, real-time loops where a cudaMalloc would stall or synchronise
 * the device, and embedders whose memory is handed out by the host framework.
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine. Its scratch (per-row counts and a small summary) lives in a
 * statically sized device array inside the library, which every GPU that
 * loads the library keeps until the process exits (about 1.3 MB).
 *
 * Limit: nqb <= VA_STATIC_MAX_BLOCKS; larger grids return VA_ERR_UNSUPPORTED
 * before any device work.
 * The first call on a device looks up that device's address of the scratch
 * array (cudaGetSymbolAddress); make that first call before any stream
 * capture. Every call shares the one scratch array, so calls that overlap on
 * the GPU (different streams, or host threads without ordering) race and must
 * be serialised by the caller. The call synchronises `stream` once, after the
 * counting pass, to read nnz; the column fill is queued on `stream` after that.
 * If nnz > col_capacity, *nnz is still set, col_idx is left untouched and
 * VA_ERR_INVALID is returned (call again with a larger array).
 * Errors: VA_ERR_INVALID (as va_mask_build; null row_ptr/nnz; col_idx NULL
 * with col_capacity > 0; capacity too small), VA_ERR_UNSUPPORTED (grid too
 * large for the static scratch, or nnz > 2^31 - 1: *nnz is set, row_ptr is
 * not usable and col_idx is untouched), VA_ERR_CUDA.
 */
#define VA_STATIC_MAX_BLOCKS 65536
int va_mask_build_static(int kind, int T, int H, int W, const va_mask_params* params, int step,
                         int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, int64_t* nnz,
                         va_stream_t stream);

/*
 * Mask cache: reuse of block masks across denoising steps (LVSA review,
 * secrett2633 blog, sec. 3: the anchors rotate with the denoising step, so a
 * step's mask repeats once the rotation comes round; Radial Attention news
 * page, hyper.ai: the radial mask is static, one for every step).
 *
 * va_mask_cache_get returns the library-owned mask for (kind, grid, params,
 * step) on the current device, building it with va_mask_build on the first
 * request and returning the same handle afterwards. Requests that differ only
 * in what the CSR does not depend on share one entry: a radial or dense mask
 * ignores `step` (and the LVSA fields); an LVSA mask with period > 0 depends
 * on the step only through the phase (anchor0 + rot_stride * step) mod
 * period, so period distinct phases cover every step. The returned handle's
 * recorded step is the one it was built for; its CSR is bit-identical to
 * va_mask_build at the requested step.
 *
 * Ownership: the cache owns its masks. Do not pass them to va_mask_free. A
 * handle stays valid until va_mask_cache_clear or va_mask_cache_destroy on
 * its cache; the cache never evicts by itself. A miss with `capacity` entries
 * already held returns VA_ERR_UNSUPPORTED and builds nothing.
 * Calls on one cache are serialised by a mutex. A hit does no device work and
 * does not touch `stream`; a miss synchronises `stream` once (as
 * va_mask_build). Clearing frees each mask on its own device; free its masks
 * only after the kernels that read them have completed.
 * Errors: VA_ERR_INVALID (null pointers, capacity outside
 * 1..VA_MASK_CACHE_MAX, and the argument errors of va_mask_build),
 * VA_ERR_UNSUPPORTED (cache full, or as va_mask_build), VA_ERR_OOM,
 * VA_ERR_CUDA.
 */
#define VA_MASK_CACHE_MAX 4096
typedef struct va_mask_cache va_mask_cache; /* opaque, library-owned */
int va_mask_cache_create(int capacity, va_mask_cache** out);
int va_mask_cache_get(va_mask_cache* cache, int kind, int T, int H, int W,
                      const va_mask_params* params, int step, const va_mask** out,
                      va_stream_t stream);
/* Counters of a cache: requests served from it, masks built, entries held.
 * Any output pointer may be NULL. Errors: VA_ERR_INVALID for a NULL cache. */
int va_mask_cache_stats(va_mask_cache* cache, int64_t* hits, int64_t* misses, int* entries);
/* Frees every mask of the cache (their handles become invalid) and keeps the
 * cache. Errors: VA_ERR_INVALID for a NULL cache. */
int va_mask_cache_clear(va_mask_cache* cache);
/* Clears and frees the cache. NULL is a no-op. */
int va_mask_cache_destroy(va_mask_cache* cache);
/* Host only: *same = 1 when the cache serves (kind, grid, params) at steps
 * step_a and step_b from one entry (their CSRs are identical), else 0.
 * Errors: the argument errors of va_mask_build (VA_ERR_INVALID,
 * VA_ERR_UNSUPPORTED); *same is 0 then. */
int va_mask_same(int kind, int T, int H, int W, const va_mask_params* params, int step_a,
                 int step_b, int* same);

/*
 * Block-sparse attention forward (LVSA review, secrett2633 blog, sec. 1:
 * attention computed only on the live blocks of a block-sparse mask; Radial
 * Attention news page, hyper.ai: the same computation under the static
 * radial mask; LinVideo, gist.science 2510.08318, technical summary sec. 1:
 * this quadratic attention is the cost that dominates video generation). The
 * pages name softmax attention without a variant, so this is the textbook
 * masked form. For every batch b, head h and query token i
 * with block I = i / block:
 *   l_j   = scale * q_i . k_j   for keys j in live key blocks of row I, j < N
 *   o_i   = sum_j exp(l_j - m) v_j / sum_j exp(l_j - m),  m = max_j l_j
 *   lse_i = m + ln sum_j exp(l_j - m)       (natural log; -inf, o_i = 0 if
 *                                            row I has no live block)
 * q, k, v, out: [B, heads, N, d] device arrays of `dtype`; lse: NULL or a
 * [B, heads, N] float32 device array. Softmax and accumulation are float32;
 * VA_BF16 inputs give a bf16 output, VA_F32 inputs a float32 output.
 * Supported: VA_BF16 with d in {64, 128} and block 128 or 64 (tcgen05
 * tensor-core kernel; with block 64 it runs 128-row tiles over pairs of
 * blocks and masks the dead 64 x 64 quarters); VA_F32 with d in {64, 128} and
 * block in {64, 128} (float32 FMA kernel).
 * Errors: VA_ERR_INVALID (null pointers, N != T*H*W of the mask, B or heads
 * < 1, misaligned pointers, a mask built on another device), VA_ERR_UNSUPPORTED
 * (other dtype/d/block), VA_ERR_CUDA (launch failure).
 */
int va_sparse_attn_fwd(const void* q, const void* k, const void* v, const va_mask* mask,
                       void* out, float* lse, int B, int heads, int N, int d, float scale,
                       int dtype, va_stream_t stream);

/*
 * Block-sparse attention backward: the gradients of va_sparse_attn_fwd's
 * output for an upstream gradient dout = dL/dout (Radial Attention, hyper.ai
 * news page: LoRA fine-tuning for 4x longer videos trains through the same
 * masked attention; the page gives no formulas, these are the chain rule of
 * the forward's definition). With p_ij = exp(scale q_i . k_j - lse_i) on the
 * live blocks (j < N) and delta_i = dout_i . out_i:
 *   ds_ij = p_ij (dout_i . v_j - delta_i)
 *   dq_i  = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i,
 *   dv_j  = sum_i p_ij dout_i
 * q, k, v, out, dout, dq, dk, dv: [B, heads, N, d] device arrays of `dtype`
 * (out and lse as the forward call with the same q, k, v, mask and scale
 * returned them); lse: [B, heads, N] float32. A row the forward gave
 * lse = -inf contributes nothing. dq, dk, dv are written (not accumulated)
 * and must not overlap the inputs. Each gradient row is reduced in a fixed
 * order (no atomics): results are deterministic. Uses the mask's transposed
 * block lists (built by va_mask_build) for dk and dv, and 8 * B * heads *
 * ceil(N / block) * block bytes of stream-ordered scratch (ceil(N / 128) * 128 for
 * bf16 with block 64).
 * Supported: VA_BF16, d in {64, 128}, block 128 or 64 on tcgen05 (block 64 as
 * 128-token tiles over pairs of blocks); VA_F32, d in {64, 128}, block in
 * {64, 128} on the FMA pipes,
 * B * heads <= 65535.
 * Errors: VA_ERR_INVALID (null or misaligned pointers, N != T*H*W of the
 * mask, B or heads < 1, non-finite scale, a mask built on another device),
 * VA_ERR_UNSUPPORTED, VA_ERR_OOM (scratch), VA_ERR_CUDA.
 */
int va_sparse_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, const va_mask* mask, void* dq,
                       void* dk, void* dv, int B, int heads, int N, int d, float scale,
                       int dtype, va_stream_t stream);

/*
 * The same attention with q, k, v, out (and lse, if not NULL) in HOST memory,
 * laid out as above; the library owns the device copies. The (batch, head)
 * slices go through a ring of device buffers in chunks: host-to-device
 * copies, the attention kernel and device-to-host copies run on three
 * internal streams ordered by events, so the transfers of one chunk overlap
 * the attention of another. The result is bit-identical to
 * va_sparse_attn_fwd on device copies of the same inputs.
 * Asynchronous on `stream` like the device call: the work starts after what
 * `stream` already holds, and later work on `stream` follows it. The host
 * buffers must stay valid, and out / lse must not be read, until `stream`
 * has completed (cudaStreamSynchronize). Page-locked host memory is needed
 * for the copies to overlap; pageable memory works with copies that stall
 * the host. Calls on one device are serialised on the internal streams.
 * Errors: as va_sparse_attn_fwd, plus VA_ERR_OOM (device buffers).
 */
int va_sparse_attn_fwd_host(const void* q, const void* k, const void* v, const va_mask* mask,
                            void* out, float* lse, int B, int heads, int N, int d, float scale,
                            int dtype, va_stream_t stream);

/*
 * Linear attention forward (LinVideo, gist.science 2510.08318, technical
 * summary sec. 1: attention in O(N) instead of O(N^2)). Non-causal, with the
 * feature map phi(x) = elu(x) + 1 (the page names none; this is the positive
 * map of Katharopoulos et al. 2020). For every batch b, head h, query i:
 *   out_i = sum_j (phi(q_i) . phi(k_j)) v_j / sum_j (phi(q_i) . phi(k_j))
 * computed as phi(q_i)^T S / phi(q_i)^T z with S = sum_j phi(k_j) v_j^T and
 * z = sum_j phi(k_j) (one read of K and V, one of Q). q, k, v, out:
 * [B, heads, N, d] device arrays. Supported: VA_BF16 with d = 64 or 128
 * (fp32 accumulation, bf16 output). Errors: VA_ERR_INVALID (null or misaligned
 * pointers, B, heads or N < 1), VA_ERR_UNSUPPORTED (other dtype or d),
 * VA_ERR_OOM, VA_ERR_CUDA.
 */
int va_linear_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int heads,
                       int N, int d, int dtype, va_stream_t stream);

/*
 * LinVideo's mixed attention of one layer (technical summary sec. 2 A: a
 * scalar r in [0, 1] selects quadratic attention at r = 1 and linear
 * attention at r = 0):
 *   out_i = r * att_i + (1 - r) * lin_i
 * with att the block-sparse softmax attention of va_sparse_attn_fwd under
 * `mask` (the dense mask gives full attention) and lin that of
 * va_linear_attn_fwd. r = 1 runs the attention only, r = 0 the linear
 * attention only. The attention part is rounded to bf16 before the blend.
 * Supported: VA_BF16, d = 64 or 128, mask block 64 or 128. Errors: as the two calls, and
 * VA_ERR_INVALID for r outside [0, 1], N != the mask's N or a mask built on
 * another device.
 */
int va_mixed_attn_fwd(const void* q, const void* k, const void* v, const va_mask* mask, float r,
                      void* out, int B, int heads, int N, int d, float scale, int dtype,
                      va_stream_t stream);

/*
 * LIPAR inter-frame pruning (LIPAR summary, sec. 2 B; readings, as the page
 * gives no formulas). x: device latent [B, T*H*W, C] of `dtype` (token
 * n = t*H*W + h*W + w). Per batch:
 *   changed(t, h, w) = t == 0 or max_c |x[t,h,w,c] - x[t-1,h,w,c]| >= tau
 *   keep(t, h, w)    = t == 0 or changed anywhere in the 3 x 3 spatial
 *                      neighbourhood of (h, w) in frame t (motion check)
 * Outputs (device, caller-owned): keep uint8 [B, N]; order int32 [B, N] whose
 * first count[b] entries list the kept tokens in token order (the compacted
 * sequence); src int32 [B, N], the compacted slot that restores token n (its
 * own slot if kept, else src of the same (h, w) in frame t - 1); count int32
 * [B]. The decisions use the largest channel difference, exact in float32.
 * Errors: VA_ERR_INVALID (null or misaligned pointers, sizes < 1, NaN tau),
 * VA_ERR_UNSUPPORTED (dtype, sizes), VA_ERR_OOM, VA_ERR_CUDA.
 */
int va_lipar_prune(const void* x, int B, int T, int H, int W, int C, float tau, int dtype,
                   uint8_t* keep, int32_t* order, int32_t* src, int32_t* count,
                   va_stream_t stream);

/*
 * Compaction of a [B, heads, N, d] device tensor to the kept tokens of
 * va_lipar_prune: out[b, h, k] = x[b, h, order[b, k]] for k < count[b] (rows
 * from count[b] on are left as they are), so out holds the shorter sequence
 * that attention then runs on. d * element size must be a multiple of 16
 * bytes; x and out 16-byte aligned. Errors: VA_ERR_INVALID,
 * VA_ERR_UNSUPPORTED, VA_ERR_CUDA.
 */
int va_lipar_gather(const void* x, const int32_t* order, const int32_t* count, int B, int heads,
                    int N, int d, int dtype, void* out, va_stream_t stream);

/*
 * Restoration (LIPAR summary, sec. 2 B): out[b, h, n] = y[b, h, src[b, n]]
 * expands a compacted [B, heads, N, d] result (first count[b] rows valid) to
 * the full sequence, a pruned token taking the result of its previous-frame
 * source. Same layout rules and errors as va_lipar_gather.
 */
int va_lipar_restore(const void* y, const int32_t* src, int B, int heads, int N, int d, int dtype,
                     void* out, va_stream_t stream);

/*
 * Lloyd k-means per (batch, head) on x [B, heads, N, d] (squared Euclidean
 * distance): SVG-EAR's clustering of query and key tokens by semantic
 * similarity (SVG-EAR, gist.science 2603.08982, technical summary sec. 2,
 * idea 1; the page names no algorithm, Lloyd's is the reading):
 *   centroid <- x[init_idx]; repeat iters times: assign each token to the
 *   nearest centroid (ties: lowest index), then replace each centroid by the
 *   mean of its members (an empty cluster keeps its centroid).
 * iters == 0 returns the assignment to the initial centroids.
 * init_idx: device int32 [B, heads, C], distinct indices in [0, N) (the
 * seeded random draw, supplied by the caller). Outputs (device, caller-owned):
 * assign int32 [B, heads, N], centroid float32 [B, heads, C, d] (means of the
 * returned assignment), count int32 [B, heads, C]. Distances are float32.
 * Deterministic: member sums are exact (bf16) or taken over member lists in
 * ascending token order (float32), so repeated calls are bit-identical.
 * Scratch: allocated and released on `stream` (stream-ordered allocator).
 * Supported: dtype VA_BF16 or VA_F32, d in {64, 128}, 1 <= C <= min(N, 4096).
 * Errors: VA_ERR_INVALID, VA_ERR_UNSUPPORTED, VA_ERR_OOM, VA_ERR_CUDA.
 */
int va_cluster(const void* x, const int32_t* init_idx, int B, int heads, int N, int d, int C,
               int iters, int dtype, int32_t* assign, float* centroid, int32_t* count,
               va_stream_t stream);

/*
 * va_cluster warm-started from given centroids instead of seed indices: the
 * clusters of the previous denoising step, say, so that a few iterations
 * refine them (SVG-EAR clusters queries and keys at every step; nearby steps
 * have nearby activations). centroid_init: device float32 [B, heads, C, d],
 * 16-byte aligned; it may be the same array as `centroid`. Starting from the
 * float copies of x[init_idx] gives exactly va_cluster's result, and k
 * iterations from the centroids after m give exactly the result after m + k.
 * Other arguments, outputs and errors as va_cluster.
 */
int va_cluster_from(const void* x, const float* centroid_init, int B, int heads, int N, int d,
                    int C, int iters, int dtype, int32_t* assign, float* centroid,
                    int32_t* count, va_stream_t stream);

/*
 * SVG-EAR compensated sparse attention with error-aware routing.
 * A block is (query cluster p, key cluster c); n_p, n_c are cluster sizes and
 * qc_p, kc_c, vc_c member means (float32) of q, k, v.
 *   probe (proxy qc_p, logits s*qc_p.k_j, m_p their max):
 *     Z_p = sum_j e^(l_j - m_p), O_p = sum_j e^(l_j - m_p) v_j / Z_p,
 *     dE = sum_{j in c} e^(l_j - m_p) v_j - n_c e^(s qc_p.kc_c - m_p) vc_c,
 *     dZ = sum_{j in c} e^(l_j - m_p)     - n_c e^(s qc_p.kc_c - m_p),
 *     err(p, c) = || dE - O_p dZ ||_2 / Z_p
 *   routing: ratio = err / n_c (float32); blocks ordered by ratio descending,
 *     ties by p then c ascending; the longest prefix whose summed cost
 *     n_p * n_c is <= floor(density * N * N) is computed exactly; blocks with
 *     an empty cluster are never selected;
 *   output for query i in cluster p: one softmax over the exact keys of the
 *     selected clusters and, for every other non-empty key cluster c, a
 *     virtual key kc_c with logit bias ln n_c and value vc_c.
 * qassign/kassign: device int32 [B, heads, N] with values in [0, Cq) / [0, Ck).
 * out: [B, heads, N, d] of dtype (bf16 for VA_BF16, float32 for VA_F32).
 * err_out: NULL or device float32 [B, heads, Cq, Ck] (the probe errors).
 * sel_out: NULL or device uint8 [B, heads, Cq, Ck] (1 = computed exactly).
 * Deterministic: the member lists hold each cluster's tokens in ascending
 * order, so repeated calls on the same inputs return bit-identical out,
 * err_out and sel_out.
 * Scratch: allocated and released on `stream` (stream-ordered allocator).
 * Supported: d in {64, 128}, 1 <= Cq, Ck <= 4096, 0 <= density <= 1.
 * Errors: VA_ERR_INVALID, VA_ERR_UNSUPPORTED, VA_ERR_OOM, VA_ERR_CUDA;
 * assignment values out of range are reported by va_device_error() as
 * VA_ERR_DEVICE.
 */
int va_compensate_route(const void* q, const void* k, const void* v, const int32_t* qassign,
                        int Cq, const int32_t* kassign, int Ck, double density, float scale,
                        int B, int heads, int N, int d, int dtype, void* out, float* err_out,
                        uint8_t* sel_out, va_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the sticky device error word of
 * the current device: VA_OK, VA_ERR_TIMEOUT or VA_ERR_DEVICE (or VA_ERR_CUDA
 * if the synchronisation itself failed).
 */
int va_device_error(va_stream_t stream);

/* Set the bound of every device-side wait in clock64 cycles (default 4e9,
 * about 2 s at 2 GHz). Values < 1000 are rejected with VA_ERR_INVALID. */
int va_set_wait_limit(int64_t cycles);

/*
 * Self-test of the bounded device waits used by every kernel (an interface
 * for failure-detection tests; the paper has no counterpart). Launches one
 * small CTA on `stream` that waits on a shared-memory mbarrier no thread
 * ever arrives at, with the wait bounded by `cycles` clock64 cycles (1e3 to
 * 1e10). The wait gives up, records VA_ERR_TIMEOUT in the device error word
 * and the kernel returns normally, so the CUDA context stays usable;
 * va_device_error() then reports VA_ERR_TIMEOUT once.
 * Errors: VA_ERR_INVALID (cycles out of range), VA_ERR_CUDA (launch).
 */
int va_selftest_wait_timeout(int64_t cycles, va_stream_t stream);

/*
 * Host-side validation of a block CSR (an interface for checks and tests; the
 * paper has no counterpart): row_ptr[nqb + 1] and col_idx[nnz] in HOST
 * memory. Valid means row_ptr[0] == 0, row_ptr[nqb] == nnz, rows
 * non-decreasing, and every row's columns strictly ascending in [0, nqb); with
 * require_diagonal, every row I also holds column I (the radial, LVSA and
 * dense rules always keep the diagonal block). Returns VA_OK, VA_ERR_DEVICE
 * for a list that breaks a rule, or VA_ERR_INVALID for null pointers or bad
 * sizes. When the environment variable VA_CHECKED is set (and not "0"),
 * va_mask_build validates its rows and transposed lists this way, and the
 * transposed lists as the exact transpose of the rows, before returning; a
 * failure frees the mask and returns VA_ERR_DEVICE.
 */
int va_csr_validate(const int32_t* row_ptr, const int32_t* col_idx, int nqb, int64_t nnz,
                    int require_diagonal);

/* Static text for a status code. */
const char* va_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int va_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VA_H */
