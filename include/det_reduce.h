/*
 * det_reduce.h -- C ABI of the deterministic multi-writer reduction library
 * (libdetreduce.so, CUDA for sm_103a).
 *
 * The operation.  For destination rows m = 0 .. M-1 of width H:
 *
 *     out[m][h] = SUM over { i : idx[i] = m } of  w[i] * x[i][h]
 *
 * computed so that the result is the same bits whatever the grid, the SM
 * count, the batch composition or how the sources are split into shards.
 * This is the MoE token combine/unpermute (out.index_add_(0, sorted_indices,
 * permuted_tokens) versus the atomic scatter_add_, "Megatron-LM determinism
 * developer reference", section 3.1, op catalog), the sparse-attention
 * backward key-gradient scatter and the MoE backward merge ("DeepSeek-V4
 * book, Ch 09: Batch invariance and determinism", sections 3.1 and 3.2), and,
 * without the index, the split-K partial-sum reduce (same chapter, section
 * 3.3).  Several writers to one address get private slots merged in one fixed
 * order ("Bit-exact training interview notes", table "where nondeterminism
 * comes from"), and every shard count goes through the same fp32 tree (same
 * page, "why pay the overhead", EP-size-invariant expert combine).
 *
 * The canonical order (fixed by this library; the pages fix the problem, not
 * a tree):
 *   1. the terms of destination m are the sources i with idx[i] = m in
 *      ascending order key (src_id[i] if given, else the physical row i);
 *   2. term p = fl32(w[i] * fl32(x[i][h])): one binary32 multiply rounded to
 *      nearest even, never fused with the add; no multiply when w is NULL;
 *   3. consecutive chunks of 32 terms are folded left to right, starting from
 *      the chunk's first term;
 *   4. chunk sums are combined by a level-wise pairwise tree: at each level
 *      neighbours (2k, 2k+1) are added and an odd last element is carried up
 *      unchanged, until one value remains;
 *   5. an empty destination gives +0.0;
 *   6. the value is stored as binary32 or rounded to bf16 (nearest even).
 * Every add is a binary32 add rounded to nearest even; subnormals are kept
 * (no flush to zero).
 *
 * Conventions.
 *  - Every function returns det_status (0 = DET_OK).  No function throws,
 *    aborts or prints.
 *  - "dev" pointers are CUDA device pointers of the current device; "host"
 *    pointers are ordinary host memory.  All tensor memory (inputs, outputs,
 *    workspaces) is owned by the caller; the library never allocates device
 *    memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued on it and the call returns without waiting,
 *    except det_reduce_plan, which waits once (see there).
 *  - Arguments are checked before anything is enqueued (fail closed): an
 *    option or argument the library cannot honour is an error, never a
 *    silent fallback.  On error nothing is written to any output.
 *  - No option in det_opts changes a single output bit.
 */
#ifndef DET_REDUCE_H
#define DET_REDUCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t det_status;

#define DET_OK 0
#define DET_ERR_ARG 1          /* NULL where data is needed, negative size, bad stride, aliasing, bad alignment */
#define DET_ERR_DTYPE 2        /* dtype code not supported */
#define DET_ERR_INDEX_RANGE 3  /* some idx[i] outside [0, M) */
#define DET_ERR_ORDER_KEY 4    /* two sources of one destination share a src_id: their order is undefined */
#define DET_ERR_WORKSPACE 5    /* workspace NULL, misaligned or smaller than the size query returned */
#define DET_ERR_CUDA 6         /* a CUDA call failed; det_last_cuda_error() gives the cudaError_t */
#define DET_ERR_TIMEOUT 7      /* a bounded device wait expired (reported when debug_checks is set) */
#define DET_ERR_UNSUPPORTED 8  /* size beyond a documented limit (N, M >= 2^31 - 1, more than DET_MAX_SHARDS shards) */

typedef int32_t det_dtype;
#define DET_F32 0   /* IEEE binary32 */
#define DET_BF16 1  /* bfloat16: the high 16 bits of a binary32 pattern */

#define DET_MAX_SHARDS 16

/*
 * Launch options.  Pass NULL for defaults.  None of them changes output bits;
 * tests sweep them to prove it.
 *  grid_ctas        0 = auto; > 0 = exact number of CTAs for the reduce
 *                   kernels (they loop over their work until done).
 *  seg_chunks_log2  -1 = auto (3); otherwise 3..6.  A destination with more
 *                   than 2^g chunks of 32 terms is split into segments of 2^g
 *                   chunks that run on different warps/CTAs; each segment is
 *                   one aligned node of the tree, written to a private fp32
 *                   partial slot, and a second pass applies the rest of the
 *                   tree in its fixed order.  Plan-time option.
 *  debug_checks     nonzero: the call waits for its kernels and reports a
 *                   CUDA error, or an expired bounded wait, as DET_ERR_CUDA /
 *                   DET_ERR_TIMEOUT (slower; for tests).
 *  gather_path      0 = auto.  1 = register-staged warp kernel, 2 = warp
 *                   kernel with cp.async copies into shared memory, 3 = TMA
 *                   bulk-staged kernels: with a waited plan whose
 *                   destinations all have at most 32 terms and rows of at
 *                   least 1 KB, one 64 KB stage per destination tile; else,
 *                   with 16-byte aligned source and out rows and H a
 *                   multiple of 16 bytes, a byte ring in shared memory for
 *                   the destinations of at most one chunk (also behind a
 *                   plan that did not wait), the longer ones on the
 *                   register-staged kernel beside it.  Auto, for rows of
 *                   at least 1 KB in one shard (in several shards, from 64
 *                   destination tiles per SM): the first where it applies;
 *                   behind a plan that did not wait, the first with its
 *                   tiling read from the device when every destination turns
 *                   out to have at most 32 terms, else path 1 after it; the
 *                   ring (one shard) when the sources are at least 1 GiB;
 *                   else path 1.
 *                   A path that does not apply fails with
 *                   DET_ERR_UNSUPPORTED.  Every path gives the same bits.
 *  tiles_per_task   0 = auto; > 0 = H-tiles one warp task of the warp kernels
 *                   covers (the work split changes no bit).
 *  async_plan       plan-time option.  0 (default): det_reduce_plan waits once
 *                   and reports index and order-key errors itself.  Nonzero:
 *                   det_reduce_plan only enqueues its kernels and returns; the
 *                   work counts stay on the device, where det_scatter_reduce
 *                   reads them, and errors are reported by det_plan_status.
 *                   If the plan recorded an error, det_scatter_reduce writes
 *                   nothing.  Lets plan and reduce run back to back (and be
 *                   captured in a CUDA graph).
 *  plan_path        plan-time option.  0 = auto.  1 = multi-kernel plan
 *                   (histogram, one radix pass per digit, work list).  2 =
 *                   single-cluster plan: one kernel on a thread-block cluster
 *                   of up to 16 CTAs holding the sources in distributed shared
 *                   memory; only without src_id, for N <= 131072 and
 *                   M <= 8192 x (cluster CTAs), and only where the device can
 *                   schedule the cluster (else DET_ERR_UNSUPPORTED).  3 =
 *                   owner plan: one kernel on clusters of 8 CTAs, one CTA per
 *                   SM, each cluster owning a range of at most 1024
 *                   destinations and reading all of idx; only without src_id,
 *                   for 1 <= N <= 262144 and M <= min(32768, 1024 x (SMs/8)),
 *                   and where the device can schedule the clusters (else
 *                   DET_ERR_UNSUPPORTED).  4 = radix plan: per 8-bit digit a
 *                   count, an offset and a scatter kernel over packed words,
 *                   the row lengths counted by the last pass, and one kernel
 *                   for the work list; only without src_id, for
 *                   1 <= N < 2^24 and M <= 65536 (else DET_ERR_UNSUPPORTED).
 *                   Auto takes path 3 where it applies and N <= 131072, else
 *                   path 2 where it applies and N <= 65536, else path 4 where
 *                   it applies, else path 1.  All build the same lists.
 *  reserved         must be zero.
 */
typedef struct det_opts {
    int32_t grid_ctas;
    int32_t seg_chunks_log2;
    int32_t debug_checks;
    int32_t gather_path;
    int32_t tiles_per_task;
    int32_t async_plan;
    int32_t plan_path;
    int32_t reserved[1];
} det_opts;

/* Opaque host handle of a built plan.  Its device arrays live in the
 * caller's plan workspace, which must stay allocated and unmodified while the
 * plan is used. */
typedef struct det_plan_s* det_plan;

/* Read-only description of a built plan (device pointers into the plan
 * workspace; counts are host values). */
typedef struct det_plan_desc {
    int64_t N, M;
    int32_t seg_chunks_log2;
    int32_t reserved;
    const int32_t* row_ptr;   /* dev [M+1]: exclusive prefix sums of destination counts, row_ptr[M] = N */
    const int32_t* perm;      /* dev [N]: perm[row_ptr[m] + r] = physical row of the r-th term of destination m */
    int64_t n_units;          /* warp tasks (before H-tiling): whole destinations + hot segments */
    int64_t n_segments;       /* hot segments = fp32 partial slots needed per H */
    int64_t n_hot_rows;       /* destinations split into segments */
    int64_t max_row_len;      /* largest number of terms of one destination */
    /* (the four counts are -1 for an async plan until det_plan_status) */
} det_plan_desc;

/* Text of a status code (static storage; never NULL). */
const char* det_status_str(det_status s);

/* The cudaError_t of the last failing CUDA call on this thread (0 if none). */
int32_t det_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
int32_t det_version(void);

/* Number of kernels this library has launched in this process (all threads,
 * all devices), for counting launches inside a timed region. */
int64_t det_kernel_launches(void);

/*
 * Bytes of device workspace a plan over N sources and M destinations needs
 * (with_src_id != 0: the plan will be given order keys).  host out-param.
 * Errors: DET_ERR_ARG (negative, NULL out), DET_ERR_UNSUPPORTED (N or M >=
 * 2^31 - 1).
 */
det_status det_plan_workspace_size(int64_t N, int64_t M, int32_t with_src_id,
                                   const det_opts* opts, size_t* bytes);

/*
 * Build the destination lists (CSR) and the work list of the reduce.
 *  idx        dev int32 [N]: destination of each physical source row.
 *  src_id     dev int64 [N] or NULL: order key of each physical row (NULL =
 *             the physical row number).  Keys must be distinct among the
 *             sources of one destination; they may be any int64 values
 *             (e.g. global token ids of a batch subset).  This is the MoE
 *             backward's stable (expert id, original token id) order, Ch 09
 *             section 3.2.
 *  workspace  dev, >= det_plan_workspace_size(N, M, src_id != NULL) bytes,
 *             256-byte aligned; holds the plan's device arrays afterwards.
 *  out_plan   host out-param; release with det_plan_destroy.
 * Steps on the device: a stable sort of the source rows by destination
 * (after a sort by src_id when given), the destination counts and their
 * exclusive scan (row_ptr), all integer and exact; then the work list (whole
 * destinations and hot segments).  Small problems without src_id run as one
 * kernel on one thread-block cluster, others as counting / scan / scatter
 * kernels per 8-bit radix digit (opts->plan_path); every method gives the
 * same arrays.  By default the call waits once for the stream to read the
 * error flags and the work counts; with opts->async_plan it only enqueues
 * (see det_plan_status).  The plan is reusable for any x, w, H, dtype and
 * shard split over the same idx.
 * Errors: DET_ERR_ARG, DET_ERR_WORKSPACE, DET_ERR_UNSUPPORTED,
 * DET_ERR_INDEX_RANGE (an idx outside [0, M)), DET_ERR_ORDER_KEY,
 * DET_ERR_CUDA.  On error *out_plan is NULL.
 */
det_status det_reduce_plan(const int32_t* idx, const int64_t* src_id, int64_t N, int64_t M,
                           void* workspace, size_t ws_bytes, const det_opts* opts,
                           void* stream, det_plan* out_plan);

/* Release the host handle (the workspace stays the caller's).  NULL is OK. */
det_status det_plan_destroy(det_plan plan);

/*
 * Wait for the plan's kernels on `stream` and report what they found:
 * DET_OK, DET_ERR_INDEX_RANGE or DET_ERR_ORDER_KEY (or DET_ERR_TIMEOUT if a
 * bounded wait of an earlier reduce with this plan expired).  For a plan
 * built with async_plan this is where errors surface; afterwards the work
 * counts are known on the host (det_plan_describe).  For a synchronous plan
 * it returns DET_OK.
 */
det_status det_plan_status(det_plan plan, void* stream);

/* Fill *desc (host) from a built plan. */
det_status det_plan_describe(det_plan plan, det_plan_desc* desc);

/*
 * Bytes of device workspace det_scatter_reduce needs for the hot-segment
 * partial slots at row width H (0 when the plan has no hot destination; for
 * an async plan whose counts are still on the device, an upper bound).
 */
det_status det_scatter_workspace_size(det_plan plan, int64_t H, size_t* bytes);

/*
 * out[m][0..H) = canonical sum over the terms of destination m (see top).
 *  x_shards    host array [P] of dev pointers; shard q holds the physical
 *              rows [R_q, R_q + shard_rows[q]), R_q = sum of earlier
 *              shard_rows, row r at x_shards[q] + (r - R_q) * ldx elements.
 *              Shards say only where bytes live; the order key is global, so
 *              P = 1, 2, 4, 8 give identical bits (simulated expert-parallel
 *              shards on one GPU).
 *  shard_rows  host int64 [P], summing to the plan's N.  1 <= P <=
 *              DET_MAX_SHARDS.
 *  x_dtype     DET_F32 or DET_BF16; ldx >= H elements.
 *  w           dev float [N] or NULL (no multiply).
 *  out         dev [M][ldo] of out_dtype, ldo >= H; overwritten, never
 *              accumulated into (elements h >= H of a row are not touched);
 *              must not overlap x, w, the plan workspace or `workspace`.
 *  workspace   dev, >= det_scatter_workspace_size(plan, H) bytes, 256-byte
 *              aligned (may be NULL when that size is 0).
 * Rows are read with 16-byte vector loads when every shard pointer is
 * 16-byte aligned and ldx, H are multiples of 16 bytes' worth of elements;
 * otherwise with scalar loads.  Both give the same bits.  Calls that take
 * the ring kernel (opts->gather_path) with one plan must not overlap on the
 * GPU: it claims work from a counter in the plan's workspace.
 * Errors: DET_ERR_ARG, DET_ERR_DTYPE, DET_ERR_WORKSPACE, DET_ERR_UNSUPPORTED,
 * DET_ERR_CUDA.
 */
det_status det_scatter_reduce(det_plan plan,
                              const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                              det_dtype x_dtype, int64_t ldx, int64_t H,
                              const float* w, void* out, int64_t ldo, det_dtype out_dtype,
                              void* workspace, size_t ws_bytes,
                              const det_opts* opts, void* stream);

/*
 * index_add_ with a deterministic order: the pages name index_add_ as the
 * deterministic replacement of the atomic scatter_add_ (Megatron-LM
 * determinism developer reference, section 3.1 op catalog).  Same arguments
 * as det_scatter_reduce, but `out` is read as well as written: every
 * destination m with at least one term becomes out[m] + S[m], one binary32
 * add (round to nearest even) of the canonical sum S[m] to the value already
 * there (bf16 out is read exactly as binary32), then stored as out_dtype;
 * destinations without terms are not touched.  Repeated calls accumulate
 * (e.g. embedding-gradient accumulation over micro-batches) and every call
 * gives the same bits for the same inputs and the same prior contents.
 * opts->gather_path 3 (16-byte aligned source rows, out rows 16-byte
 * aligned and H a multiple of 16 bytes of both x and out) runs
 * the destinations of 1..32 terms on the TMA-staged ring kernel, which also
 * copies each one's old out tile into shared memory, and the longer ones
 * on the register-staged kernel; auto does so where it applies, the sources
 * are one shard and rows are at least 1 KB, else it takes path 1.  Calls that
 * take the ring kernel with one plan must not overlap on the GPU: it claims
 * work from a counter in the plan's workspace.
 * gather_path 2 gives DET_ERR_UNSUPPORTED, as does 3 where it does not
 * apply.  Every path gives the same bits.  Other errors as
 * det_scatter_reduce.
 */
det_status det_index_add(det_plan plan,
                         const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                         det_dtype x_dtype, int64_t ldx, int64_t H,
                         const float* w, void* out, int64_t ldo, det_dtype out_dtype,
                         void* workspace, size_t ws_bytes,
                         const det_opts* opts, void* stream);

/*
 * det_scatter_reduce without a caller workspace.  The pages describe no such
 * call; it exists for callers that cannot allocate device memory when they
 * call in: code inside a larger runtime whose allocator owns all device
 * memory, a path that must not allocate after start-up, or a fixed interface
 * with no way to pass a scratch buffer.  The scratch that det_scatter_reduce
 * takes from `workspace` (fp32 partial slots for hot destinations) comes here
 * from a fixed 16 MiB array in the library's device image, which the module
 * loader reserves on every GPU that loads the library until the process exits.
 *  - Same arguments and results as det_scatter_reduce, minus the workspace.
 *  - Limit: det_scatter_workspace_size(plan, H) must be <= 16 MiB (16777216
 *    bytes), else DET_ERR_UNSUPPORTED and nothing is launched.
 *  - The first call on each device looks up the array's device address (once
 *    per device, with that device current) and keeps it; make that first call
 *    before any stream capture.  The address is kept together with the id of
 *    the context it belongs to: after a device reset the first call in the
 *    new context looks it up again (so that call, too, should not be inside
 *    a stream capture).
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs clearing (each slot is written before it is read),
 *    but calls whose work overlaps on the GPU (other streams, other threads)
 *    race on it: order them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
det_status det_scatter_reduce_noalloc(det_plan plan,
                                      const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                                      det_dtype x_dtype, int64_t ldx, int64_t H,
                                      const float* w, void* out, int64_t ldo, det_dtype out_dtype,
                                      const det_opts* opts, void* stream);

/*
 * Split-K reduce: out[e] = canonical sum over s = 0 .. S-1 (split-id order)
 * of partials[s * ldp + e], e = 0 .. count-1, no multiply (Ch 09, section
 * 3.3: each K-split writes its own buffer; a reduce kernel sums them in
 * split-id order).
 *  partials  dev float [S][ldp], ldp >= count.
 *  out       dev [count] of out_dtype; must not overlap partials.
 * Errors: DET_ERR_ARG, DET_ERR_DTYPE, DET_ERR_UNSUPPORTED, DET_ERR_CUDA.
 */
det_status det_splitk_reduce(const float* partials, int32_t S, int64_t count, int64_t ldp,
                             void* out, det_dtype out_dtype, const det_opts* opts, void* stream);

/*
 * Split-K GEMM with the split-id-ordered reduce in its epilogue: the producer
 * of the partials and their reduce in one kernel, so that the partials never
 * go to memory (Ch 09, section 3.3: the mHC backward is forced into split-K,
 * each split writes its own buffer and a reduce sums them in split-id order;
 * "Bit-exact training interview notes", table "where nondeterminism comes
 * from": several writers of one output get private slots merged in a fixed
 * order, as in a grouped-GEMM epilogue).
 *   P_s[r][c] = sum over the K/S values of k in split s (k in
 *               [s*K/S, (s+1)*K/S)) of A[r][k] * W[c][k], accumulated in
 *               binary32 by the tensor cores (bf16 products are exact; the
 *               order of that accumulation inside one split is the hardware's,
 *               the same for every call);
 *   out[r][c] = canonical sum over s = 0 .. S-1 of P_s[r][c]: the same fold
 *               as det_splitk_reduce (chunks of 32 splits left to right, then
 *               the level-wise pairwise tree), stored as out_dtype.
 *  A         dev bf16 [R][lda], K contiguous; lda >= K, lda*2 and A 16-byte
 *            aligned.
 *  W         dev bf16 [C][ldw] (the transposed right operand: row c holds
 *            column c of B), same rules; 1 <= C <= 32.
 *  K         a multiple of S, K/S a multiple of 64; 1 <= S <= 256.
 *  ab_dtype  DET_BF16 (the only input type).
 *  out       dev [R][ldo] of out_dtype, ldo >= C; overwritten.
 *  partials  NULL, or dev float [S][ldp] (ldp >= R*C): each split's P_s is
 *            also written there, row-major [R][C] (for checking the fold, or
 *            for an unfused reduce by det_splitk_reduce, which then gives
 *            the same out).
 * One CTA per 128 rows on tensor cores (tcgen05) with TMA-fed shared memory
 * (two issuing threads take the even and the odd splits; each split's MMAs
 * are issued by one thread, in K order); no workspace.  With opts->debug_checks the call waits and reports an
 * expired bounded wait as DET_ERR_TIMEOUT.
 * Errors: DET_ERR_ARG, DET_ERR_DTYPE, DET_ERR_UNSUPPORTED (C > 32, S > 256,
 * K not S x a multiple of 64), DET_ERR_CUDA, DET_ERR_TIMEOUT.
 */
det_status det_splitk_gemm_reduce(const void* A, int64_t lda, const void* W, int64_t ldw, int64_t R, int32_t C,
                                  int64_t K, int32_t S, det_dtype ab_dtype, void* out, int64_t ldo,
                                  det_dtype out_dtype, float* partials, int64_t ldp, const det_opts* opts,
                                  void* stream);

/*
 * u64 fingerprint of nbytes bytes at dev pointer p, written to dev *out.
 * The repeatability gate compares per-tensor fingerprints byte for byte
 * instead of a printed loss ("Bit-exact training interview notes", "how to
 * verify: three gates").  Definition (this library's, not torch.hash_tensor):
 *   h = mix(nbytes ^ 0x6A09E667F3BCC909)
 *       + sum_j mix(word_j ^ (j * 0x9E3779B97F4A7C15))   mod 2^64,
 * word_j = bytes [8j, 8j+8) read little-endian, zero-padded past nbytes, and
 * mix = the SplitMix64 finalizer.  Integer sums commute, so the value does
 * not depend on the grid.  p may have any alignment.  *out is overwritten.
 * Errors: DET_ERR_ARG (p NULL with nbytes > 0, out NULL or not 8-byte
 * aligned), DET_ERR_CUDA.
 */
det_status det_hash(const void* p, uint64_t nbytes, uint64_t* out, void* stream);

/*
 * Sorted router top-k: for each token t, the k experts of greatest score,
 * greatest first.  The pages name the sorted router top-k among the hot
 * spots of the deterministic path ("Megatron-LM determinism developer
 * reference", section 3.3) but fix no tie rule; this library's:
 *   order  IEEE 754 totalOrder of the binary32 scores (-0.0 below +0.0, +NaN
 *          above +inf, -NaN below -inf), and among equal bit patterns the
 *          lower expert id first;
 *   w      the chosen scores, bit for bit; with renormalize != 0 each divided
 *          (one binary32 division, nearest even) by their binary32 sum taken
 *          left to right from the greatest.
 * The score function (softmax, sigmoid, ...) is the caller's: scores may be
 * probabilities or logits.
 *  scores    dev float [T][lds], lds >= E.
 *  topk_ids  dev int32 [T][k].
 *  topk_w    dev float [T][k], or NULL for ids only (not with renormalize).
 *  1 <= k <= E.  Outputs must not overlap scores or each other.
 * Errors: DET_ERR_ARG, DET_ERR_UNSUPPORTED (E > 1024, k > 32, T*k >= 2^31-1),
 * DET_ERR_CUDA.
 */
det_status det_router_topk(const float* scores, int64_t T, int32_t E, int64_t lds, int32_t k,
                           int32_t renormalize, int32_t* topk_ids, float* topk_w, void* stream);

/* Bytes of device workspace det_moe_route_plan needs for T tokens, top-k, E
 * experts.  Errors: DET_ERR_ARG, DET_ERR_UNSUPPORTED. */
det_status det_moe_route_workspace_size(int64_t T, int32_t k, int32_t E, const det_opts* opts,
                                        size_t* bytes);

/*
 * The integer side of the MoE dispatch and combine, straight from top-k
 * routing: the dispatch layout and the combine's plan in one call.  Slot
 * i = t*k + j is token t's j-th choice topk_ids[i].  The dispatch rows are
 * the slots sorted stably by expert: expert 0's slots in ascending slot
 * order, then expert 1's, ... -- for distinct choices per token, the stable
 * (expert id, original token id) order of the MoE backward ("DeepSeek-V4
 * book, Ch 09: Batch invariance and determinism", section 3.2).  The combine
 * adds every dispatch row back into its token (the index_add_ of the
 * Megatron-LM reference's op catalog, section 3.1).
 *  topk_ids        dev int32 [T*k], each in [0, E) (a token may repeat one).
 *  topk_w          dev float [T*k] or NULL.
 *  expert_offsets  dev int32 [E+1]: expert e's rows are
 *                  [expert_offsets[e], expert_offsets[e+1]); the last is T*k.
 *  row_token       dev int32 [T*k]: token of each dispatch row (the combine's
 *                  idx).
 *  row_w           dev float [T*k] or NULL: topk_w of each dispatch row's
 *                  slot (needs topk_w).
 *  slot_row        dev int32 [T*k] or NULL: dispatch row of each slot.
 *  workspace       dev, >= det_moe_route_workspace_size(T, k, E) bytes,
 *                  256-byte aligned; holds the plan's arrays afterwards.
 *  out_plan        host out-param: the combine's plan over M = T
 *                  destinations, with the same lists and work counts that
 *                  det_reduce_plan(row_token, NULL, T*k, T) builds.  Use it
 *                  with det_scatter_reduce / det_index_add on x in dispatch
 *                  row order and w = row_w.  Release with det_plan_destroy.
 * Every token has exactly k terms, so the combine lists follow from each
 * slot's rank in (expert, j) order inside its token; the only sort is the
 * one by expert.  Small problems (E <= 256, T*k <= 131072) run as one kernel
 * on a thread-block cluster, others as the destination-list plan over the
 * expert ids plus two kernels (opts->plan_path 0 = auto, 1 = the latter, 2 =
 * the cluster kernel or DET_ERR_UNSUPPORTED); both give the same bytes.
 * opts->async_plan and opts->seg_chunks_log2 as for det_reduce_plan.
 * Outputs must not overlap the inputs, each other or the workspace.
 * Errors: DET_ERR_ARG, DET_ERR_WORKSPACE, DET_ERR_UNSUPPORTED,
 * DET_ERR_INDEX_RANGE (an id outside [0, E): no output is written),
 * DET_ERR_CUDA.  On error *out_plan is NULL.
 */
det_status det_moe_route_plan(const int32_t* topk_ids, const float* topk_w, int64_t T, int32_t k,
                              int32_t E, int32_t* expert_offsets, int32_t* row_token, float* row_w,
                              int32_t* slot_row, void* workspace, size_t ws_bytes,
                              const det_opts* opts, void* stream, det_plan* out_plan);

/*
 * Bytes of workspace det_atomic_scatter_reduce needs: 256 bytes of flags, plus
 * an fp32 [M][H] accumulator when out_dtype is DET_BF16.
 */
det_status det_atomic_workspace_size(int64_t M, int64_t H, det_dtype out_dtype, size_t* bytes);

/*
 * NOT DETERMINISTIC -- benchmark baseline only.  The atomic twin of
 * det_scatter_reduce (scatter_add_ in the op catalog): out is zeroed, then
 * each term w[i] * x[i][h] (binary32 multiply) is added to out[idx[i]][h]
 * with atomic adds whose order the scheduler picks.  bf16 output: the adds
 * go to the fp32 accumulator in the workspace, which is then rounded to bf16
 * (nearest even).  Sources whose idx is outside [0, M) are skipped and
 * counted in the workspace flags; with opts->debug_checks the call waits and
 * returns DET_ERR_INDEX_RANGE if any were seen.
 * Arguments as det_scatter_reduce, with idx (dev int32 [N]) instead of a plan.
 */
det_status det_atomic_scatter_reduce(const int32_t* idx, int64_t N, int64_t M,
                                     const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                                     det_dtype x_dtype, int64_t ldx, int64_t H,
                                     const float* w, void* out, int64_t ldo, det_dtype out_dtype,
                                     void* workspace, size_t ws_bytes,
                                     const det_opts* opts, void* stream);

/*
 * NOT DETERMINISTIC -- benchmark baseline only.  The atomic twin of
 * det_index_add: each term is atomically added to out[idx[i]][h] as it is
 * (no zeroing), so destinations without terms are untouched.  fp32 out only
 * (DET_ERR_UNSUPPORTED for bf16).  Arguments and workspace as
 * det_atomic_scatter_reduce.
 */
det_status det_atomic_index_add(const int32_t* idx, int64_t N, int64_t M,
                                const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                                det_dtype x_dtype, int64_t ldx, int64_t H,
                                const float* w, void* out, int64_t ldo, det_dtype out_dtype,
                                void* workspace, size_t ws_bytes,
                                const det_opts* opts, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DET_REDUCE_H */
