/*
 * smx.h - C ABI of the GB300 (sm_103a) row-wise numerically stable softmax.
 *
 * Operation (all calls): for each row r of a contiguous row-major [rows, cols]
 * input x, with valid prefix length L_r (valid_len[r] clamped to [0, cols], or
 * cols when valid_len is NULL),
 *
 *     m_r = max_{j < L_r} x[r, j]
 *     d_r = sum_{j < L_r} exp(x[r, j] - m_r)
 *     y[r, j] = exp(x[r, j] - m_r) / d_r   for j < L_r,   +0 for j >= L_r.
 *
 * This is the max-shifted softmax of "Softmax numerics architecture - max
 * subtract, fp32 accumulate, fusion, online" (sections "The max-subtraction
 * identity, and why it is exact" and "Online softmax: one recurrence, one fewer
 * pass") and of "Kernel visualization: online softmax" ("Overview of safe
 * softmax").  (m, d) is the block summary of "Stable softmax: keep the
 * normalizer consistent as tiles arrive" and "Online stable softmax" ("Derive the
 * update for two blocks"); d is in natural-log units.
 *
 * Declared policy for the cases those pages say need one ("Stable softmax...",
 * second paragraph; "Online stable softmax", "Masks, empty rows, and
 * precision"):
 *   - masked lanes (j >= L_r) are excluded from the max and the sum and output +0;
 *   - a row with L_r == 0, or whose valid lanes are all -inf, outputs +0 in every
 *     lane; its statistics are (-inf, 0), the identity of the merge;
 *   - a -inf valid lane outputs +0 and the rest of the row is normal;
 *   - a NaN in the valid prefix makes every valid lane NaN; statistics (NaN, NaN);
 *   - a +inf in the valid prefix (and no NaN) makes every valid lane NaN, as the
 *     stable formula evaluates inf - inf; statistics (+inf, NaN).
 *
 * Precision: inputs are fp32, fp16 or bf16; the running maximum and the sum are
 * held in fp32 whatever the input and output types ("Why the accumulator is
 * fp32 even when the inputs are not"); the output type is chosen separately.
 *
 * Memory and ownership: every data pointer is a device pointer owned by the
 * caller; the library never frees or retains it.  On first use of a device it
 * allocates one status word and creates one memory pool.  The long-row paths
 * (rows too long for one CTA) and the staged host-buffer call keep their
 * scratch (stripe and chunk summaries: 8 bytes per stripe or 4096-element
 * chunk; per-row counters; staging slots) in per-device buffers from that
 * pool that only grow: a call that needs more than any call before reallocates
 * the buffer (stream-ordered), every other call allocates nothing.  Calls that
 * use the scratch are ordered on the device: a call on a stream other than
 * the previous user's first waits (cudaStreamWaitEvent) for the event recorded
 * after that user.  smx_softmax_rows_fixed_scratch uses a fixed array instead.
 * No other call allocates.
 * Every call is asynchronous on `stream` (NULL is the legacy default stream) and
 * returns after enqueueing its kernels.
 *
 * Errors: arguments are checked on the host before any launch; a bad argument
 * returns an error code and nothing is enqueued.  A failed launch returns
 * SMX_ERR_LAUNCH.  Errors found on the device (a bounded wait that ran out)
 * are recorded in the device status word, read with smx_last_device_status().
 */
#ifndef SMX_H
#define SMX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *smx_stream_t;

typedef enum {
    SMX_F32 = 0,  /* IEEE binary32 */
    SMX_F16 = 1,  /* IEEE binary16 */
    SMX_BF16 = 2  /* bfloat16: 8 exponent bits, 7 stored significand bits */
} smx_dtype;

typedef enum {
    SMX_OK = 0,
    SMX_ERR_INVALID_ARG = 1, /* NULL pointer with rows*cols > 0, negative size, bad dtype */
    SMX_ERR_UNSUPPORTED = 2, /* no CUDA device, or the device is not sm_103 */
    SMX_ERR_ALIAS = 3,       /* input and output byte ranges overlap */
    SMX_ERR_LAUNCH = 4,      /* a kernel launch failed (the CUDA error is in smx_last_cuda_error) */
    SMX_ERR_TIMEOUT = 5,     /* device: a bounded wait for staged data ran out */
    SMX_ERR_DEVICE = 6,      /* a CUDA runtime call failed */
    SMX_ERR_TOO_LARGE = 7    /* smx_softmax_rows_fixed_scratch: a row needs more scratch than it has */
} smx_status;

/*
 * Softmax of each row.
 *   x          device, [rows, cols] row-major, in_dtype; read only.
 *   y          device, [rows, cols] row-major, out_dtype; fully written, masked
 *              lanes included.  Must not overlap x (SMX_ERR_ALIAS).
 *   rows, cols >= 0; rows == 0 or cols == 0 enqueues nothing and returns SMX_OK.
 *   valid_len  device int32[rows] or NULL; each entry is clamped to [0, cols].
 *   in_dtype, out_dtype: any of the three types, independently.
 * Any alignment and any cols are accepted; 16-byte aligned x and y with
 * cols * sizeof(type) a multiple of 16 take the vectorised kernels.
 */
smx_status smx_softmax_rows(const void *x, void *y, int64_t rows, int64_t cols,
                            const int32_t *valid_len, smx_dtype in_dtype,
                            smx_dtype out_dtype, smx_stream_t stream);

/*
 * smx_softmax_rows with the input, the output and valid_len in HOST memory:
 * the same result, for callers whose rows live on the host.  Two ways, the
 * same arithmetic:
 *  - In place: when x, y (and valid_len, if given) are page-locked buffers
 *    mapped into the device's address space (cudaHostAlloc / cudaHostRegister
 *    memory on a unified-addressing system) and the rows take a kernel that
 *    reads each element once with plain loads (the streamed and
 *    register-resident rows: at most 32,768 elements, 16,384 for fp32
 *    outputs), one launch reads x and writes y in host memory over the host
 *    link.
 *  - Staged, otherwise (pageable buffers; longer rows, which the cluster and
 *    long-row kernels take; unaligned rows): the rows pass through
 *    two device staging slots (the library's per-device scratch) in
 *    chunks of about 16 MiB of input: chunk i's copy to the device and its
 *    softmax run on `stream`, its copy back on a second stream the library
 *    owns, so both directions of the host link and the kernels run at once.
 *    Pageable memory gives the same result with the copies serialised.
 *   x, y      host, [rows][cols] row-major, in_dtype / out_dtype; must not overlap.
 *   valid_len host int32[rows] or NULL.
 * Asynchronous on `stream`: y holds the result once `stream` has completed
 * (for instance after smx_last_device_status(stream)); the host buffers must
 * stay valid and untouched until then.  Argument errors are returned before
 * anything is enqueued.
 */
smx_status smx_softmax_rows_host(const void *x, void *y, int64_t rows, int64_t cols,
                                 const int32_t *valid_len, smx_dtype in_dtype,
                                 smx_dtype out_dtype, smx_stream_t stream);

/*
 * smx_softmax_rows, computed without allocating any device memory.
 *
 * The method's pages have no counterpart to this call; it exists for callers
 * that cannot let a library allocate: a process whose device memory is all
 * handed out by its own allocator under a fixed budget, or a steady-state loop
 * that must never meet an allocator's latency or an out-of-memory failure in
 * the middle of a step.  smx_softmax_rows takes a small stream-ordered
 * allocation per call on its long-row path; this call runs that path with its
 * chunk summaries in one fixed array of 256 KiB of device memory that the
 * library holds per device from the time it is loaded.
 *
 * Arguments, results, policy and errors are those of smx_softmax_rows (the
 * outputs agree with it within the stated tolerances: the same arithmetic, in
 * the long-row kernels for every row length).  Inputs that are not 16-byte
 * aligned, or whose row size in bytes is not a multiple of 16, run the scalar
 * kernel, which takes no scratch.
 *
 * Limit: one row's chunk summaries must fit the array: at most 32768 chunks of
 * 4096 elements, i.e. cols <= 134217728; a longer aligned row returns
 * SMX_ERR_TOO_LARGE before anything is enqueued.  Rows are processed in slabs
 * small enough for the array.
 *
 * Set-up: the first call on each device queries its properties and looks up
 * the array's address (the device must be current); make that first call
 * before capturing the stream into a graph or otherwise relying on the call
 * doing nothing but enqueue kernels.  Nothing in the array needs to start at
 * zero: every summary is written before it is read, within the same call.
 *
 * Concurrency: all calls on one device share the one array.  Two calls whose
 * kernels can overlap on the device (different streams with no ordering between
 * them) race on it and may produce wrong results; order them on one stream or
 * with events.
 */
smx_status smx_softmax_rows_fixed_scratch(const void *x, void *y, int64_t rows, int64_t cols,
                                          const int32_t *valid_len, smx_dtype in_dtype,
                                          smx_dtype out_dtype, smx_stream_t stream);

/*
 * Block summary (m, d) of each row, fp32.
 *   x, rows, cols, valid_len, in_dtype: as for smx_softmax_rows.
 *   m_out, d_out: device float[rows], written.  d is sum exp(x - m) (natural
 *   units).  Policy values as in the header comment: (-inf, 0) for empty or
 *   all -inf rows, (NaN, NaN) with a NaN, (+inf, NaN) with a +inf.
 */
smx_status smx_softmax_row_stats(const void *x, float *m_out, float *d_out, int64_t rows,
                                 int64_t cols, const int32_t *valid_len, smx_dtype in_dtype,
                                 smx_stream_t stream);

/*
 * log_softmax of each row ("Softmax numerics architecture - max subtract, fp32
 * accumulate, fusion, online", section "Log-sum-exp: log-probabilities without
 * probabilities"): y[r, j] = x[r, j] - LSE_r over the valid prefix, evaluated as
 * (x - m) - log d so that a large m adds no rounding, and -inf (the log of the
 * +0 probability) in masked lanes.  Policy (the softmax policy in log space):
 * an empty or all -inf row is -inf everywhere; a NaN or +inf row has NaN in its
 * valid lanes and -inf in its masked lanes.
 *   Arguments, types, alignment, aliasing and errors: as smx_softmax_rows.
 */
smx_status smx_log_softmax_rows(const void *x, void *y, int64_t rows, int64_t cols,
                                const int32_t *valid_len, smx_dtype in_dtype,
                                smx_dtype out_dtype, smx_stream_t stream);

/*
 * Log-sum-exp of each row (same section): LSE_r = m_r + log d_r, fp32.
 *   lse_out: device float[rows], written.  -inf for an empty or all -inf row,
 *   NaN for a NaN or +inf row.  Other arguments as smx_softmax_row_stats.
 */
smx_status smx_softmax_lse(const void *x, float *lse_out, int64_t rows, int64_t cols,
                           const int32_t *valid_len, smx_dtype in_dtype, smx_stream_t stream);

/*
 * Normalise each row with given statistics: y[r, j] = exp(x[r, j] - m[r]) / d[r]
 * over the valid prefix, +0 beyond.  This is the last step of a softmax whose
 * row statistics were computed in pieces and merged ("Online stable softmax",
 * "Derive the update for two blocks": only the prefix's m and d are needed),
 * e.g. over column blocks of a row held in different buffers: row_stats per
 * block, merge_stats, then apply_stats per block.
 *   m_in, d_in: device float[rows]; (m, d) must be statistics of a set of
 *   values containing the row's valid prefix (m at least its maximum, d >= 1 when
 *   m is finite), as row_stats and merge_stats produce; otherwise the lanes are
 *   whatever the arithmetic gives.  m == -inf gives a +0 row; a NaN m or d, or
 *   m == +inf, gives NaN in the valid lanes.
 *   y must not overlap x, m_in, d_in or valid_len.  Other arguments as
 *   smx_softmax_rows.
 */
smx_status smx_softmax_apply_stats(const void *x, const float *m_in, const float *d_in, void *y,
                                   int64_t rows, int64_t cols, const int32_t *valid_len,
                                   smx_dtype in_dtype, smx_dtype out_dtype, smx_stream_t stream);

/*
 * Softmax backward ("Softmax numerics architecture...", section "The
 * Jacobian, and the backward pass that never divides"): the vector-Jacobian
 * product, without forming the Jacobian diag(p) - p p^T:
 *     dx[r, j] = p[r, j] (g[r, j] - s_r),   s_r = sum_{k < L_r} g[r, k] p[r, k]
 * over the valid prefix, dx = 0 in masked lanes.
 *   p        device [rows, cols], dtype: the forward softmax as stored.
 *   g        device [rows, cols], dtype: the upstream gradient dL/dy.
 *   dx       device [rows, cols], dx_dtype: written (masked lanes included).
 *            Must not overlap p, g or valid_len (SMX_ERR_ALIAS).
 *   valid_len, rows, cols: as smx_softmax_rows.  The sum is fp32 whatever the
 *   types.  A NaN among a row's valid p or g makes its valid lanes NaN.
 *   Long rows are read once where their stripes of p and g fit the SMs'
 *   shared memory (one cooperative launch; the partial sums are added in a
 *   fixed order, so the result does not depend on timing).
 */
smx_status smx_softmax_backward(const void *p, const void *g, void *dx, int64_t rows, int64_t cols,
                                const int32_t *valid_len, smx_dtype dtype, smx_dtype dx_dtype,
                                smx_stream_t stream);

/*
 * Cross-entropy with logits and its fused gradient ("Softmax numerics
 * architecture...", sections "Log-sum-exp: log-probabilities without
 * probabilities" and "The Jacobian, and the backward pass that never divides"):
 *     loss[r] = LSE_r - x[r, t_r] = (m_r - x[r, t_r]) + log d_r      (fp32)
 *     grad[r, j] = p[r, j] - [j == t_r]   over the valid prefix, 0 beyond.
 * The gradient is formed directly (never through -1/p), so every component
 * lies in [-1, 1].
 *   x        device [rows, cols] logits, in_dtype.
 *   target   device int64[rows]: the target index of each row.  A target
 *            outside [0, L_r) is ignored: loss 0 and a zero gradient row.
 *   loss     device float[rows], written.  NaN for a row with a valid target
 *            whose valid prefix holds a NaN or +inf or only -inf.
 *   grad     device [rows, cols] in grad_dtype, written; or NULL for the loss
 *            alone (one read of x).  Must not overlap x, target, loss or
 *            valid_len.
 *   valid_len, rows, cols: as smx_softmax_rows.
 */
smx_status smx_cross_entropy(const void *x, const int64_t *target, float *loss, void *grad,
                             int64_t rows, int64_t cols, const int32_t *valid_len, smx_dtype in_dtype,
                             smx_dtype grad_dtype, smx_stream_t stream);

/*
 * Attention forward with the online weighted numerator ("Online stable
 * softmax", "Carry a weighted value numerator for attention" and "Reference
 * summary"; "Softmax numerics architecture...", "From online softmax to tiled
 * attention"): for each head h and query row i, with s_j = scale q_i . k_j over
 * the valid keys,
 *     o_i = sum_j e^(s_j - m) v_j / l,   l = sum_j e^(s_j - m),   m = max s_j,
 *     lse_i = m + log l,
 * computed block by block with the running state (m, l, o) so that the score
 * matrix never leaves the chip.  Scores, m, l and o are fp32; the probabilities
 * enter the second product rounded to the input type.
 *   q        device [heads][seq_q][head_dim], dtype; k, v: [heads][seq_k][head_dim].
 *            (heads = batch x heads, each head contiguous.)  16-byte aligned.
 *   o        device, like q, written.  Must not overlap q, k, v or lse.
 *   lse      device float[heads][seq_q], written; or NULL.
 *   head_dim 64 or 128 (else SMX_ERR_UNSUPPORTED); heads <= 65535.
 *   scale    > 0, e.g. 1/sqrt(head_dim).
 *   causal   0: every key; 1: key j is valid for query i when
 *            j <= i + seq_k - seq_q (bottom-right aligned).  A row with no
 *            valid key is the declared empty row: o = 0, lse = -inf.
 *   dtype    SMX_F16 or SMX_BF16 (the tensor-core input types).
 */
smx_status smx_attention_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                                 int64_t heads, int64_t seq_q, int64_t seq_k, int head_dim,
                                 double scale, int causal, smx_dtype dtype, smx_stream_t stream);

/*
 * Element-wise merge of two arrays of block summaries ("Online stable softmax",
 * "Derive the update for two blocks"):
 *   m' = max(m_a, m_b),  d' = d_a exp(m_a - m') + d_b exp(m_b - m').
 * An operand with m == -inf is the empty block and yields the other operand
 * unchanged; a NaN m gives (NaN, NaN); m' == +inf gives (+inf, NaN).
 *   all pointers: device float[n]; m_out/d_out may alias m_a/d_a or m_b/d_b
 *   exactly (in place), but must not partially overlap them.
 */
smx_status smx_softmax_merge_stats(const float *m_a, const float *d_a, const float *m_b,
                                   const float *d_b, float *m_out, float *d_out, int64_t n,
                                   smx_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the status word of the
 * current device: SMX_OK, or the first device-side error (SMX_ERR_TIMEOUT)
 * recorded by a kernel since the last read.
 */
smx_status smx_last_device_status(smx_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *smx_status_string(smx_status status);

/* The cudaError_t value (as int) of the last failed CUDA call on this thread, 0 if none. */
int smx_last_cuda_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int smx_version(void);

/*
 * Testing hooks.  Process-wide, not thread-safe; they exist so that tests can
 * reach every kernel on the shapes they choose.
 *
 * smx_debug_force_path(p): 0 = automatic choice; 1 = register-resident rows;
 *   2 = thread-block-cluster rows; 3 = generic (scalar, two-pass) rows;
 *   4 = persistent rows with the next rows prefetched (cp.async); 5 = long
 *   rows in chunks, in slabs of rows (chunk summaries, then merge and
 *   normalise; one slab of all rows unless smx_debug_set_split_slab); 6 =
 *   long rows read once, each row in column stripes held in the shared
 *   memory of a cooperative grid (softmax, log_softmax, cross-entropy with a
 *   gradient, and the backward: the stripes of p and g).  A forced path that
 *   cannot run the shape falls back to the automatic choice.
 * smx_debug_set_cluster(n): cap the cluster size of path 2 (1, 2, 4, 8, 16;
 *   0 = automatic); smem_bytes caps its shared-memory staging (0 = automatic).
 * smx_debug_set_wait_limit(n): n > 0: polls of a staging barrier (path 2)
 *   or of a tensor-core barrier (the tcgen05 attention kernel) before the
 *   kernel gives up and records SMX_ERR_TIMEOUT; 0 = default; n < 0: each CTA
 *   of path 2, and of the tcgen05 attention kernel, first waits -n polls on a
 *   barrier that nothing signals, records SMX_ERR_TIMEOUT when that wait runs
 *   out (it always does), then works normally -- a deterministic probe of the
 *   error path.
 * smx_debug_last_path(): the path (1..6) the last softmax/stats call on this
 *   thread used, 0 if none.
 * smx_debug_last_launches(): kernels the last call on this thread launched.
 * smx_debug_set_regs_shape(threads, vpt): on paths 1 and 4, use CTAs of
 *   `threads` threads per row (32 = one warp per row, path 1 only) holding `vpt`
 *   16-byte vectors each, when that shape covers the row (0, 0 = automatic).
 * smx_debug_set_stream_depth(n): rows prefetched per walker (CTA or warp) on path 4 (2, 3 or
 *   4; 0 = automatic).
 * smx_debug_set_stream_ctas(n): n resident CTAs per SM on path 4, at most as
 *   many as fit (0 = automatic; also path 5).
 * smx_debug_set_split_slab(bytes): slab size of path 5 (0 = one slab of all rows).
 * smx_debug_set_inflight(read_only, backward): bytes of reads to keep in flight
 *   per SM (which sets the persistent CTAs per SM) for the read-only
 *   statistics / LSE rows and for the backward (0 = default).
 * smx_debug_set_stream_warp(off): 1 = path 4 walks every row with a whole CTA;
 *   0 = rows that fit one warp are walked a row per warp (default).
 * smx_debug_set_split_fused(on): 1 = path 5 runs one cooperative launch for
 *   all slabs with per-row completion counts (where supported); 0 = two
 *   launches per slab, the statistics pass and then the normalising pass
 *   (default).
 * smx_debug_set_host_chunk(bytes, slots, staged): smx_softmax_rows_host's
 *   chunk size in input bytes and its number of device staging slots (2 to
 *   4), 0 = default for either; staged = 1 sends mapped page-locked buffers
 *   through the staging slots too (0 = in place where possible).
 * smx_debug_set_attention_kernel(which): the attention forward's kernel:
 *   -1 = chosen by the call (default): 3 for causal calls, 0 otherwise;
 *   0 = one 128-row query tile per CTA, two CTAs an SM, on the tcgen05
 *   tensor cores, operands copied by the row threads; 1 = persistent CTAs of
 *   one tile, K and V fetched by tensor-map bulk copies in their own warps;
 *   2 = the mma.sync kernel (warp-level tensor-core instructions); 3 =
 *   persistent CTAs of two query tiles, one CTA an SM, sharing tensor-map
 *   fetched K and V stages.  Kernels 1 and 3 take calls with seq_k > 0
 *   (kernel 0 the rest).  Other values select -1.
 * smx_debug_set_split_hints(stats, apply): L2 policy of path 5's reads in its
 *   statistics and normalising passes: 0 = none, 1 = evict last, 2 = evict
 *   first; -1 = automatic (1 and 2).
 * smx_debug_set_cluster_staging(m): how path 2 stages its shared-memory part:
 *   1 = bulk asynchronous copies (TMA) with one mbarrier per piece, 2 = per-
 *   thread cp.async; 0 = automatic.
 * smx_debug_alloc_count(): device allocations, events and streams the library
 *   has created in this process (a steady loop of calls adds none).
 * smx_debug_probe_math(a, b, out, n, which, stream): out[i] = the library's
 *   device primitive `which` at a[i] (and b[i]), for measuring its error:
 *   0 = ex2.approx.ftz.f32 2^a, 1 = ex2.approx.f32 2^a (keeps subnormal
 *   results), 2 = rcp.approx.ftz.f32 1/a, 3 = the refined reciprocal the
 *   kernels normalise with, 4 = the compensated e^(a - b) of fp32 outputs,
 *   5 = one term e^(a - b) as the statistics path forms it.  a, b, out:
 *   device float[n] (b only for 4 and 5).  The pages have no counterpart.
 * smx_debug_set_stripe_tuning(lag, piece_bytes, l2_ahead): path 6's rows of
 *   lag between a stripe's summary and its normalisation (1..6, at most the
 *   ring's slots - 2; 0 =
 *   default), the size of the bulk copies a stripe is fetched in (a multiple
 *   of 16; 0 = one copy per stripe; -1 = default) and how many rows past
 *   each fill the producer prefetches that row's stripe into L2 (0 = off;
 *   -1 = default).
 * smx_debug_set_count_probe(polls): polls > 0: the per-row count waits of
 *   the cooperative long-row kernels (path 6, and path 5 in its single-launch
 *   form) wait for one more stripe or chunk than the row has, give up after
 *   `polls` polls and record SMX_ERR_TIMEOUT (the output is then undefined) --
 *   a deterministic probe of that error path; 0 = off.
 */
void smx_debug_force_path(int path);
void smx_debug_set_cluster(int max_cluster, int64_t smem_bytes);
void smx_debug_set_wait_limit(int64_t polls);
int smx_debug_last_path(void);
int smx_debug_last_launches(void);
void smx_debug_set_regs_shape(int threads, int vpt);
void smx_debug_set_stream_depth(int depth);
void smx_debug_set_stream_ctas(int per_sm);
void smx_debug_set_cluster_staging(int mode);
void smx_debug_set_split_slab(int64_t bytes);
void smx_debug_set_split_hints(int stats, int apply);
void smx_debug_set_stream_warp(int off);
void smx_debug_set_split_fused(int on);
void smx_debug_set_attention_kernel(int which);
void smx_debug_set_host_chunk(int64_t bytes, int slots, int staged);
void smx_debug_set_inflight(int64_t read_only_bytes, int64_t backward_bytes);
int64_t smx_debug_alloc_count(void);
void smx_debug_set_count_probe(int64_t polls);
void smx_debug_set_stripe_tuning(int lag, int piece_bytes, int l2_ahead);
smx_status smx_debug_probe_math(const float *a, const float *b, float *out, int64_t n, int which,
                                smx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SMX_H */
