/*
 * ctr.h -- C-ABI of libctr, the GB300 (sm_103a) CTR sparse-embedding path.
 *
 * The path: batch ID dedup -> pooled embedding-bag gather -> pairwise dot
 * interaction -> interaction backward -> per-unique-row gradient reduce and
 * SGD row update.  Every step runs in this library's CUDA kernels.
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.   Every pointer is DEVICE memory owned by the caller unless its
 *           comment says "host".  The library never allocates: scratch space
 *           comes from the caller's workspace `ws` (size from the matching
 *           *_workspace_size call, 256-byte aligned).
 * Streams.  Calls enqueue work on `stream` (a cudaStream_t; NULL = the legacy
 *           default stream) and return without synchronising, except
 *           ctr_check_status.
 * Errors.   Host-side validation returns a negative ctr_status before any
 *           launch.  Conditions only the device can see (an ID outside its
 *           table, offsets that are not monotone) set a sticky error word in the
 *           first 256 bytes of `ws`; ctr_check_status reports and clears it.
 *           The kernels never trap: a bad ID is skipped (treated as a zero
 *           row) and flagged.  A CUDA launch error maps to CTR_ERR_CUDA.
 * Bags.     Bags are CSR and field-major: bag (f, b) holds
 *           indices[offsets[f*B + b] .. offsets[f*B + b + 1]), f < num_fields,
 *           b < batch.  Each occurrence counts (a count matrix, not a 0/1 one).
 * Tables.   Several tables live in one buffer [total_rows, d]; table t owns
 *           global rows row_base[t] .. row_base[t+1]-1, and field f reads table
 *           bag_to_table[f].  Rows are contiguous, d elements each.
 * Determinism.  For a given input every output is bit-identical run to run:
 *           no float atomics, fixed reduction orders.
 */
#ifndef CTR_H
#define CTR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ctr_stream_t; /* identical to cudaStream_t */

typedef enum {
  CTR_OK = 0,
  CTR_ERR_INVALID_ARG = -1,        /* null pointer, bad size, bad enum */
  CTR_ERR_UNSUPPORTED = -2,        /* valid but outside what the kernels cover */
  CTR_ERR_WORKSPACE = -3,          /* ws missing, misaligned or too small */
  CTR_ERR_INDEX_OUT_OF_RANGE = -4, /* device: an ID outside its table */
  CTR_ERR_CUDA = -5,               /* a CUDA runtime call or launch failed */
  CTR_ERR_TIMEOUT = -6,            /* device: a bounded wait ran out */
  CTR_ERR_NOT_IMPLEMENTED = -7,
  CTR_ERR_BAD_OFFSETS = -8         /* device: offsets not monotone or not ending at n_ids */
} ctr_status;

typedef enum { CTR_F32 = 0, CTR_BF16 = 1 } ctr_dtype;
typedef enum { CTR_POOL_SUM = 0, CTR_POOL_MEAN = 1 } ctr_pool;

/* Limits of the host-side per-field and per-table arrays. */
#define CTR_MAX_FIELDS 512
#define CTR_MAX_TABLES 512

/* Human-readable name of a ctr_status value (static string). */
const char* ctr_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int ctr_version(void);

/* Zero the sticky error word at the head of `ws` (async on `stream`).
 * Call once on a fresh workspace before its first use. */
int ctr_status_reset(void* ws, ctr_stream_t stream);

/* Synchronise `stream`, read the sticky error word of `ws`, clear it, and
 * return CTR_OK or the first device-side error recorded since the last reset. */
int ctr_check_status(void* ws, ctr_stream_t stream);

/* Per-kernel timing hook (diagnostics).  After this call, every launch of the
 * named kernel records `before_event` on the launching stream just before the
 * launch and `after_event` just after it (cudaEvent_t handles owned by the
 * caller; both NULL turns the hook off).  Kernels:
 *   CTR_KERNEL_GATHER            the pooled-gather kernel of ctr_embedding_bag_fwd
 *   CTR_KERNEL_BWD_TILES         the short-run tile kernel of ctr_embedding_bag_bwd_update
 *   CTR_KERNEL_BWD_PIECES        its long-run piece kernel
 *   CTR_KERNEL_SORT              all radix passes of ctr_dedup (first to last)
 *   CTR_KERNEL_INTERACTION       the kernel of ctr_dot_interaction
 *   CTR_KERNEL_INTERACTION_BWD   the kernel of ctr_dot_interaction_bwd
 *   CTR_KERNEL_GATHER_ROWS       the kernel of ctr_gather_rows
 * The setting is process-wide and not synchronised with calls running on
 * other host threads. */
typedef enum {
  CTR_KERNEL_GATHER = 1,
  CTR_KERNEL_BWD_TILES = 2,
  CTR_KERNEL_BWD_PIECES = 3,
  CTR_KERNEL_SORT = 4,
  CTR_KERNEL_INTERACTION = 5,
  CTR_KERNEL_INTERACTION_BWD = 6,
  CTR_KERNEL_GATHER_ROWS = 7
} ctr_kernel;
#define CTR_KERNEL_COUNT 8
int ctr_set_timing_events(int kernel, void* before_event, void* after_event);

/* Number of kernel launches this library has issued in this process, on all
 * devices and streams, since it was loaded (diagnostics: the difference across
 * a region counts the library's launches in it).  Host-side atomic counter;
 * never fails. */
uint64_t ctr_launch_count(void);

/* Gather variant of ctr_embedding_bag_fwd for fp32 tables with d = 128 and no
 * FM output: on != 0 selects the TMA row gather (cp.async.bulk.tensor with
 * tile::gather4 into a shared-memory ring), 0 (the default) the register-window
 * gather, which measured faster on GB300.  Both sum each bag in index order.
 * Process-wide; returns the previous setting. */
int ctr_set_tma_gather(int on);

/* Diagnostics: the wall-clock limit (nanoseconds, default 1e9) of each wait of
 * a ctr_dedup radix pass on a predecessor tile's counts.  A wait that runs out
 * records CTR_ERR_TIMEOUT in the workspace (read by ctr_check_status), the
 * pass keeps every write inside its buffers, and the call's outputs are then
 * meaningless.  A short limit makes ordinary waits run out: it exists to test
 * that path.  Process-wide, read at each launch; returns the previous limit. */
uint64_t ctr_set_wait_limit_ns(uint64_t ns);

/* Short-run pass of the row update for fp32 rows under plain SGD (no
 * optimizer state, no stochastic rounding) of d = 128, or of d <= 64 with d a
 * multiple of 4: mode 2 processes the short runs in slices of at most 64
 * columns (two for d = 128, one for d <= 64), two occurrences per warp step,
 * so the pooled-gradient rows of one table take half the L2 space at d = 128
 * and narrow rows keep twice the lanes busy; mode 1 never does; 0 (the
 * default) does for d <= 64 always, and for d = 128 when one table's
 * pooled-gradient rows (batch x 512 bytes) exceed 32 MB.  Every mode gives a
 * deterministic result within the same summation bound (each run's sum order
 * is fixed; the sliced pass adds the run's even and odd positions separately,
 * then the two partials).  Process-wide; returns the previous mode (a mode
 * outside 0..2 selects 0). */
int ctr_set_tile_slices(int mode);

/* ------------------------------------------------------------------------ */
/* Input generation (not part of the method)                                 */
/* ------------------------------------------------------------------------ */
/* Fill rows [row0, row0 + rows) of a table buffer with the counter-based
 * generator.  `table` points at global row row0; element (r, c) gets the value
 * of global element index (row0 + r) * d + c:
 *   gen_kind 0 (uniform, fp32 tables): h = splitmix64(seed ^ idx);
 *       v = (float)((int)(h >> 40) - 2^23) * scale
 *   gen_kind 1 (normal4, bf16 tables): Irwin-Hall sum of four 22-bit fields of
 *       splitmix64(seed ^ 2 idx) and splitmix64(seed ^ (2 idx + 1)), minus
 *       2^23 - 2, times scale, rounded to bf16 (nearest even).
 * splitmix64 is the output function of Steele, Lea and Flood (OOPSLA 2014). */
int ctr_fill_table(void* table, ctr_dtype dtype, int64_t rows, int32_t d, int64_t row0, int gen_kind,
                   uint64_t seed, float scale, ctr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a1. Dedup: the virtual sparse feature                                     */
/* ------------------------------------------------------------------------ */
/* Source: "How TensorNet Supercharges Sparse Feature Training on TensorFlow",
 * Core Optimizations, embedding_lookup: collect the batch's IDs, sort them and
 * assign each distinct ID a continuous index; the batch-sized embedding matrix
 * has one row per distinct ID (its capacity is the batch's ID count).
 *
 * Keys are global rows k_i = row_base[bag_to_table[f]] + ids[i] (so equal IDs
 * of different tables stay apart, and per-table dedup falls out of one sort).
 * Requires total_rows = row_base[num_tables] <= 2^32 and n_ids < 2^31.
 *
 * Inputs
 *   ids            int64 [n_ids]        table-local IDs, field-major CSR
 *   offsets        int64 [F*B + 1]      offsets[0] = 0, offsets[F*B] = n_ids
 *   bag_to_table   host int32 [F]       table of each field
 *   row_base       host int64 [T + 1]   first global row of each table
 *   n_ids          host                 number of IDs (the caller sizes buffers by it)
 * Outputs (capacity n_ids each; a NULL int32 output is skipped)
 *   unique_rows    int64 [n_ids]        distinct keys, ascending; first n_unique valid
 *   n_unique       int64 [1]            number of distinct keys (device scalar)
 *   inverse        int32 [n_ids]        rank of key i in unique_rows (the virtual sparse feature)
 *   sorted_pos     int32 [n_ids]        stable sort permutation: position of the s-th key
 *   sorted_bag     int32 [n_ids]        bag (f*B + b) of sorted_pos[s]
 *   run_offsets    int32 [n_ids + 1]    run of unique u is sorted slots run_offsets[u] ..
 *                                       run_offsets[u+1]-1; run_offsets[n_unique] = n_ids
 *   unique_offsets int64 [T + 1]        uniques of table t are unique_rows[unique_offsets[t] ..
 *                                       unique_offsets[t+1]); unique_offsets[T] = n_unique
 * sorted_pos is the costliest output: when it is NULL (and total_rows <= 64 *
 * n_ids, when the ranks come from a presence bitmap over the table rows) the
 * sort carries bags instead of positions and writes sorted_bag directly.
 * Device errors: CTR_ERR_INDEX_OUT_OF_RANGE (an ID outside its table; its key
 * is then replaced by the last row of its table), CTR_ERR_BAD_OFFSETS,
 * CTR_ERR_TIMEOUT (a radix pass waited over 1 s on an earlier tile).
 * Workspace: ctr_dedup_workspace_size(n_ids, F, B, total_rows) bytes; it
 * grows with total_rows / 8 on the bitmap path. */
size_t ctr_dedup_workspace_size(int64_t n_ids, int32_t num_fields, int32_t batch, int64_t total_rows);
int ctr_dedup(const int64_t* ids, const int64_t* offsets, int32_t num_fields, int32_t batch,
              const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables, int64_t n_ids,
              int64_t* unique_rows, int64_t* n_unique, int32_t* inverse, int32_t* sorted_pos, int32_t* sorted_bag,
              int32_t* run_offsets, int64_t* unique_offsets, void* ws, size_t ws_bytes, ctr_stream_t stream);

/* The same dedup in two parts, so a caller can schedule the other work of a
 * step between them.  CTR_DEDUP_PREPARE launches everything before the radix
 * passes (the keys, and on the presence-bitmap path the bitmap, unique_rows,
 * n_unique, unique_offsets and inverse); CTR_DEDUP_SORT launches the radix
 * passes and what follows them (sorted_pos, sorted_bag, run_offsets, and on
 * the path that sorts the rows themselves the unique outputs too).
 * CTR_DEDUP_ALL = both = ctr_dedup.  A SORT call must follow the PREPARE call
 * in stream order (or behind an event), with the same arguments and the same
 * workspace, which carries the state between them; outputs a part does not
 * write are undefined until the other part has run.  Errors as ctr_dedup;
 * CTR_ERR_INVALID_ARG for a phase mask outside 1..3. */
#define CTR_DEDUP_PREPARE 1
#define CTR_DEDUP_SORT 2
#define CTR_DEDUP_ALL 3
int ctr_dedup_phases(const int64_t* ids, const int64_t* offsets, int32_t num_fields, int32_t batch,
                     const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables, int64_t n_ids,
                     int64_t* unique_rows, int64_t* n_unique, int32_t* inverse, int32_t* sorted_pos,
                     int32_t* sorted_bag, int32_t* run_offsets, int64_t* unique_offsets, int32_t phases, void* ws,
                     size_t ws_bytes, ctr_stream_t stream);

/* TensorNet's batch-sized matrix (same passage): U[u] = table[unique_rows[u]]
 * for u < *n_unique.  capacity (host) bounds n_unique; rows of U at or beyond
 * n_unique are left untouched.  U is [capacity, d] of the table's dtype. */
int ctr_gather_rows(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows, const int64_t* unique_rows,
                    const int64_t* n_unique, int64_t capacity, void* U, void* ws, size_t ws_bytes,
                    ctr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a2. Pooled embedding-bag forward                                          */
/* ------------------------------------------------------------------------ */
/* Source: "DHEN" notes, section 2.1 (each categorical term has a trainable
 * d-vector) and section 3.1, Solution 2 (sum the active embeddings); "Meta
 * DLRM", section 02 (categorical features go through embeddings).
 *
 *   out(b, f) = sum_{i in bag(f,b)} table[row_i]          (CTR_POOL_SUM)
 *             = that sum / len(bag)   (0 for an empty bag)  (CTR_POOL_MEAN)
 * accumulated in fp32, rounded once to out_dtype.
 * Row selection: if bag_to_table != NULL, indices are table-local int64 IDs and
 * row_i = row_base[bag_to_table[f]] + ids[i] (host arrays as in ctr_dedup);
 * if bag_to_table == NULL, indices are rows of `table` directly (e.g. the
 * int32 inverse map into the unique-row matrix U), num_tables ignored.
 * indices_are_int32 selects int32 or int64 indices; n_indices (host) is the
 * length of `indices` (a bag reaching past it is skipped and flagged).
 * out(b, f) is the d-vector at out + b*out_stride_b + f*out_stride_f
 * (element strides; e.g. the pooled slots of an interaction input [B, F+1, d]
 * are out = X + d, out_stride_b = (F+1)*d, out_stride_f = d).
 * table dtype CTR_F32 or CTR_BF16; out_dtype CTR_F32, or CTR_BF16 (bf16 tables).
 * Device errors: CTR_ERR_INDEX_OUT_OF_RANGE (row skipped), CTR_ERR_BAD_OFFSETS
 * (bag skipped, written as zeros).
 * Workspace: ctr_embedding_bag_workspace_size() bytes (the error word). */
size_t ctr_embedding_bag_workspace_size(void);
int ctr_embedding_bag_fwd(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows, const void* indices,
                          int indices_are_int32, int64_t n_indices, const int64_t* offsets, int32_t num_fields, int32_t batch,
                          const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables, ctr_pool pool,
                          void* out, ctr_dtype out_dtype, int64_t out_stride_b, int64_t out_stride_f, void* ws,
                          size_t ws_bytes, ctr_stream_t stream);

/* The same pooled gather, also writing the factorization-machine second-order
 * term of each bag ("DHEN" notes, section 3.1, Solution 2: the sum over pairs
 * of active features of <v_i, v_j> equals 1/2 (|sum v|^2 - sum |v|^2), one
 * pass over the rows):
 *   fm_out[f*B + b] = 1/2 ( |sum_{i in bag} row_i|^2 - sum_{i in bag} |row_i|^2 )
 * over the bag's occurrences (a repeated ID is a repeated feature), from the
 * raw sum whatever the pooling mode; 0 for bags with fewer than two IDs.
 * fp32 accumulation and arithmetic (the difference of the two terms loses
 * relative accuracy when they nearly cancel, as the identity's own form does).
 * fm_out: fp32 [F*B] device, required.  Supported for rows that are a whole
 * number of 16-byte chunks; CTR_ERR_UNSUPPORTED otherwise. */
int ctr_embedding_bag_fwd_fm(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows, const void* indices,
                             int indices_are_int32, int64_t n_indices, const int64_t* offsets, int32_t num_fields,
                             int32_t batch, const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables,
                             ctr_pool pool, void* out, ctr_dtype out_dtype, int64_t out_stride_b,
                             int64_t out_stride_f, float* fm_out, void* ws, size_t ws_bytes, ctr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a3. Pairwise dot interaction                                              */
/* Workspace of both interaction calls: ctr_interaction_workspace_size()     */
/* bytes (the error word; the tensor-core kernel records CTR_ERR_TIMEOUT    */
/* there if one of its bounded waits runs out).                              */
/* ------------------------------------------------------------------------ */
/* Source: "Meta DLRM", section 02 (the interaction is the dot product between
 * every pair of embedding vectors and the processed dense features, cross terms
 * only); "DHEN" notes, section 3.1, Eq. (3) (pairwise inner products
 * concatenated with the dense features).
 *
 * X [batch, n, d], slot 0 = the dense vector, slots 1..n-1 = pooled embeddings.
 *   out[b] = [ X[b,0,:] | Z ],  Z[i(i-1)/2 + j] = <X[b,i,:], X[b,j,:]>,
 *            1 <= i < n, 0 <= j < i   (strict lower triangle, row by row)
 * out is [batch, d + n(n-1)/2] of the input dtype.  fp32: CUDA-core FMA.
 * bf16: tcgen05 tensor cores (fp32 accumulate in TMEM, bf16 output) when
 * n <= 32 and d is a multiple of 64 up to 256; other shapes use a CUDA-core
 * kernel with fp32 accumulation.  The fast kernels need X and out 16-byte
 * aligned; other pointers take the generic kernel. */
size_t ctr_interaction_workspace_size(void);
int ctr_dot_interaction(const void* X, ctr_dtype dtype, int32_t batch, int32_t n, int32_t d, void* out, void* ws,
                        size_t ws_bytes, ctr_stream_t stream);

/* Derivative of ctr_dot_interaction (fp32), not on the pages:
 *   dX[b,i,:] = sum_{j != i} dZ(i,j) X[b,j,:]  (+ dout[b, 0:d] for i = 0)
 * with dZ(i,j) = dout[b, d + hi(hi-1)/2 + lo], hi = max(i,j), lo = min(i,j).
 * dout [batch, d + n(n-1)/2], X and dX [batch, n, d]. */
int ctr_dot_interaction_bwd(const float* dout, const float* X, int32_t batch, int32_t n, int32_t d, float* dX,
                            void* ws, size_t ws_bytes, ctr_stream_t stream);

/* Interaction variants.  CTR_INTERACT_CROSS is ctr_dot_interaction above.
 * CTR_INTERACT_WITH_SELF keeps the diagonal too ("DHEN" notes, section 3.1:
 * the AdvancedDLRM module takes all inner products <x_i, x_j> for i <= j):
 *   out[b] = [ X[b,0,:] | Z ],  Z[i(i+1)/2 + j] = <X[b,i,:], X[b,j,:]>, 0 <= j <= i < n
 * CTR_INTERACT_FULL_GRAM emits the whole Gram matrix ("DHEN" notes, section
 * 3.3, Eq. (7): the cross network's input X X^T), no dense vector:
 *   out[b] = Z,  Z[i n + j] = <X[b,i,:], X[b,j,:]>,  0 <= i, j < n
 * The order of the products and the leading dense vector are layout choices.
 * ctr_interaction_width(n, d, mode) is the output row length (-1 for bad
 * arguments).  The kernels, dtypes and alignment rules are those of
 * ctr_dot_interaction.  The derivative (fp32) is, with G the upstream gradient
 * of the emitted products (0 for products the mode omits) and S = G + G^T:
 *   dX[b,i,:] = sum_j S[i][j] X[b,j,:]  (+ dout[b, 0:d] for i = 0, first two modes). */
typedef enum { CTR_INTERACT_CROSS = 0, CTR_INTERACT_WITH_SELF = 1, CTR_INTERACT_FULL_GRAM = 2 } ctr_interaction_mode;
int64_t ctr_interaction_width(int32_t n, int32_t d, int mode);
int ctr_dot_interaction_mode(const void* X, ctr_dtype dtype, int32_t batch, int32_t n, int32_t d, int mode, void* out,
                             void* ws, size_t ws_bytes, ctr_stream_t stream);
int ctr_dot_interaction_bwd_mode(const float* dout, const float* X, int32_t batch, int32_t n, int32_t d, int mode,
                                 float* dX, void* ws, size_t ws_bytes, ctr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a5. Sparse backward: per-unique-row gradient reduce + SGD row update       */
/* ------------------------------------------------------------------------ */
/* Source: "How TensorNet ...", Synchronous Architecture (only the sparse
 * features present in the batch are synchronised) and Core Optimizations (the
 * batch-sized matrix of unique rows).  The SGD rule is not on the pages.
 *
 * For each unique u < *n_unique, over its run of sorted occurrences s (from
 * ctr_dedup):
 *   g_u = sum_s scale(bag_s) * grad_pooled(bag_s),  scale = 1 (SUM) or
 *         1 / len(bag) (MEAN),   bag_s = sorted_bag[s] = f*B + b,
 *         grad_pooled(bag) = the fp32 d-vector at grad_pooled + b*g_stride_b + f*g_stride_f
 *   table[unique_rows[u]] <- table[unique_rows[u]] - lr * g_u
 * Each row is written exactly once; no float atomics.  The sum runs in a fixed
 * order (pieces of at most 128 occurrences summed in sorted order, then a fixed
 * tree over the pieces of a long run), so results are deterministic.
 * fp32 tables: one fused multiply-add, rounded once.  bf16 tables: the update
 * is computed in fp32 and rounded to bf16 (nearest even).
 * grad_unique_out (optional, [n_ids, d] fp32): receives g_u in row u.
 * n_ids (host) is the capacity used to size grids; *n_unique <= n_ids.
 * Workspace: ctr_bwd_update_workspace_size(n_ids, d) bytes. */
size_t ctr_bwd_update_workspace_size(int64_t n_ids, int32_t d);
int ctr_embedding_bag_bwd_update(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                 const int64_t* offsets, int32_t num_fields, int32_t batch, ctr_pool pool,
                                 const int64_t* unique_rows, const int64_t* n_unique, const int32_t* run_offsets,
                                 const int32_t* sorted_bag, int64_t n_ids, float lr, void* table, ctr_dtype dtype,
                                 int32_t d, int64_t total_rows, float* grad_unique_out, void* ws, size_t ws_bytes,
                                 ctr_stream_t stream);

/* The same update in phases, for callers that overlap them on two streams.
 *   CTR_BWD_SHORT_RUNS  runs of at most 128 occurrences: summed and their rows
 *                       updated
 *   CTR_BWD_LONG_RUNS   every longer run: listed, cut into pieces of 128 and
 *                       each piece summed into the workspace
 *   CTR_BWD_FINISH      the long runs' pieces combined and their rows updated
 * ctr_embedding_bag_bwd_update runs all three in this order (short runs first:
 * the long runs then find many pooled-gradient rows still in L2).  LONG_RUNS and
 * SHORT_RUNS touch disjoint rows and disjoint workspace words, so they may run
 * concurrently on two streams with the same arguments and workspace; FINISH
 * must be ordered after LONG_RUNS (and both after the dedup that produced the
 * runs).  `phases` is a non-empty mask of the three; the phases it names run
 * in the order above on `stream`. */
typedef enum { CTR_BWD_SHORT_RUNS = 2, CTR_BWD_LONG_RUNS = 1, CTR_BWD_FINISH = 4 } ctr_bwd_phase;
int ctr_embedding_bag_bwd_update_phases(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                        const int64_t* offsets, int32_t num_fields, int32_t batch, ctr_pool pool,
                                        const int64_t* unique_rows, const int64_t* n_unique,
                                        const int32_t* run_offsets, const int32_t* sorted_bag, int64_t n_ids, float lr,
                                        void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                                        float* grad_unique_out, int phases, void* ws, size_t ws_bytes,
                                        ctr_stream_t stream);

/* The same update under an optimizer with per-row state, kept only for the
 * rows the batch touches (the pages name no update rule; these are readings):
 *   CTR_OPT_SGD               w -= lr g                                   (no state)
 *   CTR_OPT_ADAGRAD           s += g^2;  w -= lr g / (sqrt(s) + eps)      state0 [total_rows, d]
 *   CTR_OPT_ROWWISE_ADAGRAD   s += mean over the row of g^2;
 *                             w -= lr g / (sqrt(s) + eps)                state0 [total_rows]
 *   CTR_OPT_ADAM              m = b1 m + (1 - b1) g;  v = b2 v + (1 - b2) g^2;
 *                             w -= lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 *                             (Kingma and Ba 2015)          state0 = m, state1 = v [total_rows, d]
 * g is the row's reduced gradient (as in ctr_embedding_bag_bwd_update); state
 * arrays are fp32 device memory owned by the caller, indexed by global row,
 * 16-byte aligned, and only the batch's rows are read and written.  t = step
 * (>= 1) is this update's step number for Adam's bias correction; eps > 0.
 * phases as in ctr_embedding_bag_bwd_update_phases.  The optimizer
 * arithmetic is fp32.
 *
 * Stochastic rounding ("DHEN" notes, section 6.4: low-precision embeddings
 * with stochastic rounding; applied here to bf16 tables, with any kind): the
 * new value x (fp32) of element (row, c) becomes the bf16 neighbour above it
 * in magnitude with probability f = (|x| - lo) / (hi - lo), lo and hi its bf16
 * neighbours, else lo: with u the element's 16 random bits, x rounds up when
 * f + u / 2^16 >= 1, i.e. u is added to the 16 bits bf16 drops and the carry
 * kept.  The 4 values of column chunk q = c / 4 take bits 16 (c mod 4) ..
 * 16 (c mod 4) + 15 of splitmix64(sr_seed ^ (row d / 4 + q)).  Values at or
 * beyond the largest finite bf16 round to nearest.  fp32 tables ignore it. */
typedef enum { CTR_OPT_SGD = 0, CTR_OPT_ADAGRAD = 1, CTR_OPT_ROWWISE_ADAGRAD = 2, CTR_OPT_ADAM = 3 } ctr_opt_kind;
typedef struct {
  int kind;       /* ctr_opt_kind */
  float eps;
  float beta1;    /* Adam */
  float beta2;    /* Adam */
  int64_t step;   /* Adam: t >= 1 */
  float* state0;  /* Adagrad sum of squares, or Adam m */
  float* state1;  /* Adam v */
  int32_t stochastic_rounding;  /* bf16 tables: round the new rows stochastically (below) */
  uint64_t sr_seed;             /* its random bits; use a new seed every step */
} ctr_optimizer;
int ctr_embedding_bag_bwd_update_opt(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                     const int64_t* offsets, int32_t num_fields, int32_t batch, ctr_pool pool,
                                     const int64_t* unique_rows, const int64_t* n_unique, const int32_t* run_offsets,
                                     const int32_t* sorted_bag, int64_t n_ids, float lr, void* table, ctr_dtype dtype,
                                     int32_t d, int64_t total_rows, float* grad_unique_out, int phases,
                                     const ctr_optimizer* opt, void* ws, size_t ws_bytes, ctr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Allocation-free dedup (no counterpart in the paper)                       */
/* ------------------------------------------------------------------------ */
/* ctr_dedup for callers that may not allocate device memory on this path: a
 * plugin inside a runtime that owns every device allocation, a server whose
 * memory budget is fixed at start-up, or a latency-critical loop where an
 * allocation could stall the device.  Same inputs and outputs as ctr_dedup,
 * but the scratch space is a fixed array inside the library (48 MB per GPU
 * that loads the library, held until exit) instead of a caller workspace.
 *   n_ids            at most 1048576 (2^20), for any total row count (the
 *                    array covers the largest scratch ctr_dedup_workspace_size
 *                    gives at 2^20 IDs, 46 MB at total rows = 64 x 2^20);
 *                    larger calls return CTR_ERR_UNSUPPORTED and launch
 *                    nothing.
 *   device_status    optional device int32: receives this call's device-side
 *                    error code (0, CTR_ERR_INDEX_OUT_OF_RANGE or
 *                    CTR_ERR_BAD_OFFSETS) once the call's work has run.
 * All calls share the array and it keeps the previous call's contents; its
 * error word is cleared at the start of every call.  Calls that overlap on
 * the GPU race on the array: order them (one stream, or explicit events).
 * The first call on a device looks up the array's address with that device
 * current and caches it; make that first call before any stream capture, and
 * do not call this entry point on a device again after cudaDeviceReset in the
 * same process (the cached address belongs to the old context).
 * Nothing here calls cudaMalloc, cudaFree or any other allocator. */
int ctr_dedup_static(const int64_t* ids, const int64_t* offsets, int32_t num_fields, int32_t batch,
                     const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables, int64_t n_ids,
                     int64_t* unique_rows, int64_t* n_unique, int32_t* inverse, int32_t* sorted_pos,
                     int32_t* sorted_bag, int32_t* run_offsets, int64_t* unique_offsets, int32_t* device_status,
                     ctr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CTR_H */
