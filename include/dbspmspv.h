/*
 * dbspmspv.h -- C ABI of a GB300 (sm_103a) implementation of DB-SpMSpV:
 * dual-view blocked sparse-matrix x sparse-vector multiplication y = A x for
 * a reusable matrix A and an input vector x that changes on every call.
 *
 * Method: Cong et al., "DB-SpMSpV: Dual-View Blocked Sparse Matrix-Sparse
 * Vector Multiplication for Dynamic GPU Workloads", ICPP '26.
 *   - build once, call many times with a changing x (Sections 1 and 4.3;
 *     "the DB-format conversion is performed offline and reused", Section 5.5);
 *   - 16x16 blocks, block-CSR and block-CSC views over one payload (3.2.1);
 *   - vector-block masks and nonzero-block statistics built on the GPU (4.1);
 *   - push/pull selection by nonzero-vector-block ratio, th3 = 0.01 (3.3.1);
 *   - per-block microkernels chosen from block type and blk_x_mask (3.3.1,
 *     3.3.3, Algorithms 2-4);
 *   - load-weighted pull tiles and flattened push tasks (3.3.2);
 *   - Boolean or/and semiring with a visited mask and DB-BFS (4.2, Alg. 5).
 *
 * Conventions (apply to every function below):
 *   - Every function returns a dbs_status; nothing aborts, throws or traps.
 *   - "stream" is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls marked ASYNC only enqueue work on that stream and return;
 *     their device outputs are valid once the stream reaches that point.
 *     Device-side failures of an ASYNC call (a bounded wait that timed out)
 *     are latched in the workspace and reported by dbs_workspace_check().
 *   - "device" pointers are CUDA global-memory pointers on the current device;
 *     "host" pointers are ordinary CPU memory.  The caller owns every input
 *     and output buffer; the library owns the matrix and the workspace.
 *   - A(i, j) stored means x_j contributes to y_i; push walks column j.
 *   - x_j is active iff it is listed and its value is != 0 (so -0.0 is
 *     inactive and NaN is active); with no values every listed index is
 *     active.  Listed indices must be unique and in [0, n).
 *   - Output pattern is structural: y_i is produced iff some stored A(i, j)
 *     has an active x_j, even when the values cancel to zero.
 *   - Limits: m, n < 2^31; nonzero 16x16 blocks < 2^32; payload < 64 GiB.
 */
#ifndef DBSPMSPV_H
#define DBSPMSPV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DBS_OK = 0,
    DBS_ERR_INVALID_ARG = 1,   /* bad pointer, size, index, duplicate or option */
    DBS_ERR_OOM = 2,           /* host or device allocation failed (nothing leaked) */
    DBS_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    DBS_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up */
    DBS_ERR_UNSUPPORTED = 5,   /* valid request this build does not serve */
    DBS_ERR_INTERNAL = 6       /* a device-side capacity or consistency check failed */
} dbs_status;

typedef enum {
    DBS_PLUS_TIMES_F32 = 0,    /* y_i = sum_j A(i,j) * x_j in fp32 */
    DBS_OR_AND_BOOL = 1        /* y_i = OR_j (A(i,j) and x_j active) and not visited_i */
} dbs_semiring;

typedef enum {
    DBS_PATH_AUTO = 0,         /* device-side choice (Section 3.3.1; see dbs_exec_opts) */
    DBS_PATH_PUSH = 1,         /* column-driven over the block-CSC view */
    DBS_PATH_PULL = 2,         /* row-driven over the block-CSR view */
    DBS_PATH_SPMV = 3          /* dbs_spmspv_dense only, on a matrix built with dense_spmv:
                                  the kept adaptive CSR SpMV (the paper's Limitations) */
} dbs_path;

/* Low-level block formats (Section 3.2.1, Figure 5(b), Figure 6). */
typedef enum {
    DBS_FMT_COO = 0,           /* packed 4+4-bit coordinates + values (nnz < th0) */
    DBS_FMT_DENSE = 1,         /* 256 values + column masks (nnz > th1) */
    DBS_FMT_FORCE_CSR = 2,     /* row_ptr + row_mask + values in row order */
    DBS_FMT_FORCE_CSC = 3,     /* col_ptr + col_mask + values in column order */
    DBS_FMT_PATCHED_CSR = 4    /* ForceCSR + col_ptr + row_idx_csc2csr bytes */
} dbs_format;
#define DBS_FMT_AUTO (-1)
#define DBS_NUM_FORMATS 5

/* Build options.  dbs_build_opts_default() fills the paper's settings. */
typedef struct {
    int32_t th0;               /* nnz < th0 -> COO (paper: 32) */
    int32_t th1;               /* nnz > th1 -> Dense (paper: 128) */
    double th2;                /* skew ratio above which a block is ForceCSR/ForceCSC (paper: 2.0) */
    int32_t force_format;      /* DBS_FMT_AUTO, or one dbs_format for every block (ablation) */
    int32_t tile_weight;       /* pull tile weight cap; block weights Dense 4, ForceCSR /
                                  ForceCSC / patched CSR 2, COO 1 (Section 3.3.2).  A tile
                                  is one warp's task and holds at most 256 blocks.
                                  0 = sized from the matrix and the GPU's SM count. */
    int32_t tile_max_row_blocks; /* row blocks one pull tile may span (1..32); 1 with
                                  tile_weight 16 reproduces the paper's segments. 0 = 32 */
    int32_t keep_host;         /* keep a host copy of the blocked format (export) */
    int32_t host_only;         /* build the format on the host only; no device memory
                                  is touched (the matrix can be inspected and exported
                                  but not multiplied).  For CPU-side checks. */
    int32_t num_threads;       /* host builder threads; 0 = all hardware threads */
    int32_t device_convert;    /* 1 with inputs_on_device: the whole conversion runs on
                                  the GPU (validation, blocks, formats, payload, offsets,
                                  block-CSC view, tiles); nothing proportional to the
                                  matrix crosses to the host.  Device memory beyond the
                                  input and the result: 4 B per block + 12 B per column
                                  block, or 12 B per row block + 8 B per 4,096 entries
                                  if more (see build_peak_bytes).  Needs the columns of
                                  every row ascending, else the host converts.  Same
                                  result byte for byte.  Default 0. */
    int32_t dense_spmv;        /* 1 with a valued matrix: also keep a device copy of the
                                  input CSR (8 B per entry and per row) and an adaptive
                                  CSR SpMV plan over it; dbs_spmspv_dense then hands an x
                                  whose sampled nonzero fraction reaches
                                  dbs_exec_opts.spmv_x_frac to that SpMV, which runs
                                  first and makes the blocked kernel return at once (the
                                  paper's Limitations: conventional SpMV is preferable
                                  for dense inputs).  Default 0. */
} dbs_build_opts;

void dbs_build_opts_default(dbs_build_opts *opts);

/* Execution options of a workspace.  dbs_exec_opts_default() fills them. */
typedef struct {
    double th3;                /* push iff N_nzblk < th3 * N_blk (paper: 0.01); used when
                                  push_work_frac is 0 */
    int32_t local_pull_min;    /* patched-CSR blocks use the row-wise (pull) microkernel
                                  when popc(active block columns) >= this; else the
                                  column-wise (push) one.  Unstated in the paper; default
                                  0 (always row-wise: measured faster on GB300). */
    int32_t collect_stats;     /* 1: count visited / hit blocks, touched nnz and
                                  algorithmic bytes on the device (a few atomics per CTA) */
    int64_t wait_timeout_ns;   /* bound on every device-side wait (grid barriers);
                                  default 2 s.  On expiry the kernel latches
                                  DBS_ERR_TIMEOUT and returns. */
    double push_work_frac;     /* > 0: push iff the matrix blocks of the active column
                                  blocks (push's work) number fewer than push_work_frac * B
                                  (pull's scan); default 0.45, the crossover measured on
                                  GB300.  0: the paper's th3 rule. */
    double spmv_x_frac;        /* dbs_spmspv_dense, auto path, matrix with dense_spmv: the
                                  CSR SpMV runs when the nonzero fraction of a fixed
                                  sample of x (8 evenly spaced runs of 32 entries, read
                                  alike by every block) is at least this; default 0.08 */
} dbs_exec_opts;

void dbs_exec_opts_default(dbs_exec_opts *opts);

typedef struct dbs_matrix dbs_matrix;        /* opaque; library-owned device memory */
typedef struct dbs_workspace dbs_workspace;  /* opaque; per-stream scratch */

/* Section 3.2.1 (the DB format), Section 3.3.2 (pull segments), Section 5.5
 * (offline conversion).  Builds the blocked dual-view matrix from CSR.
 *   m, n        rows and columns (0 <= m, n < 2^31)
 *   nnz         number of stored entries (= row_ptr[m])
 *   row_ptr     int64[m+1], non-decreasing, row_ptr[0] = 0
 *   col_idx     int32[nnz], in [0, n), unique within a row (any order)
 *   vals        float32[nnz], or NULL for a pattern-only matrix (Boolean
 *               semiring only)
 *   inputs_on_device  0: the three arrays are host pointers; 1: device pointers
 *   opts        NULL = dbs_build_opts_default()
 *   stream      stream for the upload (the call synchronizes it before returning)
 *   out         receives the matrix; unchanged on error
 * SYNCHRONOUS.  Errors: DBS_ERR_INVALID_ARG (bad sizes, out-of-range or
 * duplicate column, non-monotone row_ptr, bad option), DBS_ERR_OOM, DBS_ERR_CUDA.
 * On error nothing is leaked. */
dbs_status dbs_matrix_build_csr(int64_t m, int64_t n, int64_t nnz, const int64_t *row_ptr,
                                const int32_t *col_idx, const float *vals, int inputs_on_device,
                                const dbs_build_opts *opts, void *stream, dbs_matrix **out);

/* Frees everything the matrix owns.  NULL is accepted.  The caller must make
 * sure no enqueued call still uses it. */
dbs_status dbs_matrix_destroy(dbs_matrix *A);

/* Section 5.5, Table 4: storage of the blocked format next to plain CSR and
 * CSR + CSC (4-byte indices; 4-byte values when valued). */
typedef struct {
    int64_t m, n, nnz;
    int64_t nbr, nbc;                       /* ceil(m/16), ceil(n/16) */
    int64_t nblocks;                        /* nonzero 16x16 blocks */
    int64_t blocks_by_format[DBS_NUM_FORMATS];
    int64_t nnz_by_format[DBS_NUM_FORMATS];
    int64_t ntiles;                         /* pull tiles */
    int64_t payload_bytes;                  /* low-level block payload */
    int64_t view_bytes;                     /* high-level views, tiles, pointers */
    int64_t total_bytes;                    /* payload + views (device footprint) */
    int64_t csr_bytes;                      /* plain CSR of the same matrix */
    int64_t csr_csc_bytes;                  /* CSR + CSC duplication */
    int32_t valued;                         /* 1 if built with values */
    int32_t on_device;                      /* 0 for host_only builds */
    double build_seconds;                   /* host time of the conversion */
    int64_t spmv_bytes;                     /* dense_spmv: the kept CSR and its SpMV plan
                                               (not in total_bytes) */
    int64_t build_peak_bytes;               /* most device memory the build held at once
                                               (library allocations only: the matrix,
                                               its SpMV plan and all scratch; not the
                                               caller's input) */
} dbs_matrix_info;

/* Fills *out.  Host-only, no synchronization. */
dbs_status dbs_matrix_info_get(const dbs_matrix *A, dbs_matrix_info *out);

/* Figure 5(b): exports the high-level views to caller-allocated HOST arrays
 * (any pointer may be NULL to skip it):
 *   blk_row_ptr int64[nbr+1], blk_col_idx int64[B]      block-CSR view
 *   blk_col_ptr int64[nbc+1], blk_row_idx int64[B]      block-CSC view
 *   blk_csc2csr int64[B]     CSC position -> primary (block-CSR) block id
 *   blk_nnz int32[B], blk_format int32[B]               per primary block
 * Uses the host copy when present, else copies from the device (synchronous). */
dbs_status dbs_matrix_export_views(const dbs_matrix *A, int64_t *blk_row_ptr, int64_t *blk_col_idx,
                                   int64_t *blk_col_ptr, int64_t *blk_row_idx,
                                   int64_t *blk_csc2csr, int32_t *blk_nnz, int32_t *blk_format);

/* Decodes the low-level payload back to CSR (HOST arrays, row_ptr int64[m+1],
 * col_idx int32[nnz], vals float32[nnz] or NULL) with columns ascending per
 * row.  A round trip returns the input bit for bit.  Synchronous. */
dbs_status dbs_matrix_export_csr(const dbs_matrix *A, int64_t *row_ptr, int32_t *col_idx,
                                 float *vals);

/* Diagnostic copy of one internal array of the matrix (the device layout of
 * the blocked format: row-block pointers u32[nbr+1], block descriptors
 * {u32, u32}[B], payload offsets u32[B], column-block pointers u32[nbc+1],
 * block-CSC descriptors {u32, u32}[B], block-CSC payload offsets u32[B],
 * payload 16-byte units [P], pull tiles {u32 x4}[T], rows holding an entry
 * u16[nbr]) into HOST memory.  *bytes gets
 * the array's size; the copy happens when dst is non-NULL and capacity is
 * large enough (else DBS_ERR_INVALID_ARG).  Synchronous. */
typedef enum {
    DBS_RAW_RB_PTR = 0, DBS_RAW_BLK_DESC, DBS_RAW_BLK_REF, DBS_RAW_CB_PTR, DBS_RAW_CSC_DESC,
    DBS_RAW_CSC_REF, DBS_RAW_PAYLOAD, DBS_RAW_TILES, DBS_RAW_RB_ROWS, DBS_RAW_COUNT
} dbs_raw_array;
dbs_status dbs_matrix_export_raw(const dbs_matrix *A, int32_t which, void *dst, int64_t capacity, int64_t *bytes);

/* Scratch for SpMSpV and BFS on one matrix: a dense copy of x, the vector-block
 * masks, active lists, push task list, the output accumulator, counters and
 * the grid-barrier state.  Calls sharing a workspace must be ordered on one
 * stream.  Every call leaves the scratch cleared for the next one. */
dbs_status dbs_workspace_create(const dbs_matrix *A, dbs_workspace **out);
dbs_status dbs_workspace_destroy(dbs_workspace *ws);
dbs_status dbs_workspace_set_opts(dbs_workspace *ws, const dbs_exec_opts *opts);

/* Synchronizes the stream, returns the status latched by the device since the
 * last check (DBS_OK, DBS_ERR_TIMEOUT or DBS_ERR_INTERNAL) and clears it, so
 * the workspace can be used again.  Calls enqueued after a latched error do
 * no work and leave their outputs untouched. */
dbs_status dbs_workspace_check(dbs_workspace *ws, void *stream);

/* Sections 3.3.1-3.3.3 and 4.1: one SpMSpV y = A x with a sparse x.  ASYNC.
 * "device" arrays below may also be pinned host memory mapped into the
 * device's address space: the kernels then read x and write y there in place
 * (on GB300, coherently over NVLink-C2C), which saves the staging copies.
 *   sr            DBS_PLUS_TIMES_F32 (matrix must be valued) or DBS_OR_AND_BOOL
 *   x_idx         device int32[x_nnz], unique indices in [0, n)
 *   x_val         device float32[x_nnz]; NULL = every listed index active
 *                 (required non-NULL for plus-times)
 *   x_nnz         host count (0 allowed)
 *   visited_mask  Boolean only: device uint16[ceil(m/16)], bit r of word b set
 *                 = row 16b+r is excluded from y (Algorithm 5); NULL = none
 *   y_idx         device int32[m] capacity: ascending output row indices
 *   y_val         device float32[m] capacity for plus-times; NULL for Boolean
 *   y_nnz         device int64[1]: number of output entries
 *   path          DBS_PATH_AUTO / _PUSH / _PULL
 * Errors returned immediately: DBS_ERR_INVALID_ARG, DBS_ERR_UNSUPPORTED
 * (plus-times on a pattern-only matrix), DBS_ERR_CUDA (launch failure).
 * An index outside [0, n) is skipped by the kernel and latched as
 * DBS_ERR_INVALID_ARG (dbs_workspace_check); the call's outputs are then
 * undefined.  With repeated indices one of their values is used. */
dbs_status dbs_spmspv(const dbs_matrix *A, dbs_semiring sr, const int32_t *x_idx,
                      const float *x_val, int64_t x_nnz, const uint16_t *visited_mask,
                      int32_t *y_idx, float *y_val, int64_t *y_nnz, dbs_path path,
                      dbs_workspace *ws, void *stream);

/* Section 4.3 (DB-Decoding): x given as a dense device float32[n] whose zero
 * entries are inactive; the vector-block masks are built from it with warp
 * ballots (Section 4.1).  y is a dense device float32[m]; rows with no active
 * contribution are written as 0.  Plus-times only.  With a matrix built with
 * dense_spmv, path DBS_PATH_SPMV (or the auto path when the sampled nonzero
 * fraction of x reaches spmv_x_frac) computes the same y by the kept CSR SpMV,
 * entries whose x is zero skipped; DBS_PATH_SPMV without it is
 * DBS_ERR_INVALID_ARG.  ASYNC. */
dbs_status dbs_spmspv_dense(const dbs_matrix *A, const float *x, float *y, dbs_path path,
                            dbs_workspace *ws, void *stream);

/* Section 4.3 (DB-Decoding: a single-token linear layer whose activations
 * are sparsified by magnitude thresholding): y = A x' with
 *     x'_j = x_j  if |x_j| > tau  (NaN entries count as active),
 *     x'_j = 0    otherwise,
 * on the pull path.  The activation mask of each 16-entry vector block is
 * formed from x inside the traversal (Section 4.1's mask generation fused
 * into the kernel that consumes it), so the call is one ordinary kernel
 * launch with no device-wide barrier, no path decision and no workspace
 * scratch: one block of threads owns each row block.  Use it when the input
 * is known to be dense enough for pull (decoding activations at about 10 %
 * density); dbs_spmspv_dense is the general form with the selector.
 *   x    device (or host-mapped) float32[n], 16-byte aligned
 *   tau  threshold, >= 0 (tau = 0: every nonzero entry is active)
 *   y    device float32[m]; every row is written (0 where nothing is active)
 * Summation order within a row is fixed by the matrix (each thread sums
 * its blocks, then a fixed tree combines the threads), so repeated calls
 * give identical bits; it is not the sequential order.  Capturable in a
 * CUDA graph.  Errors: DBS_ERR_INVALID_ARG (null pointers, tau < 0 or NaN,
 * misaligned x), DBS_ERR_UNSUPPORTED (pattern-only matrix), DBS_ERR_CUDA.
 * ASYNC. */
dbs_status dbs_decode_layer(const dbs_matrix *A, const float *x, float tau, float *y, dbs_workspace *ws,
                            void *stream);

/* Dense-input regime: adaptive CSR SpMV (the adaptive CSR SpMV execution
 * page: scalar rows, subgroup rows, workgroup rows and long-row split, one
 * mapping of work to lanes per row shape), for an x dense enough that
 * SpMSpV's vector metadata buys nothing -- the DB-SpMSpV paper's
 * Limitations note that conventional SpMV may be preferable there.
 *
 * dbs_spmv_plan_create classifies the rows of a caller-owned device CSR once,
 * on the GPU and without host readback of the row shapes: rows of up to 4,
 * 8, 16, 32, 64 and 1024 entries go to groups of 1, 2, 4, 8, 16 and 32 lanes
 * of a warp (the subgroup family, one thread for the shortest), rows of up
 * to 16384 to one 256-thread block, longer rows are split into 8192-entry
 * chunks whose partial sums the last chunk to finish adds up in chunk order.
 * The row queues hold each row's first entry and length, so the multiply
 * does not go back to row_ptr.
 *   m, n, nnz   rows, columns (< 2^31) and entries
 *   row_ptr     device int64[m+1]; col_idx device int32[nnz]; vals device
 *               float32[nnz].  Caller-owned; they must stay valid and
 *               unchanged while the plan lives.  Row pointers are clamped to
 *               [0, nnz] and column indices outside [0, n) contribute
 *               nothing, so a malformed CSR cannot cause a stray access.
 *   stream      the classification runs there; the call synchronizes it.
 * Errors: DBS_ERR_INVALID_ARG, DBS_ERR_UNSUPPORTED (nnz >= 2^32),
 * DBS_ERR_OOM, DBS_ERR_CUDA.  SYNCHRONOUS. */
typedef struct dbs_spmv_plan dbs_spmv_plan;
dbs_status dbs_spmv_plan_create(int64_t m, int64_t n, int64_t nnz, const int64_t *row_ptr, const int32_t *col_idx,
                                const float *vals, void *stream, dbs_spmv_plan **out);

/* y = A x: x device float32[n] (every entry used, zeros included), y device
 * float32[m], every row written (0 for rows without entries).  One ordinary
 * launch, deterministic summation order, capturable in a CUDA graph.  Calls
 * on one plan must be ordered on one stream (they share the split rows'
 * partial sums and counters).  ASYNC. */
dbs_status dbs_spmv(dbs_spmv_plan *plan, const float *x, float *y, void *stream);

/* Rows per bucket (HOST int64[8], may be NULL: rows on 1, 2, 4, 8, 16 and
 * 32 lanes, block rows, split rows) and split chunks (may be NULL) of a plan.
 * Synchronous. */
dbs_status dbs_spmv_plan_info(const dbs_spmv_plan *plan, int64_t *bucket_rows, int64_t *split_chunks);

/* Frees the plan's scratch (not the CSR).  NULL is accepted. */
dbs_status dbs_spmv_plan_destroy(dbs_spmv_plan *plan);

/* Section 4.2 (DB-BFS): level-synchronous BFS from src on a square matrix;
 * each level is next = (A or.and frontier) and not visited, with push/pull
 * re-chosen per level (or forced by path).  The whole level loop runs on the
 * device.  levels: device int32[n], level of each vertex or -1 if unreached.
 * nlevels_host: optional host int32*; if non-NULL the call synchronizes the
 * stream and stores the number of levels (max level + 1).  ASYNC otherwise. */
dbs_status dbs_bfs(const dbs_matrix *A, int64_t src, int32_t *levels, int32_t *nlevels_host,
                   dbs_path path, dbs_workspace *ws, void *stream);

/* Statistics of the last call on this workspace.  Synchronizes the stream.
 * Counts other than path/N_nzblk/y_nnz are filled only with collect_stats. */
typedef struct {
    int32_t path;               /* 1 push, 2 pull (BFS: last level) */
    int32_t status;             /* latched device status (not cleared here) */
    int64_t n_nzblk;            /* nonzero vector blocks of x (BFS: summed over levels) */
    int64_t n_blk;              /* ceil(n/16) */
    int64_t x_active;           /* active x entries */
    int64_t visited_blocks;     /* matrix blocks whose column block is nonzero in x */
    int64_t hit_blocks;         /* visited blocks whose columns intersect x's mask */
    int64_t touched_nnz;        /* nnz of visited blocks */
    int64_t bytes_alg;          /* algorithmic bytes: the bytes of views, block payload
                                   slices, vector and output that the chosen path must
                                   move for this x (a lower bound on DRAM traffic) */
    int64_t y_nnz;              /* output entries (BFS: vertices reached) */
    int32_t bfs_levels;         /* BFS: number of levels */
    int32_t bfs_push_levels;    /* BFS: levels run on the push path */
    int64_t phase_ns[3];        /* device time seen by block 0 (collect_stats only):
                                   metadata, traversal (BFS: all levels), output */
} dbs_stats;

dbs_status dbs_last_stats(dbs_workspace *ws, void *stream, dbs_stats *out);

/* Section 4.2 / Figure 7 diagnostics of the last dbs_bfs on this workspace
 * (the frontier evolution the paper profiles in Figure 3): for each level
 * l < min(max_levels, 64, number of levels), the frontier's nonzero vector
 * blocks, the matrix blocks in those column blocks (the blocks push visits),
 * the path taken (1 push, 2 pull), the level's device time in ns (traversal
 * + update, as seen by block 0) and the part of it up to the end of the
 * traversal.  HOST arrays, any may be NULL.  Synchronizes the stream.
 * DBS_ERR_INVALID_ARG if the last call was not a BFS. */
dbs_status dbs_bfs_level_stats(dbs_workspace *ws, void *stream, int32_t max_levels, int64_t *frontier_blocks,
                               int64_t *push_work, int32_t *path, int64_t *level_ns, int64_t *traversal_ns);

/* Self-test of the bounded device wait: launches the grid barrier with one
 * block withheld, so every other block's wait expires after
 * opts.wait_timeout_ns; the kernel latches DBS_ERR_TIMEOUT and returns.
 * dbs_workspace_check() then reports it.  No GPU fault is involved. */
dbs_status dbs_selftest_wait_timeout(dbs_workspace *ws, void *stream);

/* Allocation-free variant of dbs_spmspv_dense (the paper has no counterpart:
 * it is an interface for callers that may not allocate GPU memory after
 * start-up, such as real-time serving loops, where cudaMalloc's implicit
 * device synchronisation and late failures are not acceptable, or hosts that
 * reserve a fixed memory budget up front).  Same inputs and outputs as
 * dbs_spmspv_dense (x: device float32[n], y: device float32[m]), always on
 * the pull path, plus-times only.  Its scratch -- grid-barrier state,
 * counters and the vector-block masks, about 513 KiB -- is a fixed device
 * array inside the library that every GPU loading the library holds until
 * the process exits; the call itself allocates nothing.
 *   Limits: n <= 2^22 (4,194,304) columns, else DBS_ERR_INVALID_ARG; the
 *   matrix must be valued (else DBS_ERR_UNSUPPORTED) and on the current
 *   device.
 *   The first call on a device resolves the array's device address and the
 *   launch grid for that device (make it before any stream capture).
 *   All calls share the one array: calls that may overlap on the GPU (on
 *   different streams, or from different threads) race and must be
 *   serialised by the caller.  Each call clears the state it needs.
 *   A device-side wait that timed out leaves y undefined and is reported by
 *   dbs_spmspv_dense_noalloc_check.
 * ASYNC. */
dbs_status dbs_spmspv_dense_noalloc(const dbs_matrix *A, const float *x, float *y, void *stream);

/* Status of the last dbs_spmspv_dense_noalloc call on the current device:
 * synchronizes `stream` (the stream that call used), reads the error word of
 * the fixed scratch array (cudaMemcpyFromSymbol, no allocation) and returns
 * DBS_OK, or what that call latched on the device (DBS_ERR_TIMEOUT when a
 * bounded grid-barrier wait expired; y is then undefined).  The next
 * dbs_spmspv_dense_noalloc call clears the word, so query in between.
 * DBS_ERR_INVALID_ARG if no call has run on this device yet. */
dbs_status dbs_spmspv_dense_noalloc_check(void *stream);

/* Test hook (the paper has no counterpart): injects one allocation failure.
 * The k-th allocation attempt from now on (k = 0: the next one) fails as if
 * memory were exhausted -- device allocations (cudaMalloc) and the host
 * allocations of dbs_matrix_build_csr, dbs_workspace_create and
 * dbs_spmv_plan_create alike.  A call that meets it returns DBS_ERR_OOM
 * after releasing everything it had allocated.  k < 0 switches the hook
 * off; it also switches itself off after firing.  *previous (may be NULL)
 * receives the countdown it replaced: -1 when the last setting has fired
 * or was off, else the attempts that were still to come.  Process-wide and
 * not thread-safe with respect to concurrent builds; for tests. */
dbs_status dbs_debug_fail_alloc(int64_t k, int64_t *previous);

/* Human-readable name of a status. */
const char *dbs_status_string(dbs_status s);

/* Library version string, e.g. "dbspmspv 0.1 sm_103a". */
const char *dbs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DBSPMSPV_H */
