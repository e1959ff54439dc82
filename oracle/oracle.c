/*
 * CPU oracle for DB-SpMSpV -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
 * load this library.  It shares no code, header, table or helper with the
 * CUDA library: it is written from the paper's definitions, plainly and
 * slowly, in fp64, so that a reader can check it against the text by eye.
 *
 * Source: Cong et al., "DB-SpMSpV: Dual-View Blocked Sparse Matrix-Sparse
 * Vector Multiplication for Dynamic GPU Workloads" (ICPP '26).
 *   - oracle_spmspv_push : Section 2.1, Algorithm 1 (top, push over CSC),
 *                          followed by compaction of the touched rows.
 *   - oracle_spmspv_pull : Section 2.1, Algorithm 1 (bottom, pull over CSR),
 *                          used only as a cross-check of the push oracle.
 *   - oracle_bfs_queue   : textbook FIFO breadth-first search (Section 4.2
 *                          defines DB-BFS as level-synchronous BFS; its levels
 *                          are unique, so a queue BFS fixes them).
 *   - oracle_bfs_spmspv  : Section 4.2 / Algorithm 5 semantics: each level is
 *                          next = (A or.and frontier) and not visited.
 *   - oracle_spmv_csr    : the dense-input regime (the adaptive CSR SpMV page's
 *                          output contract: one product per CSR row over all
 *                          of its entries, x used as given, zeros included).
 *   - oracle_activation_mask : Section 4.3 / Section 5 (DB-Decoding): the
 *                          activation is sparsified by magnitude thresholding;
 *                          entry j is kept iff |x_j| > tau (NaN kept).  The
 *                          kept entries are the x of oracle_spmspv_push.
 *   - oracle_spmspv_pull_par, oracle_bfs_pull_par : the all-cores CPU
 *                          baseline -- Algorithm 1 (bottom) with the rows split
 *                          among OpenMP threads, and a level-synchronous BFS
 *                          made of such pulls; checked against the push
 *                          oracle and the queue BFS.
 *   - oracle_block_views : Section 3.2.1 and Figure 5(b): 16x16 blocking,
 *                          block-CSR view, block-CSC view, csc2csr mapping,
 *                          per-block nnz, and the low-level format class from
 *                          the th0/th1/th2 density and skew rule.
 *
 * Readings of points the paper leaves open:
 *   - Output pattern is structural: row i is in y iff some stored A(i,j) has
 *     an active x_j, even if the values cancel to zero.
 *   - x_j is active iff x_j != 0 (so -0.0 is inactive and NaN is active);
 *     with no values given every listed index is active.
 *   - Boolean semiring: y_i = OR_j (A(i,j) and x_j active) and not visited_i.
 *   - Skew rule: skew_a = max_l n_l(a) / (nnz/16 + eps); a block is ForceCSC
 *     if skew_r / skew_c > th2, else ForceCSR if skew_c / skew_r > th2, else
 *     patched CSR; th0 and th1 compare strictly (nnz < th0 -> COO,
 *     nnz > th1 -> Dense).
 *
 * Parity pins (tests/test_oracle.py): brute-force dense matvec on tiny
 * inputs, integer-valued exactness, unit vectors, permutations, push == pull,
 * closed-form BFS levels on grids / paths / stars, Figure 5's printed views.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Column-major copy of the input CSR, built once and reused across calls.  */

typedef struct {
    int64_t m, n, nnz;
    int64_t *col_ptr;   /* n + 1 */
    int64_t *row_idx;   /* nnz   */
    double  *val;       /* nnz, or NULL for a pattern-only matrix */
} oracle_csc;

void oracle_csc_free(oracle_csc *A)
{
    if (!A) return;
    free(A->col_ptr);
    free(A->row_idx);
    free(A->val);
    free(A);
}

/* Counting sort of the CSR entries by column; rows stay ascending inside a
 * column because the CSR is visited in row order. */
oracle_csc *oracle_csc_build(int64_t m, int64_t n, const int64_t *row_ptr,
                             const int32_t *col_idx, const float *vals)
{
    oracle_csc *A = (oracle_csc *)calloc(1, sizeof(oracle_csc));
    if (!A) return NULL;
    int64_t nnz = row_ptr[m];
    A->m = m; A->n = n; A->nnz = nnz;
    A->col_ptr = (int64_t *)calloc((size_t)n + 1, sizeof(int64_t));
    A->row_idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nnz > 0 ? nnz : 1));
    A->val = vals ? (double *)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1)) : NULL;
    int64_t *next = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!A->col_ptr || !A->row_idx || (vals && !A->val) || !next) {
        free(next);
        oracle_csc_free(A);
        return NULL;
    }
    for (int64_t k = 0; k < nnz; ++k) A->col_ptr[col_idx[k] + 1] += 1;
    for (int64_t j = 0; j < n; ++j) A->col_ptr[j + 1] += A->col_ptr[j];
    for (int64_t j = 0; j < n; ++j) next[j] = A->col_ptr[j];
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
            int64_t j = col_idx[k];
            int64_t dst = next[j]++;
            A->row_idx[dst] = i;
            if (vals) A->val[dst] = (double)vals[k];
        }
    }
    free(next);
    return A;
}

/* ------------------------------------------------------------------------ */
/* Algorithm 1 (top): push.  For every active x_j walk column j and add      */
/* A(i,j) * x_j into a dense accumulator; then compact the touched rows.     */
/*                                                                           */
/* semiring 0 = plus-times: y_val[t] = sum, y_abs[t] = sum of |A(i,j) x_j|.   */
/* semiring 1 = or-and:     y_val / y_abs untouched (may be NULL); rows with */
/*                          visited[i] != 0 are dropped.                      */
/* Returns the number of output entries, or -1 on allocation failure.        */
int64_t oracle_spmspv_push(const oracle_csc *A, int semiring,
                           int64_t x_nnz, const int32_t *x_idx, const float *x_val,
                           const uint8_t *visited,
                           int32_t *y_idx, double *y_val, double *y_abs)
{
    int64_t m = A->m;
    double *acc = (double *)calloc((size_t)(m > 0 ? m : 1), sizeof(double));
    double *sab = (double *)calloc((size_t)(m > 0 ? m : 1), sizeof(double));
    uint8_t *touched = (uint8_t *)calloc((size_t)(m > 0 ? m : 1), 1);
    if (!acc || !sab || !touched) { free(acc); free(sab); free(touched); return -1; }

    for (int64_t e = 0; e < x_nnz; ++e) {
        double xj = x_val ? (double)x_val[e] : 1.0;
        if (x_val && !(x_val[e] != 0.0f)) continue;      /* inactive entry */
        int64_t j = x_idx[e];
        for (int64_t k = A->col_ptr[j]; k < A->col_ptr[j + 1]; ++k) {
            int64_t i = A->row_idx[k];
            touched[i] = 1;
            if (semiring == 0) {
                double a = A->val ? A->val[k] : 1.0;
                double p = a * xj;          /* exact: 24 x 24 bits fit in 53 */
                acc[i] += p;
                sab[i] += fabs(p);
            }
        }
    }

    int64_t t = 0;
    for (int64_t i = 0; i < m; ++i) {
        if (!touched[i]) continue;
        if (semiring == 1 && visited && visited[i]) continue;
        y_idx[t] = (int32_t)i;
        if (semiring == 0) {
            if (y_val) y_val[t] = acc[i];
            if (y_abs) y_abs[t] = sab[i];
        }
        ++t;
    }
    free(acc); free(sab); free(touched);
    return t;
}

/* ------------------------------------------------------------------------ */
/* Algorithm 1 (bottom): pull.  Every row gathers A(i,j) * x_j over its      */
/* stored entries whose x_j is active.  Same outputs as the push oracle.     */
int64_t oracle_spmspv_pull(int64_t m, int64_t n, const int64_t *row_ptr,
                           const int32_t *col_idx, const float *vals, int semiring,
                           int64_t x_nnz, const int32_t *x_idx, const float *x_val,
                           const uint8_t *visited,
                           int32_t *y_idx, double *y_val, double *y_abs)
{
    double *xd = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    uint8_t *act = (uint8_t *)calloc((size_t)(n > 0 ? n : 1), 1);
    if (!xd || !act) { free(xd); free(act); return -1; }
    for (int64_t e = 0; e < x_nnz; ++e) {
        if (x_val && !(x_val[e] != 0.0f)) continue;
        xd[x_idx[e]] = x_val ? (double)x_val[e] : 1.0;
        act[x_idx[e]] = 1;
    }
    int64_t t = 0;
    for (int64_t i = 0; i < m; ++i) {
        double sum = 0.0, sab = 0.0;
        int hit = 0;
        for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
            int64_t j = col_idx[k];
            if (!act[j]) continue;
            hit = 1;
            if (semiring == 0) {
                double p = (vals ? (double)vals[k] : 1.0) * xd[j];
                sum += p;
                sab += fabs(p);
            }
        }
        if (!hit) continue;
        if (semiring == 1 && visited && visited[i]) continue;
        y_idx[t] = (int32_t)i;
        if (semiring == 0) {
            if (y_val) y_val[t] = sum;
            if (y_abs) y_abs[t] = sab;
        }
        ++t;
    }
    free(xd); free(act);
    return t;
}

/* ------------------------------------------------------------------------ */
/* Textbook FIFO BFS.  Vertex u reaches i when A(i,u) is stored (y = A x     */
/* propagates x_u into row i), i.e. the neighbours of u are column u.        */
/* levels[v] = hop distance from src, -1 if unreached.  Returns the number   */
/* of levels (max level + 1), or -1 on allocation failure.                   */
int64_t oracle_bfs_queue(const oracle_csc *A, int64_t src, int32_t *levels)
{
    int64_t n = A->n;
    int64_t *queue = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!queue) return -1;
    for (int64_t v = 0; v < n; ++v) levels[v] = -1;
    int64_t head = 0, tail = 0, nlev = 0;
    levels[src] = 0;
    queue[tail++] = src;
    while (head < tail) {
        int64_t u = queue[head++];
        if (levels[u] + 1 > nlev) nlev = levels[u] + 1;
        for (int64_t k = A->col_ptr[u]; k < A->col_ptr[u + 1]; ++k) {
            int64_t i = A->row_idx[k];
            if (levels[i] < 0) {
                levels[i] = levels[u] + 1;
                queue[tail++] = i;
            }
        }
    }
    free(queue);
    return nlev;
}

/* Level-synchronous BFS on the oracle SpMSpV: frontier = x, visited mask,  */
/* next = (A or.and frontier) and not visited (Section 4.2, Algorithm 5).    */
/* Returns the number of levels, -1 on allocation failure, -2 if more than   */
/* n levels were taken (impossible for a correct BFS).                       */
int64_t oracle_bfs_spmspv(const oracle_csc *A, int64_t src, int32_t *levels)
{
    int64_t n = A->n;
    int32_t *front = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    uint8_t *visited = (uint8_t *)calloc((size_t)(n > 0 ? n : 1), 1);
    if (!front || !next || !visited) { free(front); free(next); free(visited); return -1; }
    for (int64_t v = 0; v < n; ++v) levels[v] = -1;
    int64_t nf = 1, level = 0;
    front[0] = (int32_t)src;
    visited[src] = 1;
    levels[src] = 0;
    while (nf > 0) {
        if (level > n) { nf = -2; break; }   /* a BFS has at most n levels */
        int64_t nn = oracle_spmspv_push(A, 1, nf, front, NULL, visited, next, NULL, NULL);
        if (nn < 0) { nf = -1; break; }
        ++level;
        for (int64_t t = 0; t < nn; ++t) {
            visited[next[t]] = 1;
            levels[next[t]] = (int32_t)level;
        }
        int32_t *tmp = front; front = next; next = tmp;
        nf = nn;
    }
    free(front); free(next); free(visited);
    return nf < 0 ? nf : level;
}

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* ------------------------------------------------------------------------ */
/* Section 3.2.1 / Figure 5(b): the high-level dual views and the low-level  */
/* format class of every nonzero bs x bs block.                              */
/*                                                                           */
/* Outputs (caller-allocated; B <= nnz):                                     */
/*   blk_row_ptr[nbr+1], blk_col_idx[B]        block-CSR view (primary order) */
/*   blk_col_ptr[nbc+1], blk_row_idx[B]        block-CSC view                 */
/*   blk_csc2csr[B]                            CSC position -> primary id     */
/*   blk_nnz[B], blk_class[B]                  0 COO, 1 Dense, 2 ForceCSR,    */
/*                                             3 ForceCSC, 4 patched CSR      */
/* Returns B, or -1 on allocation failure.                                   */
int64_t oracle_block_views(int64_t m, int64_t n, const int64_t *row_ptr,
                           const int32_t *col_idx, int bs,
                           int th0, int th1, double th2,
                           int64_t *blk_row_ptr, int64_t *blk_col_idx,
                           int64_t *blk_col_ptr, int64_t *blk_row_idx,
                           int64_t *blk_csc2csr, int32_t *blk_nnz, int32_t *blk_class)
{
    int64_t nbr = (m + bs - 1) / bs, nbc = (n + bs - 1) / bs;
    /* per row block: mark the column blocks that hold an entry */
    int32_t *cnt = (int32_t *)calloc((size_t)(nbc > 0 ? nbc : 1), sizeof(int32_t));
    int32_t *rowc = (int32_t *)malloc(sizeof(int32_t) * (size_t)bs * (size_t)(nbc > 0 ? nbc : 1));
    int32_t *colc = (int32_t *)malloc(sizeof(int32_t) * (size_t)bs * (size_t)(nbc > 0 ? nbc : 1));
    int64_t *seen = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nbc > 0 ? nbc : 1));
    if (!cnt || !rowc || !colc || !seen) { free(cnt); free(rowc); free(colc); free(seen); return -1; }
    int64_t B = 0;
    blk_row_ptr[0] = 0;
    for (int64_t rb = 0; rb < nbr; ++rb) {
        int64_t r0 = rb * bs, r1 = r0 + bs < m ? r0 + bs : m;
        int64_t nseen = 0;
        for (int64_t i = r0; i < r1; ++i)
            for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
                int64_t cb = col_idx[k] / bs;
                if (cnt[cb] == 0) {
                    memset(rowc + cb * bs, 0, sizeof(int32_t) * (size_t)bs);
                    memset(colc + cb * bs, 0, sizeof(int32_t) * (size_t)bs);
                    seen[nseen++] = cb;
                }
                cnt[cb] += 1;
                rowc[cb * bs + (i - r0)] += 1;
                colc[cb * bs + (col_idx[k] % bs)] += 1;
            }
        qsort(seen, (size_t)nseen, sizeof(int64_t), cmp_i64);
        for (int64_t s = 0; s < nseen; ++s) {
            int64_t cb = seen[s];
            int32_t z = cnt[cb];
            int32_t maxr = 0, maxc = 0;
            for (int l = 0; l < bs; ++l) {
                if (rowc[cb * bs + l] > maxr) maxr = rowc[cb * bs + l];
                if (colc[cb * bs + l] > maxc) maxc = colc[cb * bs + l];
            }
            int32_t cls;
            if (z < th0) cls = 0;
            else if (z > th1) cls = 1;
            else {
                const double eps = 1e-9;
                double skew_r = (double)maxr / ((double)z / (double)bs + eps);
                double skew_c = (double)maxc / ((double)z / (double)bs + eps);
                if (skew_r / skew_c > th2) cls = 3;        /* ForceCSC */
                else if (skew_c / skew_r > th2) cls = 2;   /* ForceCSR */
                else cls = 4;                              /* patched CSR */
            }
            blk_col_idx[B] = cb;
            blk_nnz[B] = z;
            blk_class[B] = cls;
            ++B;
            cnt[cb] = 0;
        }
        blk_row_ptr[rb + 1] = B;
    }
    free(cnt); free(rowc); free(colc); free(seen);

    /* block-CSC view: counting sort of the primary blocks by column block */
    for (int64_t cb = 0; cb <= nbc; ++cb) blk_col_ptr[cb] = 0;
    for (int64_t p = 0; p < B; ++p) blk_col_ptr[blk_col_idx[p] + 1] += 1;
    for (int64_t cb = 0; cb < nbc; ++cb) blk_col_ptr[cb + 1] += blk_col_ptr[cb];
    int64_t *next = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nbc > 0 ? nbc : 1));
    if (!next) return -1;
    for (int64_t cb = 0; cb < nbc; ++cb) next[cb] = blk_col_ptr[cb];
    for (int64_t rb = 0; rb < nbr; ++rb)
        for (int64_t p = blk_row_ptr[rb]; p < blk_row_ptr[rb + 1]; ++p) {
            int64_t q = next[blk_col_idx[p]]++;
            blk_row_idx[q] = rb;
            blk_csc2csr[q] = p;
        }
    free(next);
    return B;
}

/* ------------------------------------------------------------------------ */
/* DB-Decoding activation mask (magnitude thresholding): writes the indices */
/* j with NOT(|x_j| <= tau) -- |x_j| > tau, NaN included -- in ascending     */
/* order and returns how many there are.                                    */
int64_t oracle_activation_mask(int64_t n, const float *x, float tau, int32_t *idx_out)
{
    int64_t k = 0;
    for (int64_t j = 0; j < n; ++j) {
        double a = fabs((double)x[j]);
        if (!(a <= (double)tau)) idx_out[k++] = (int32_t)j;
    }
    return k;
}

/* ------------------------------------------------------------------------ */
/* Plain CSR SpMV: y_i = sum over the entries k of row i of a_k * x[col_k]   */
/* (every entry, whatever x holds; columns outside [0, n) skipped), with     */
/* abs_i = sum of |a_k * x[col_k]| for the tolerance.                       */
void oracle_spmv_csr(int64_t m, int64_t n, const int64_t *row_ptr, const int32_t *col_idx, const float *vals,
                     const float *x, double *y, double *abs_out)
{
    for (int64_t i = 0; i < m; ++i) {
        double acc = 0.0, sab = 0.0;
        for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
            int64_t j = col_idx[k];
            if (j < 0 || j >= n) continue;
            double p = (double)vals[k] * (double)x[j];
            acc += p;
            sab += fabs(p);
        }
        y[i] = acc;
        abs_out[i] = sab;
    }
}

/* ------------------------------------------------------------------------ */
/* All-cores CPU baseline (not a pin: it is checked against the functions   */
/* above).  Algorithm 1 (bottom), the row-wise pull, with the rows split     */
/* among OpenMP threads; and a level-synchronous BFS whose levels are each   */
/* one such pull (Section 4.2: next = (A or.and frontier) and not visited). */
/* Without OpenMP both run on one thread.                                    */
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_par_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Same contract as oracle_spmspv_pull.  Each thread owns a contiguous range  */
/* of rows and writes their sums and hit flags into dense arrays; the         */
/* ascending output is compacted afterwards.                                  */
int64_t oracle_spmspv_pull_par(int64_t m, int64_t n, const int64_t *row_ptr,
                               const int32_t *col_idx, const float *vals, int semiring,
                               int64_t x_nnz, const int32_t *x_idx, const float *x_val,
                               const uint8_t *visited,
                               int32_t *y_idx, double *y_val, double *y_abs)
{
    double *xd = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    uint8_t *act = (uint8_t *)calloc((size_t)(n > 0 ? n : 1), 1);
    double *ysum = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    double *yab = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    uint8_t *hit = (uint8_t *)malloc((size_t)(m > 0 ? m : 1));
    if (!xd || !act || !ysum || !yab || !hit) {
        free(xd); free(act); free(ysum); free(yab); free(hit);
        return -1;
    }
    for (int64_t e = 0; e < x_nnz; ++e) {
        if (x_val && !(x_val[e] != 0.0f)) continue;
        xd[x_idx[e]] = x_val ? (double)x_val[e] : 1.0;
        act[x_idx[e]] = 1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i) {
        double sum = 0.0, sab = 0.0;
        uint8_t h = 0;
        for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
            int64_t j = col_idx[k];
            if (!act[j]) continue;
            h = 1;
            if (semiring == 0) {
                double p = (vals ? (double)vals[k] : 1.0) * xd[j];
                sum += p;
                sab += fabs(p);
            }
        }
        if (semiring == 1 && visited && visited[i]) h = 0;
        hit[i] = h;
        ysum[i] = sum;
        yab[i] = sab;
    }
    int64_t t = 0;
    for (int64_t i = 0; i < m; ++i) {
        if (!hit[i]) continue;
        y_idx[t] = (int32_t)i;
        if (semiring == 0) {
            if (y_val) y_val[t] = ysum[i];
            if (y_abs) y_abs[t] = yab[i];
        }
        ++t;
    }
    free(xd); free(act); free(ysum); free(yab); free(hit);
    return t;
}

/* Level-synchronous BFS over the CSR of a square matrix: at level L every   */
/* unreached row i with a stored A(i,j) whose j was reached at level L - 1    */
/* is reached at level L; rows are split among the threads.  Returns the     */
/* number of levels, or -1 on allocation failure.                            */
int64_t oracle_bfs_pull_par(int64_t n, const int64_t *row_ptr, const int32_t *col_idx, int64_t src,
                            int32_t *levels)
{
    uint8_t *next = (uint8_t *)calloc((size_t)(n > 0 ? n : 1), 1);
    if (!next) return -1;
    for (int64_t v = 0; v < n; ++v) levels[v] = -1;
    levels[src] = 0;
    int64_t level = 0;
    for (;;) {
        int64_t found = 0;
        /* this pass reads levels and writes only next */
#pragma omp parallel for schedule(dynamic, 4096) reduction(+ : found)
        for (int64_t i = 0; i < n; ++i) {
            if (levels[i] >= 0) continue;
            for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
                if (levels[col_idx[k]] == (int32_t)level) {
                    next[i] = 1;
                    ++found;
                    break;
                }
            }
        }
        if (found == 0) break;
        ++level;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i)
            if (next[i]) { levels[i] = (int32_t)level; next[i] = 0; }
    }
    free(next);
    return level + 1;
}
