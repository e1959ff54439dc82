// Dense-input regime: adaptive CSR SpMV (sm_103a), y = A x for a dense x.
//
// Restates the execution families of the adaptive CSR SpMV page (GPU
// adaptive SpMV execution: scalar rows, subgroup rows, workgroup rows,
// long-row split) for CUDA, for inputs dense enough that SpMSpV's vector
// metadata buys nothing (the DB-SpMSpV paper's Limitations: conventional SpMV
// may be preferable for dense inputs).
//
//   plan (once per CSR, on the GPU, no host readback): every row is put in
//   a bucket by its length -- scalar (one thread, up to 4 entries), subgroup
//   rows (a group of 2, 4, 8, 16 or 32 lanes of a warp, the width the
//   smallest power of two giving each lane at most 4 entries, 32 for rows up
//   to 1024: the page's subgroup family, narrowed so that short rows do not
//   leave most of a warp idle), block rows (one 256-thread block: the page's
//   workgroup) or split rows (chunks of SPMV_CHUNK entries, one block each,
//   whose partial sums the last chunk to finish adds up: the page's long-row
//   strategy).  Rows keep their order inside a bucket.  This is the page's
//   "GPU classifier that buckets rows and generates indirect queues".
//   multiply: one ordinary persistent launch walks the queues (split chunks
//   and block rows first, then the subgroup and scalar rows); every row of y
//   is written exactly once, rows without entries as 0, so y needs no
//   clearing and consecutive calls need no host work.  A lane's entries are
//   loaded in groups of four before any product is formed.
//
// Column indices outside [0, n) contribute nothing; row pointers are clamped
// to [0, nnz], so a malformed CSR gives wrong numbers but no stray access.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "../../include/dbspmspv.h"
#include "internal.h"

#include "spmv_dev.h"

using namespace dbs::spmvd;

namespace {

// Plan pass 1: rows (and split chunks) per bucket in each plan block.
__global__ void __launch_bounds__(NT) k_plan_count(PlanDev D)
{
    uint32_t c[NB] = {};
    const int64_t base = (int64_t)blockIdx.x * PLAN_ROWS;
    for (int i = 0; i < ROWS_PER_THREAD; ++i) {
        const int64_t r = base + (int64_t)i * NT + threadIdx.x;
        if (r >= D.m) break;
        int64_t s, e;
        row_range(D, r, s, e);
        const int b = bucket_of(e - s);
        ++c[b];
        if (b == B_SPLIT) c[NBK] += n_chunks(e - s);
    }
    for (int k = 0; k < NB; ++k) {
        uint32_t tot;
        block_scan(c[k], &tot);
        if (threadIdx.x == 0) D.blk_counts[(size_t)blockIdx.x * NB + k] = tot;
    }
}

// Plan pass 2: exclusive offsets of every plan block per counter (one block).
__global__ void __launch_bounds__(NT) k_plan_scan(PlanDev D, uint32_t nblocks)
{
    for (int k = 0; k < NB; ++k) {
        uint32_t carry = 0;
        for (uint32_t b0 = 0; b0 < nblocks; b0 += NT) {
            const uint32_t b = b0 + threadIdx.x;
            const uint32_t v = b < nblocks ? D.blk_counts[(size_t)b * NB + k] : 0u;
            uint32_t tot;
            const uint32_t o = block_scan(v, &tot);
            if (b < nblocks) D.blk_offs[(size_t)b * NB + k] = carry + o;
            carry += tot;
        }
        if (threadIdx.x == 0) D.tot[k] = carry;
    }
}

// Plan pass 3: write the rows in order into their buckets, and the split
// rows' chunk table.
__global__ void __launch_bounds__(NT) k_plan_fill(PlanDev D)
{
    uint32_t off[NB];
    for (int k = 0; k < NB; ++k) off[k] = D.blk_offs[(size_t)blockIdx.x * NB + k];
    const int64_t base = (int64_t)blockIdx.x * PLAN_ROWS;
    for (int i = 0; i < ROWS_PER_THREAD; ++i) {
        const int64_t r = base + (int64_t)i * NT + threadIdx.x;
        int b = -1;
        int64_t len = 0;
        if (r < D.m) {
            int64_t s, e;
            row_range(D, r, s, e);
            len = e - s;
            b = bucket_of(len);
        }
        const uint32_t nc = b == B_SPLIT ? n_chunks(len) : 0u;
        uint32_t t[NB];
        uint32_t pos[NB];
        for (int k = 0; k < NBK; ++k) pos[k] = block_scan(b == k ? 1u : 0u, &t[k]);
        pos[NBK] = block_scan(nc, &t[NBK]);
        if (b >= 0 && b < B_SPLIT) {
            int64_t s, e;
            row_range(D, r, s, e);
            D.rows[b][off[b] + pos[b]] = make_uint4((uint32_t)r, (uint32_t)s, (uint32_t)(e - s), 0u);
        }
        if (b == B_SPLIT) {
            const uint32_t si = off[B_SPLIT] + pos[B_SPLIT], c0 = off[NBK] + pos[NBK];
            D.split[si] = SplitRow{(uint32_t)r, c0, nc, 0u};
            for (uint32_t k = 0; k < nc; ++k) D.chunks[c0 + k] = make_uint2(si, k);
        }
        for (int k = 0; k < NB; ++k) off[k] += t[k];
    }
}


// One persistent launch over the queues (x used as given).
__global__ void __launch_bounds__(NT) k_spmv(PlanDev D, const float *__restrict__ x, float *__restrict__ y)
{
    spmv_items<false>(D, x, y);
}

// The SpMV of a dense-x SpMSpV call (dbs_spmspv_dense on a matrix with a
// kept plan): entries whose x is zero are skipped (the structural product).
// GATED: only when the sample says x is dense; the blocked kernel launched
// after it reads the same sample and does the call otherwise.  Block 0
// records the path taken in *path_word (3) when it runs.
template <bool GATED>
__global__ void __launch_bounds__(NT) k_spmv_dense(PlanDev D, const float *__restrict__ x, float *__restrict__ y,
                                                   double frac, unsigned *path_word)
{
    if (GATED && !dense_x_sample(x, D.n, frac)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0 && path_word) *path_word = 3u;
    spmv_items<true>(D, x, y);
}

}  // namespace

namespace {

template <class T>
bool alloc0(T **p, size_t count)
{
    const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
    if (dbs::dev_malloc(p, bytes) != cudaSuccess) { cudaGetLastError(); *p = nullptr; return false; }
    if (cudaMemset(*p, 0, bytes) != cudaSuccess) { cudaGetLastError(); return false; }
    return true;
}

void plan_free(dbs_spmv_plan *p)
{
    PlanDev &D = p->D;
    for (int k = 0; k < B_SPLIT; ++k) dbs::dev_free(D.rows[k]);
    dbs::dev_free(D.split); dbs::dev_free(D.chunks); dbs::dev_free(D.part); dbs::dev_free(D.cnt);
    dbs::dev_free(D.blk_counts); dbs::dev_free(D.blk_offs); dbs::dev_free(D.tot);
}

}  // namespace

dbs_status dbs::spmv_launch_dense(const dbs_spmv_plan *p, float *part, uint32_t *cnt, const float *x, float *y,
                                  double frac, bool gated, unsigned *path_word, cudaStream_t s)
{
    if (p->D.m == 0) return DBS_OK;
    PlanDev D = p->D;
    D.part = part;
    D.cnt = cnt;
    if (gated) k_spmv_dense<true><<<p->grid, NT, 0, s>>>(D, x, y, frac, path_word);
    else k_spmv_dense<false><<<p->grid, NT, 0, s>>>(D, x, y, frac, path_word);
    return cudaGetLastError() == cudaSuccess ? DBS_OK : DBS_ERR_CUDA;
}

int64_t dbs::spmv_plan_bytes(const dbs_spmv_plan *p)
{
    if (!p) return 0;
    const int64_t m1 = p->D.m + 1, nb = (int64_t)p->nplan * NB + NB;
    return B_SPLIT * m1 * 16 + (int64_t)p->max_split * (16 + 4) + (int64_t)p->max_chunks * (8 + 4) + 2 * nb * 4 + NB * 4;
}

extern "C" {

dbs_status dbs_spmv_plan_create(int64_t m, int64_t n, int64_t nnz, const int64_t *row_ptr, const int32_t *col_idx,
                                const float *vals, void *stream, dbs_spmv_plan **out)
{
    if (!out || m < 0 || n < 0 || nnz < 0 || m >= (int64_t(1) << 31) || n >= (int64_t(1) << 31) || !row_ptr ||
        (nnz > 0 && (!col_idx || !vals)))
        return DBS_ERR_INVALID_ARG;
    // entry offsets in the row queues are 32-bit
    if (nnz >= (int64_t(1) << 32)) return DBS_ERR_UNSUPPORTED;
    dbs_spmv_plan *p = dbs::alloc_fault() ? nullptr : new (std::nothrow) dbs_spmv_plan();
    if (!p) return DBS_ERR_OOM;
    PlanDev &D = p->D;
    D.m = m; D.n = n; D.nnz = nnz; D.rp = row_ptr; D.ci = col_idx; D.va = vals;
    int sms = 0;
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return DBS_ERR_CUDA;
    }
    // persistent grid: as many blocks as stay resident together (the items
    // are dealt out by block index, so a block that waits for a slot would
    // add its items to the end of the launch)
    int per_sm = 8;
    {
        int o[3] = {0, 0, 0};
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o[0], k_spmv, NT, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o[1], k_spmv_dense<true>, NT, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o[2], k_spmv_dense<false>, NT, 0) != cudaSuccess) {
            cudaGetLastError();
            delete p;
            return DBS_ERR_CUDA;
        }
        per_sm = std::min(o[0], std::min(o[1], o[2]));
    }
    p->grid = std::max(1, sms * std::max(1, per_sm));
    p->nplan = (uint32_t)((m + PLAN_ROWS - 1) / PLAN_ROWS);
    const size_t max_chunks = (size_t)(nnz / SPMV_CHUNK) + (size_t)(nnz / (LEN_CTA + 1)) + 2;
    const size_t max_split = (size_t)(nnz / (LEN_CTA + 1)) + 1;
    p->max_chunks = max_chunks;
    p->max_split = max_split;
    bool ok = true;
    for (int k = 0; k < B_SPLIT && ok; ++k) ok = alloc0(&D.rows[k], (size_t)m + 1);
    ok = ok && alloc0(&D.split, max_split) && alloc0(&D.chunks, max_chunks) &&
              alloc0(&D.part, max_chunks) && alloc0(&D.cnt, max_split) &&
              alloc0(&D.blk_counts, (size_t)p->nplan * NB + NB) && alloc0(&D.blk_offs, (size_t)p->nplan * NB + NB) &&
              alloc0(&D.tot, NB);
    if (!ok) { plan_free(p); delete p; return DBS_ERR_OOM; }
    cudaStream_t s = (cudaStream_t)stream;
    if (p->nplan > 0) {
        k_plan_count<<<p->nplan, NT, 0, s>>>(D);
        k_plan_scan<<<1, NT, 0, s>>>(D, p->nplan);
        k_plan_fill<<<p->nplan, NT, 0, s>>>(D);
    }
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        plan_free(p);
        delete p;
        return DBS_ERR_CUDA;
    }
    *out = p;
    return DBS_OK;
}

dbs_status dbs_spmv(dbs_spmv_plan *p, const float *x, float *y, void *stream)
{
    if (!p || (p->D.n > 0 && !x) || (p->D.m > 0 && !y)) return DBS_ERR_INVALID_ARG;
    if (p->D.m == 0) return DBS_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    if (dev != p->device) return DBS_ERR_INVALID_ARG;
    k_spmv<<<p->grid, NT, 0, (cudaStream_t)stream>>>(p->D, x, y);
    if (cudaGetLastError() != cudaSuccess) return DBS_ERR_CUDA;
    return DBS_OK;
}

dbs_status dbs_spmv_plan_info(const dbs_spmv_plan *p, int64_t *bucket_rows, int64_t *split_chunks)
{
    if (!p) return DBS_ERR_INVALID_ARG;
    uint32_t t[NB];
    if (cudaMemcpy(t, p->D.tot, sizeof(t), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    if (bucket_rows)
        for (int k = 0; k < NBK; ++k) bucket_rows[k] = t[k];
    if (split_chunks) *split_chunks = t[NBK];
    return DBS_OK;
}

dbs_status dbs_spmv_plan_destroy(dbs_spmv_plan *p)
{
    if (!p) return DBS_OK;
    plan_free(p);
    delete p;
    return DBS_OK;
}

}  // extern "C"
