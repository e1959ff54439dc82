// Adaptive CSR SpMV device code (sm_103a), shared by the dense-input calls
// (spmv.cu: plan and dbs_spmv) and by the dense-x SpMSpV kernel, which hands
// a dense enough x to it (kernels.cu).
//
// Restates the execution families of the adaptive CSR SpMV page (GPU
// adaptive SpMV execution: scalar rows, subgroup rows, workgroup rows,
// long-row split) for CUDA: every row is put in a bucket by its length --
// scalar (one thread, up to 4 entries), subgroup rows (a group of 2, 4, 8,
// 16 or 32 lanes of a warp, the width the smallest power of two giving each
// lane at most 4 entries, 32 for rows up to 1024), block rows (one 256-thread
// block: the page's workgroup) or split rows (chunks of SPMV_CHUNK entries,
// one block each, whose partial sums the last chunk to finish adds up: the
// page's long-row strategy).  Every row of y is written exactly once, rows
// without entries as 0.
//
// Column indices outside [0, n) contribute nothing; row pointers are clamped
// to [0, nnz], so a malformed CSR gives wrong numbers but no stray access.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace dbs {
namespace spmvd {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr unsigned FULL = 0xFFFFFFFFu;
constexpr int ROWS_PER_THREAD = 8;                  // plan: rows classified per thread
constexpr int PLAN_ROWS = NT * ROWS_PER_THREAD;     // rows per plan block
constexpr int64_t PER_LANE = 4;                     // entries per lane below 32-lane rows
constexpr int64_t LEN_WARP = 1024;                  // longest row for one warp
constexpr int64_t LEN_CTA = 16384;                  // longest row for one block
constexpr int64_t SPMV_CHUNK = 8192;                // entries per split chunk
// buckets: 0-5 rows on 1, 2, 4, 8, 16, 32 lanes; 6 block rows; 7 split rows
constexpr int NBK = 8;
constexpr int B_BLOCK = 6, B_SPLIT = 7;
constexpr int NB = NBK + 1;                         // counters: buckets + split chunks

struct SplitRow {
    uint32_t row;
    uint32_t chunk0;    // first chunk (and partial-sum slot) of the row
    uint32_t nchunks;
    uint32_t pad;
};

struct PlanDev {
    int64_t m, n, nnz;
    const int64_t *rp;
    const int32_t *ci;
    const float *va;
    uint4 *rows[B_SPLIT];       // buckets 0-6 (lane groups, block rows): {row, first entry, length, 0}
    SplitRow *split;            // split rows
    uint2 *chunks;              // {split row index, chunk number within the row}
    float *part;                // one partial sum per chunk
    uint32_t *cnt;              // chunks done per split row (zero between calls)
    uint32_t *blk_counts;       // plan: [blocks][NB]
    uint32_t *blk_offs;         // plan: [blocks][NB]
    uint32_t *tot;              // NB totals
};

__device__ __forceinline__ void row_range(const PlanDev &D, int64_t r, int64_t &s, int64_t &e)
{
    s = min(max(__ldg(D.rp + r), (int64_t)0), D.nnz);
    e = min(max(__ldg(D.rp + r + 1), s), D.nnz);
}

__device__ __forceinline__ int bucket_of(int64_t len)
{
    if (len > LEN_CTA) return B_SPLIT;
    if (len > LEN_WARP) return B_BLOCK;
    int b = 0;
    while (b < 5 && len > PER_LANE << b) ++b;     // 2^b lanes, at most 4 entries each (32 lanes: up to 1024)
    return b;
}

__device__ __forceinline__ uint32_t n_chunks(int64_t len) { return (uint32_t)((len + SPMV_CHUNK - 1) / SPMV_CHUNK); }

// Block-wide exclusive scan (all threads call it).
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *total)
{
    __shared__ uint32_t s_w[NW];
    __shared__ uint32_t s_t;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s_w[w] = inc;
    __syncthreads();
    if (w == 0) {
        const uint32_t x = lane < NW ? s_w[lane] : 0u;
        uint32_t xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(FULL, xi, o);
            if (lane >= o) xi += t;
        }
        if (lane < NW) s_w[lane] = xi - x;
        if (lane == NW - 1) s_t = xi;
    }
    __syncthreads();
    const uint32_t r = s_w[w] + inc - v;
    *total = s_t;
    __syncthreads();
    return r;
}


// Sum of one value per thread over the block; the result on every thread.
__device__ __forceinline__ float block_sum(float v)
{
    __shared__ float s_p[NW];
    __shared__ float s_r;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane == 0) s_p[w] = v;
    __syncthreads();
    if (w == 0) {
        float x = lane < NW ? s_p[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
        if (lane == 0) s_r = x;
    }
    __syncthreads();
    const float r = s_r;
    __syncthreads();
    return r;
}

// Sum of a_k x[col_k] over k = s + start, s + start + stride, ... < e, four
// entries' loads issued before their products.  ZC: entries whose x is zero
// are skipped (the structural product of DB-SpMSpV, where x_j = 0 is
// inactive); without it every entry is used as the SpMV page states.
template <bool ZC = false>
__device__ __forceinline__ float dot_range(const PlanDev &D, const float *__restrict__ x, int64_t s, int64_t e,
                                           int64_t start, int stride)
{
    float acc = 0.0f;
    for (int64_t k = s + start; k < e; k += 4 * (int64_t)stride) {
        uint32_t c[4];
        float a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t q = k + (int64_t)u * stride;
            c[u] = q < e ? (uint32_t)__ldg(D.ci + q) : 0xFFFFFFFFu;
            a[u] = q < e ? __ldg(D.va + q) : 0.0f;
        }
        float xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) xv[u] = c[u] < (uint32_t)D.n ? __ldg(x + c[u]) : 0.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c[u] < (uint32_t)D.n && (!ZC || xv[u] != 0.0f)) acc = fmaf(a[u], xv[u], acc);
    }
    return acc;
}

// Rows of buckets 0-4 (2^b lanes, at most 4 entries per lane): two rows per
// lane group and item (2 * (NT >> b) rows), all eight entries' loads of a
// lane issued before any product, so a group keeps both rows in flight.
template <int LOGW, bool ZC = false>
__device__ __forceinline__ void group_rows_short(const PlanDev &D, const float *__restrict__ x, float *__restrict__ y,
                                                 uint32_t item, uint32_t nrows)
{
    constexpr int W = 1 << LOGW, R = NT / W;
    const int tid = threadIdx.x, g = tid & (W - 1);
    const uint32_t j0 = item * (2u * R) + (uint32_t)(tid >> LOGW), j[2] = {j0, j0 + R};
    uint32_t r[2] = {0u, 0u};
    int64_t s[2] = {0, 0}, e[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (j[h] < nrows) {
            const uint4 q = D.rows[LOGW][j[h]];
            r[h] = q.x;
            s[h] = q.y;
            e[h] = (int64_t)q.y + q.z;
        }
    uint32_t c[2][4];
    float a[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t q = s[h] + g + (int64_t)u * W;
            c[h][u] = q < e[h] ? (uint32_t)__ldg(D.ci + q) : 0xFFFFFFFFu;
            a[h][u] = q < e[h] ? __ldg(D.va + q) : 0.0f;
        }
    float v[2] = {0.0f, 0.0f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) xv[u] = c[h][u] < (uint32_t)D.n ? __ldg(x + c[h][u]) : 0.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c[h][u] < (uint32_t)D.n && (!ZC || xv[u] != 0.0f)) v[h] = fmaf(a[h][u], xv[u], v[h]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) v[h] += __shfl_xor_sync(FULL, v[h], o);
        if (g == 0 && j[h] < nrows) y[r[h]] = v[h];
    }
}

// Rows of bucket 5 (32 lanes, up to 1024 entries): NT / 32 rows per item.
template <int LOGW, bool ZC = false>
__device__ __forceinline__ void group_rows(const PlanDev &D, const float *__restrict__ x, float *__restrict__ y,
                                           uint32_t item, uint32_t nrows)
{
    constexpr int W = 1 << LOGW;
    const int tid = threadIdx.x, g = tid & (W - 1);
    const uint32_t j = item * (NT / W) + (uint32_t)(tid >> LOGW);
    float v = 0.0f;
    uint32_t r = 0;
    if (j < nrows) {
        const uint4 q = D.rows[LOGW][j];
        r = q.x;
        v = dot_range<ZC>(D, x, q.y, (int64_t)q.y + q.z, g, W);
    }
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    if (g == 0 && j < nrows) y[r] = v;
}


// The multiply: items are [split chunks | block rows | lane-group rows of
// 32, 16, 8, 4, 2 and 1 lanes: NT / 32 rows per item for 32 lanes, 2 * NT /
// width below], walked by a persistent grid of NT-thread blocks (every
// thread of a block calls this).
template <bool ZC>
__device__ __forceinline__ void spmv_items(const PlanDev &D, const float *__restrict__ x, float *__restrict__ y)
{
    __shared__ int s_last;
    uint32_t lim[NBK + 1];
    {
        uint32_t acc = D.tot[NBK];                       // split chunks
        lim[0] = acc;
        acc += D.tot[B_BLOCK];                           // block rows
        lim[1] = acc;
        for (int b = 5; b >= 0; --b) {                   // lane groups, widest first
            const uint32_t per = b == 5 ? NT >> 5 : 2u * (NT >> b);
            acc += (D.tot[b] + per - 1) / per;
            lim[2 + (5 - b)] = acc;
        }
    }
    const uint32_t total = lim[7];
    const int tid = threadIdx.x;
    for (uint32_t it = blockIdx.x; it < total; it += gridDim.x) {
        if (it < lim[0]) {
            const uint2 ch = D.chunks[it];
            const SplitRow sr = D.split[ch.x];
            int64_t s, e;
            row_range(D, sr.row, s, e);
            const int64_t cs = s + (int64_t)ch.y * SPMV_CHUNK, ce = min(e, cs + SPMV_CHUNK);
            const float v = block_sum(dot_range<ZC>(D, x, cs, ce, tid, NT));
            if (tid == 0) {
                D.part[sr.chunk0 + ch.y] = v;
                __threadfence();
                s_last = atomicAdd(D.cnt + ch.x, 1u) == sr.nchunks - 1u;
            }
            __syncthreads();
            if (s_last) {
                // last chunk of the row: add the partial sums in chunk order
                __threadfence();
                float p = 0.0f;
                for (uint32_t k = tid; k < sr.nchunks; k += NT) p += __ldcg(D.part + sr.chunk0 + k);
                const float tot = block_sum(p);
                if (tid == 0) {
                    y[sr.row] = tot;
                    D.cnt[ch.x] = 0u;
                }
            }
            __syncthreads();
        } else if (it < lim[1]) {
            const uint4 q = D.rows[B_BLOCK][it - lim[0]];
            const float v = block_sum(dot_range<ZC>(D, x, q.y, (int64_t)q.y + q.z, tid, NT));
            if (tid == 0) y[q.x] = v;
        } else if (it < lim[2]) {
            group_rows<5, ZC>(D, x, y, it - lim[1], D.tot[5]);
        } else if (it < lim[3]) {
            group_rows_short<4, ZC>(D, x, y, it - lim[2], D.tot[4]);
        } else if (it < lim[4]) {
            group_rows_short<3, ZC>(D, x, y, it - lim[3], D.tot[3]);
        } else if (it < lim[5]) {
            group_rows_short<2, ZC>(D, x, y, it - lim[4], D.tot[2]);
        } else if (it < lim[6]) {
            group_rows_short<1, ZC>(D, x, y, it - lim[5], D.tot[1]);
        } else {
            group_rows_short<0, ZC>(D, x, y, it - lim[6], D.tot[0]);
        }
    }
}



// Whether a dense x is dense enough for the SpMV: the nonzero fraction of a
// fixed sample of x -- 8 runs of 32 consecutive entries, evenly spaced (all
// of x when n <= 256) -- is at least `frac`.  Every NT-thread block that
// calls it reads the same entries and reaches the same answer; all threads
// of the block call it.
__device__ __forceinline__ bool dense_x_sample(const float *__restrict__ x, int64_t n, double frac)
{
    static_assert(NT == 256, "one sampled entry per thread");
    const int t = threadIdx.x;
    int64_t j;
    uint32_t ns;
    if (n <= NT) {
        j = t;
        ns = (uint32_t)n;
    } else {
        j = (int64_t)(t >> 5) * (n / 8) + (t & 31);
        ns = NT;
    }
    const int tot = __syncthreads_count(j < n && __ldg(x + j) != 0.0f);
    return ns > 0 && (double)tot >= frac * (double)ns;
}

}  // namespace spmvd
}  // namespace dbs

struct dbs_spmv_plan {
    dbs::spmvd::PlanDev D{};
    int device = -1;
    int grid = 0;
    uint32_t nplan = 0;
    size_t max_chunks = 0, max_split = 0;   // split-row scratch sizes (partial sums, counters)
};
