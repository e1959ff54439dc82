// Internal structures of the dbspmspv library (not part of the C ABI).
#pragma once
#include <stdint.h>

#include <vector>

#include <cuda_runtime_api.h>

#include "../../include/dbspmspv.h"
#include "format.h"

namespace dbs {

struct alignas(8) U2 { uint32_t x, y; };
struct alignas(16) U4 { uint32_t x, y, z, w; };

// Host copy of the blocked format (kept with keep_host or host_only).
struct HostFormat {
    std::vector<uint32_t> rb_ptr;     // nbr + 1
    std::vector<U2> blk_desc;         // B: {col block, meta}
    std::vector<uint32_t> blk_ref;    // B
    std::vector<uint32_t> cb_ptr;     // nbc + 1
    std::vector<U2> csc_desc;         // B: {row block, meta}
    std::vector<uint32_t> csc_ref;    // B
    std::vector<U4> payload;          // P
    std::vector<U4> tiles;            // T: {p0, payload offset, rb0, span | flags | count}
    std::vector<uint16_t> rb_rows;    // nbr: rows of each row block that hold an entry (bit r = row r)
};

// Allocation-failure injection for tests (dbs_debug_fail_alloc): true when
// this allocation attempt is the one chosen to fail.
bool alloc_fault();
// Every device allocation of the library: cudaMalloc behind the injection
// hook, with its size recorded for dev_free and the calling thread's
// MemWatch.
cudaError_t dev_malloc_bytes(void **p, size_t bytes);
template <class T>
inline cudaError_t dev_malloc(T **p, size_t bytes)
{
    void *q = nullptr;
    const cudaError_t e = dev_malloc_bytes(&q, bytes);
    *p = static_cast<T *>(q);
    return e;
}
// Frees a dev_malloc allocation (NULL is ignored).
void dev_free(void *p);
// Live and peak device bytes allocated and freed by one thread while the
// watch is installed (a matrix build).
struct MemWatch {
    int64_t live = 0, peak = 0;
};
void mem_watch(MemWatch *w);   // NULL removes it
// A host allocation of the builder, workspace or plan: throws
// std::bad_alloc when the injection hook chooses it.
void host_alloc_point();

// Device bytes held by an SpMV plan (its queues and scratch).
int64_t spmv_plan_bytes(const dbs_spmv_plan *p);
// The SpMV of a dense-x SpMSpV call over a kept plan, with the caller's
// split-row scratch; `gated`: only if x's sampled nonzero fraction reaches
// `frac`.  Writes 3 to *path_word when it runs (may be NULL).
dbs_status spmv_launch_dense(const dbs_spmv_plan *p, float *part, uint32_t *cnt, const float *x, float *y,
                             double frac, bool gated, unsigned *path_word, cudaStream_t s);

// Pull-tile weight cap W (Section 3.3.2 segments): the option, or by
// default about 64 tiles per SM, within [16, TILE_MAX_BLOCKS].
uint32_t tile_weight_cap(const dbs_build_opts &o, uint64_t total_weight);

// The device arrays of a matrix converted on the GPU, and its counts.
struct DeviceFormat {
    uint32_t *rb_ptr = nullptr;
    U2 *blk_desc = nullptr;
    uint32_t *blk_ref = nullptr;
    uint32_t *cb_ptr = nullptr;
    U2 *csc_desc = nullptr;
    uint32_t *csc_ref = nullptr;
    U4 *payload = nullptr;
    U4 *tiles = nullptr;
    uint16_t *rb_rows = nullptr;
    int64_t B = 0, P = 0, T = 0;
    int64_t blocks_by_format[DBS_NUM_FORMATS] = {}, nnz_by_format[DBS_NUM_FORMATS] = {};
};

// Device-side conversion (build_gpu.cu) of a device CSR: every array of the
// matrix is built on the GPU, byte for byte the host builder's.  Sets
// *fallback (and converts nothing) when a row's columns are not ascending;
// invalid row pointers or columns return DBS_ERR_INVALID_ARG.
dbs_status device_convert(int64_t m, int64_t n, int64_t nnz, const int64_t *d_rp, const int32_t *d_ci,
                          const float *d_va, const dbs_build_opts &o, cudaStream_t s, DeviceFormat *F,
                          bool *fallback);

}  // namespace dbs

struct dbs_matrix {
    int64_t m = 0, n = 0, nnz = 0;
    int64_t nbr = 0, nbc = 0, B = 0, P = 0, T = 0;
    bool valued = false;
    bool on_device = false;
    int device = -1;
    // device copies (NULL when host_only)
    uint32_t *d_rb_ptr = nullptr;
    dbs::U2 *d_blk_desc = nullptr;
    uint32_t *d_blk_ref = nullptr;
    uint32_t *d_cb_ptr = nullptr;
    dbs::U2 *d_csc_desc = nullptr;
    uint32_t *d_csc_ref = nullptr;
    dbs::U4 *d_payload = nullptr;
    dbs::U4 *d_tiles = nullptr;
    uint16_t *d_rb_rows = nullptr;
    dbs::HostFormat *host = nullptr;
    // dense_spmv: a library-owned copy of the input CSR and its SpMV plan
    int64_t *d_csr_rp = nullptr;
    int32_t *d_csr_ci = nullptr;
    float *d_csr_va = nullptr;
    dbs_spmv_plan *plan = nullptr;
    dbs_matrix_info info{};
};
