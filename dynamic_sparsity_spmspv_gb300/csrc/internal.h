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
    std::vector<uint32_t> csc2csr;    // B (host only)
    std::vector<U4> payload;          // P
    std::vector<U4> tiles;            // T: {p0, payload offset, rb0, span | flags | count}
    std::vector<uint16_t> rb_rows;    // nbr: rows of each row block that hold an entry (bit r = row r)
};

// Allocation-failure injection for tests (dbs_debug_fail_alloc): true when
// this allocation attempt is the one chosen to fail.
bool alloc_fault();
// cudaMalloc behind the injection hook.
template <class T>
inline cudaError_t dev_malloc(T **p, size_t bytes)
{
    if (alloc_fault()) { *p = nullptr; return cudaErrorMemoryAllocation; }
    return cudaMalloc((void **)p, bytes);
}
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

// Device-side conversion (build_gpu.cu): fills H.rb_ptr, H.blk_desc and
// H.blk_ref, allocates and encodes the payload on the device.  Sets
// *fallback (and converts nothing) when a row's columns are not ascending.
dbs_status device_convert(int64_t m, int64_t n, int64_t nnz, const int64_t *d_rp, const int32_t *d_ci,
                          const float *d_va, const dbs_build_opts &o, cudaStream_t s, HostFormat &H, int64_t *B,
                          int64_t *P, uint4 **d_payload, bool *fallback);

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
