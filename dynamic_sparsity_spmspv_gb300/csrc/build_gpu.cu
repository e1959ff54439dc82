// Device-side conversion of a device CSR into the blocked dual-view format
// (Section 3.2.1; the paper converts offline, Section 5.5).  The
// entry-proportional work -- finding the nonzero 16x16 blocks, classifying
// them, encoding their payloads -- runs on the GPU; the block-proportional
// bookkeeping (payload offsets, block-CSC view, pull tiles) stays with the
// host builder's code, so both builders produce the same bytes.
//
// No sort.  With the columns of every row ascending, the blocks of a row
// block are found by a 16-way merge: one warp per row block, lane r walks
// row r, each step takes the smallest column block at the lanes' heads and
// every lane consumes its run of entries in that column block.  A block's
// entries then arrive in row-major order with their row-major ranks from a
// lane prefix, and every column-ordered position follows from the block's
// per-column row masks.  Device memory beyond the input and the finished
// matrix is one count per row block plus 13 bytes per block (descriptor,
// payload units, payload offset) -- no nnz-sized temporaries, unlike a
// sort-based converter.
#include <cuda_runtime.h>

#include <vector>

#include "internal.h"

using namespace dbs;

namespace {

constexpr int CT = 256;                 // threads per block: 8 warps, one row block each
constexpr uint32_t NO_CB = 0xFFFFFFFFu;
constexpr unsigned FULL = 0xFFFFFFFFu;

enum : unsigned { ERR_RANGE = 1u, ERR_DUP = 2u, ERR_ORDER = 4u };

struct ConvParams {
    int64_t m, n, nbr;
    const int64_t *rp;
    const int32_t *ci;
    const float *va;        // NULL: pattern only
    int th0, th1;
    double th2;
    int force_format;       // -1 automatic
    uint32_t *rb_count;     // blocks per row block
    const uint32_t *rb_ptr; // block-CSR row-block pointers
    uint2 *desc;            // per block {column block, meta}
    uint8_t *units;         // per block payload units
    const uint32_t *ref;    // per block payload offset
    uint4 *payload;
    unsigned *err;
};

// Section 3.2.1 classification with the host builder's fp64 operations,
// each rounded on its own (no fused multiply-add), so both builders agree.
__device__ uint32_t classify_dev(const ConvParams &C, int nnz, int maxr, int maxc)
{
    if (C.force_format >= 0) return (uint32_t)C.force_format;
    if (nnz < C.th0) return FMT_COO;
    if (nnz > C.th1) return FMT_DENSE;
    const double eps = 1e-9;
    const double d = __dadd_rn(__ddiv_rn((double)nnz, (double)BS), eps);
    const double skew_r = __ddiv_rn((double)maxr, d), skew_c = __ddiv_rn((double)maxc, d);
    if (__ddiv_rn(skew_r, skew_c) > C.th2) return FMT_FCSC;
    if (__ddiv_rn(skew_c, skew_r) > C.th2) return FMT_FCSR;
    return FMT_PCSR;
}

// The merge state of one lane (row) of a row block.
struct RowCursor {
    int64_t pos, end;
    uint32_t head;          // column block at pos, NO_CB when the row is done
};

__device__ __forceinline__ uint32_t cb_at(const ConvParams &C, const RowCursor &r)
{
    return r.pos < r.end ? (uint32_t)__ldg(C.ci + r.pos) >> 4 : NO_CB;
}

__device__ __forceinline__ RowCursor open_row(const ConvParams &C, int64_t rb, int lane)
{
    RowCursor r{0, 0, NO_CB};
    const int64_t row = rb * BS + lane;
    if (lane < BS && row < C.m) {
        r.pos = __ldg(C.rp + row);
        r.end = __ldg(C.rp + row + 1);
        r.head = cb_at(C, r);
    }
    return r;
}

__device__ __forceinline__ uint32_t warp_min(uint32_t v) { return __reduce_min_sync(FULL, v); }

// One merge step: the smallest column block at the heads (NO_CB when the row
// block is done); this lane's run of entries in it is [*s, *s + *cnt).
__device__ __forceinline__ uint32_t merge_step(const ConvParams &C, RowCursor &r, int64_t *s, uint32_t *cnt)
{
    const uint32_t mn = warp_min(r.head);
    *s = r.pos;
    *cnt = 0;
    if (mn != NO_CB && r.head == mn) {
        while (r.pos < r.end && ((uint32_t)__ldg(C.ci + r.pos) >> 4) == mn) { ++r.pos; ++*cnt; }
        r.head = cb_at(C, r);
    }
    return mn;
}

// Pass 1: validate the rows and count the blocks of every row block.
__global__ void __launch_bounds__(CT) k_conv_count(ConvParams C)
{
    const int lane = threadIdx.x & 31;
    const int64_t rb = (int64_t)blockIdx.x * (CT / 32) + (threadIdx.x >> 5);
    if (rb >= C.nbr) return;
    RowCursor r = open_row(C, rb, lane);
    unsigned bad = 0;
    for (int64_t k = r.pos; k < r.end; ++k) {
        const int32_t c = __ldg(C.ci + k);
        if (c < 0 || (int64_t)c >= C.n) bad |= ERR_RANGE;
        else if (k > r.pos) {
            const int32_t p = __ldg(C.ci + k - 1);
            if (c == p) bad |= ERR_DUP;
            else if (c < p) bad |= ERR_ORDER;
        }
    }
    bad = __reduce_or_sync(FULL, bad);
    if (bad) {
        if (lane == 0) atomicOr(C.err, bad);
        return;
    }
    uint32_t nb = 0;
    for (;;) {
        int64_t s;
        uint32_t cnt;
        if (merge_step(C, r, &s, &cnt) == NO_CB) break;
        ++nb;
    }
    if (lane == 0) C.rb_count[rb] = nb;
}

// Statistics of the block of the current merge step, on every lane.
struct BlockStats {
    uint32_t nnz, maxr, maxc, cm;   // cm: column occupancy (bit c: column c holds an entry)
    uint32_t rmask;                 // this lane's row mask (bit c: entry in column c)
    uint32_t cmask_own;             // lanes 0-15: rows holding an entry in column `lane`
    uint32_t cc_own;                // lanes 0-15: entries in column `lane`
    uint32_t rbase;                 // row-major rank of this lane's first entry
};

__device__ __forceinline__ BlockStats block_stats(const ConvParams &C, int64_t s, uint32_t cnt, int lane)
{
    BlockStats b{};
    for (uint32_t i = 0; i < cnt; ++i) b.rmask |= 1u << ((uint32_t)__ldg(C.ci + s + i) & 15u);
    b.nnz = __reduce_add_sync(FULL, cnt);
    b.maxr = __reduce_max_sync(FULL, cnt);
    b.cm = __reduce_or_sync(FULL, b.rmask);
    uint32_t maxc = 0;
    for (int c = 0; c < 16; ++c) {
        const uint32_t rows = __ballot_sync(FULL, (b.rmask >> c) & 1u) & 0xFFFFu;
        maxc = max(maxc, (uint32_t)__popc(rows));
        if (lane == c) { b.cmask_own = rows; b.cc_own = __popc(rows); }
    }
    b.maxc = maxc;
    uint32_t inc = cnt;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += t;
    }
    b.rbase = inc - cnt;
    return b;
}

// Pass 2: descriptor and payload size of every block.
__global__ void __launch_bounds__(CT) k_conv_desc(ConvParams C)
{
    const int lane = threadIdx.x & 31;
    const int64_t rb = (int64_t)blockIdx.x * (CT / 32) + (threadIdx.x >> 5);
    if (rb >= C.nbr) return;
    RowCursor r = open_row(C, rb, lane);
    uint32_t p = __ldg(C.rb_ptr + rb);
    const bool valued = C.va != nullptr;
    for (;; ++p) {
        int64_t s;
        uint32_t cnt;
        const uint32_t cb = merge_step(C, r, &s, &cnt);
        if (cb == NO_CB) break;
        const BlockStats b = block_stats(C, s, cnt, lane);
        const uint32_t fmt = classify_dev(C, (int)b.nnz, (int)b.maxr, (int)b.maxc);
        uint32_t meta, units;
        if (fmt == FMT_COO && !valued && b.nnz <= INLINE_MAX_NNZ) {
            // inline block: coordinate bytes of row-major entries 0..nnz-1,
            // unused bytes repeating entry 0
            uint32_t w = 0;
            for (uint32_t i = 0; i < cnt; ++i) {
                const uint32_t k = b.rbase + i;
                const uint32_t code = ((uint32_t)lane << 4) | ((uint32_t)__ldg(C.ci + s + i) & 15u);
                for (uint32_t j = 0; j < 3u; ++j)
                    if ((j < b.nnz ? j : 0u) == k) w |= code << (8u * j);
            }
            w = __reduce_or_sync(FULL, w);
            meta = META_INLINE | ((b.nnz - 1u) << 24) | w;
            units = 0;
        } else {
            meta = meta_pack(b.cm, fmt, b.nnz);
            units = payload_units(fmt, b.nnz, valued);
        }
        if (lane == 0) {
            C.desc[p] = make_uint2(cb, meta);
            C.units[p] = (uint8_t)units;
        }
    }
}

// Pass 3: encode every stored block's payload at its offset (the payload
// array is zero-filled first, so padding bytes stay 0).
__global__ void __launch_bounds__(CT) k_conv_encode(ConvParams C)
{
    __shared__ uint32_t s_cp[CT / 32][16], s_cm[CT / 32][16];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t rb = (int64_t)blockIdx.x * (CT / 32) + w;
    if (rb >= C.nbr) return;
    RowCursor r = open_row(C, rb, lane);
    uint32_t p = __ldg(C.rb_ptr + rb);
    const bool valued = C.va != nullptr;
    for (;; ++p) {
        int64_t s;
        uint32_t cnt;
        const uint32_t cb = merge_step(C, r, &s, &cnt);
        if (cb == NO_CB) break;
        const uint2 d = C.desc[p];
        if (meta_inline(d.y)) continue;
        const uint32_t fmt = meta_fmt(d.y);
        const BlockStats b = block_stats(C, s, cnt, lane);
        uint8_t *out = reinterpret_cast<uint8_t *>(C.payload + __ldg(C.ref + p));
        float *vals = reinterpret_cast<float *>(out + val_offset(fmt, b.nnz));
        // column pointers (exclusive prefix of the column counts) and masks
        uint32_t cinc = lane < 16 ? b.cc_own : 0u;
        for (int o = 1; o < 16; o <<= 1) {
            const uint32_t t = __shfl_up_sync(FULL, cinc, o);
            if (lane >= o) cinc += t;
        }
        if (lane < 16) {
            s_cp[w][lane] = cinc - b.cc_own;
            s_cm[w][lane] = b.cmask_own;
        }
        __syncwarp();
        const uint32_t lr = (uint32_t)lane;
        if (lane < 16) {
            if (fmt == FMT_DENSE) {
                reinterpret_cast<uint16_t *>(out + dense_mask_off(valued))[lane] = (uint16_t)b.cmask_own;
            } else if (fmt == FMT_FCSR || fmt == FMT_PCSR) {
                out[OFF_PTR + lane] = (uint8_t)b.rbase;
                reinterpret_cast<uint16_t *>(out + OFF_MASK)[lane] = (uint16_t)b.rmask;
                if (fmt == FMT_PCSR) out[OFF_PCOLPTR + lane] = (uint8_t)s_cp[w][lane];
            } else if (fmt == FMT_FCSC) {
                out[OFF_PTR + lane] = (uint8_t)s_cp[w][lane];
                reinterpret_cast<uint16_t *>(out + OFF_MASK)[lane] = (uint16_t)b.cmask_own;
            }
        }
        for (uint32_t i = 0; i < cnt; ++i) {
            const uint32_t lc = (uint32_t)__ldg(C.ci + s + i) & 15u, k = b.rbase + i;
            const float v = valued ? __ldg(C.va + s + i) : 0.0f;
            const uint32_t q = s_cp[w][lc] + __popc(s_cm[w][lc] & ((1u << lr) - 1u));   // column-ordered position
            switch (fmt) {
            case FMT_COO:
                out[k] = (uint8_t)((lr << 4) | lc);
                if (valued) vals[k] = v;
                break;
            case FMT_DENSE:
                if (valued) vals[lc * 16u + lr] = v;
                break;
            case FMT_FCSR:
                if (valued) vals[k] = v;
                break;
            case FMT_FCSC:
                if (valued) vals[q] = v;
                break;
            default:   // patched CSR
                out[OFF_RCSC + q] = (uint8_t)((lr << 4) | i);
                if (valued) vals[k] = v;
                break;
            }
        }
        __syncwarp();
    }
}

}  // namespace

namespace dbs {

// Runs the conversion on the device.  On return (DBS_OK): H.rb_ptr,
// H.blk_desc (local row blocks not yet set) and H.blk_ref are filled on the
// host, *B and *P hold the block and payload-unit counts, and *d_payload is
// a device allocation holding the encoded payload (P units).  `fallback`
// is set when a row's columns are not ascending (the host builder handles
// any order).  Validation failures return DBS_ERR_INVALID_ARG.
static dbs_status device_convert_impl(int64_t m, int64_t n, int64_t nnz, const int64_t *d_rp, const int32_t *d_ci,
                                      const float *d_va, const dbs_build_opts &o, cudaStream_t s, HostFormat &H,
                                      int64_t *B, int64_t *P, uint4 **d_payload, bool *fallback,
                                      void *(&scratch)[6]);

dbs_status device_convert(int64_t m, int64_t n, int64_t nnz, const int64_t *d_rp, const int32_t *d_ci,
                          const float *d_va, const dbs_build_opts &o, cudaStream_t s, HostFormat &H, int64_t *B,
                          int64_t *P, uint4 **d_payload, bool *fallback)
{
    // the device scratch of a conversion that a host allocation failure
    // interrupts is released here
    void *scratch[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    try {
        return device_convert_impl(m, n, nnz, d_rp, d_ci, d_va, o, s, H, B, P, d_payload, fallback, scratch);
    } catch (const std::bad_alloc &) {
        for (void *q : scratch) cudaFree(q);
        *d_payload = nullptr;
        return DBS_ERR_OOM;
    }
}

static dbs_status device_convert_impl(int64_t m, int64_t n, int64_t nnz, const int64_t *d_rp, const int32_t *d_ci,
                                      const float *d_va, const dbs_build_opts &o, cudaStream_t s, HostFormat &H,
                                      int64_t *B, int64_t *P, uint4 **d_payload, bool *fallback,
                                      void *(&scratch)[6])
{
    *fallback = false;
    *d_payload = nullptr;
    const int64_t nbr = (m + BS - 1) / BS;
    ConvParams C{};
    C.m = m; C.n = n; C.nbr = nbr;
    C.rp = d_rp; C.ci = d_ci; C.va = d_va;
    C.th0 = o.th0; C.th1 = o.th1; C.th2 = o.th2; C.force_format = o.force_format;
    uint32_t *d_count = nullptr, *d_rb_ptr = nullptr, *d_ref = nullptr;
    unsigned *d_err = nullptr;
    uint2 *d_desc = nullptr;
    uint8_t *d_units = nullptr;
    auto cleanup = [&]() {
        cudaFree(d_count); cudaFree(d_rb_ptr); cudaFree(d_ref); cudaFree(d_err); cudaFree(d_desc); cudaFree(d_units);
        for (void *&q : scratch) q = nullptr;
    };
    // what the caller frees if a host allocation throws
    auto track = [&]() {
        scratch[0] = d_count; scratch[1] = d_rb_ptr; scratch[2] = d_ref; scratch[3] = d_err; scratch[4] = d_desc;
        scratch[5] = d_units;
    };
    auto cuda_fail = [&]() { cudaGetLastError(); cleanup(); return DBS_ERR_CUDA; };
    const unsigned grid = (unsigned)((nbr + CT / 32 - 1) / (CT / 32));
    if (dev_malloc(&d_count, sizeof(uint32_t) * (size_t)(nbr + 1)) != cudaSuccess ||
        dev_malloc(&d_err, sizeof(unsigned)) != cudaSuccess) { cudaGetLastError(); cleanup(); return DBS_ERR_OOM; }
    if (cudaMemsetAsync(d_err, 0, sizeof(unsigned), s) != cudaSuccess ||
        cudaMemsetAsync(d_count, 0, sizeof(uint32_t) * (size_t)(nbr + 1), s) != cudaSuccess) return cuda_fail();
    track();
    C.rb_count = d_count;
    C.err = d_err;
    if (grid) k_conv_count<<<grid, CT, 0, s>>>(C);
    host_alloc_point();
    std::vector<uint32_t> cnt((size_t)nbr);
    unsigned err = 0;
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(&err, d_err, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        (nbr && cudaMemcpyAsync(cnt.data(), d_count, sizeof(uint32_t) * (size_t)nbr, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
        cudaStreamSynchronize(s) != cudaSuccess) return cuda_fail();
    if (err & (ERR_RANGE | ERR_DUP)) { cleanup(); return DBS_ERR_INVALID_ARG; }
    if (err & ERR_ORDER) { cleanup(); *fallback = true; return DBS_OK; }

    // block-CSR pointers
    H.rb_ptr.assign((size_t)nbr + 1, 0u);
    uint64_t tot = 0;
    for (int64_t rb = 0; rb < nbr; ++rb) {
        tot += cnt[(size_t)rb];
        if (tot >= (uint64_t(1) << 32)) { cleanup(); return DBS_ERR_UNSUPPORTED; }
        H.rb_ptr[(size_t)rb + 1] = (uint32_t)tot;
    }
    *B = (int64_t)tot;
    const size_t nB = (size_t)tot;
    if (dev_malloc(&d_rb_ptr, sizeof(uint32_t) * (size_t)(nbr + 1)) != cudaSuccess ||
        dev_malloc(&d_desc, sizeof(uint2) * (nB + 1)) != cudaSuccess ||
        dev_malloc(&d_units, nB + 16) != cudaSuccess ||
        dev_malloc(&d_ref, sizeof(uint32_t) * (nB + 1)) != cudaSuccess) { cudaGetLastError(); cleanup(); return DBS_ERR_OOM; }
    track();
    if (cudaMemcpyAsync(d_rb_ptr, H.rb_ptr.data(), sizeof(uint32_t) * (size_t)(nbr + 1), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return cuda_fail();
    C.rb_ptr = d_rb_ptr;
    C.desc = d_desc;
    C.units = d_units;
    if (grid) k_conv_desc<<<grid, CT, 0, s>>>(C);
    host_alloc_point();
    std::vector<uint8_t> units(nB);
    H.blk_desc.resize(nB);
    if (cudaGetLastError() != cudaSuccess ||
        (nB && cudaMemcpyAsync(H.blk_desc.data(), d_desc, sizeof(uint2) * nB, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
        (nB && cudaMemcpyAsync(units.data(), d_units, nB, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
        cudaStreamSynchronize(s) != cudaSuccess) return cuda_fail();

    // payload offsets, with the host builder's alignment rule
    H.blk_ref.resize(nB);
    const bool valued = d_va != nullptr;
    uint64_t pu = 0;
    for (size_t p = 0; p < nB; ++p) {
        const uint32_t meta = H.blk_desc[p].y;
        if (valued && !meta_inline(meta) && meta_fmt(meta) == FMT_DENSE)
            pu = (pu + DENSE_ALIGN_UNITS - 1) / DENSE_ALIGN_UNITS * DENSE_ALIGN_UNITS;
        H.blk_ref[p] = (uint32_t)pu;
        pu += units[p];
        if (pu >= (uint64_t(1) << 32)) { cleanup(); return DBS_ERR_UNSUPPORTED; }
    }
    *P = (int64_t)pu;
    uint4 *d_pay = nullptr;
    const size_t pay_bytes = std::max<size_t>((size_t)pu * 16, 16);
    if (dev_malloc(&d_pay, pay_bytes) != cudaSuccess) { cudaGetLastError(); cleanup(); return DBS_ERR_OOM; }
    if (cudaMemsetAsync(d_pay, 0, pay_bytes, s) != cudaSuccess ||
        (nB && cudaMemcpyAsync(d_ref, H.blk_ref.data(), sizeof(uint32_t) * nB, cudaMemcpyHostToDevice, s) != cudaSuccess)) {
        cudaFree(d_pay);
        return cuda_fail();
    }
    C.ref = d_ref;
    C.payload = d_pay;
    if (grid) k_conv_encode<<<grid, CT, 0, s>>>(C);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaFree(d_pay);
        return cuda_fail();
    }
    cleanup();
    *d_payload = d_pay;
    return DBS_OK;
}

}  // namespace dbs
