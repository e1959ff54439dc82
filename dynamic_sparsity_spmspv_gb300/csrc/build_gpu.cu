// Device-side conversion of a device CSR into the blocked dual-view format
// (Section 3.2.1; the paper converts offline, Section 5.5).  Every pass runs
// on the GPU: the blocks, their formats and payloads, the payload offsets,
// the block-CSC view, the pull tiles, the per-row-block row masks and the
// storage counts.  The host only reads a few counts between passes to size
// the next allocation.  The result is byte-for-byte the host builder's.
//
// Blocks without a sort.  With the columns of every row ascending, the
// blocks of a row block are found by a 16-way merge: one warp per row block,
// lane r walks row r, each step takes the smallest column block at the
// lanes' heads and every lane consumes its run of entries in that column
// block.  A block's entries then arrive in row-major order with their
// row-major ranks from a lane prefix, and every column-ordered position
// follows from the block's per-column row masks.
//
// Block-CSC view: blocks are counted per column block, scattered into their
// column block's range with atomic cursors, and each range is then sorted
// by primary block id (one warp for ranges of up to 32 blocks, a CTA's
// bitonic sort in shared memory for longer ones, and sorted 4096-block
// chunks merged by rank for the longest), which is the stable order of the
// host's counting sort.
//
// Pull tiles: the greedy cut of Section 3.3.2 depends on where the previous
// tile ended, so the end of a tile starting at each block is computed in
// parallel first, and one CTA then follows the chain of tile starts from
// block 0 through windows of those ends staged in shared memory.
//
// Row blocks with many entries (hub rows) are split into several merge
// tasks over equal shares of the column blocks, one warp each.
//
// Device memory beyond the input CSR and the finished matrix: 4 bytes per
// block and 12 per column block, or, while the blocks are found, 4 per row
// block and 8 per merge task (one per row block plus one per 4,096 entries
// of a long one), whichever is more; plus scan partials.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "internal.h"

using namespace dbs;

namespace {

constexpr int CT = 256;                 // threads per block: 8 warps, one row block each
constexpr uint32_t NO_CB = 0xFFFFFFFFu;
constexpr unsigned FULL = 0xFFFFFFFFu;

enum : unsigned { ERR_RANGE = 1u, ERR_DUP = 2u, ERR_ORDER = 4u, ERR_PTR = 8u, ERR_INTERNAL = 16u, ERR_SIZE = 32u };

struct ConvParams {
    int64_t m, n, nnz, nbr, nbc, B, ntasks;
    const int64_t *rp;
    const int32_t *ci;
    const float *va;        // NULL: pattern only
    int th0, th1;
    double th2;
    int force_format;       // -1 automatic
    uint32_t *rb_ptr;       // block-CSR row-block pointers
    uint32_t *rb_t0;        // first merge task of each row block (counts before the scan)
    uint32_t *t_rb;         // row block of each merge task
    uint32_t *t_off;        // blocks of each merge task, then its first block (after the scan)
    uint2 *desc;            // per block {column block, meta}
    uint32_t *ref;          // per block payload offset
    uint4 *payload;
    unsigned *err;
};

// Merge tasks: a row block's blocks are found by one warp, or, for a row
// block with many entries (a hub row of a power-law graph), by several
// warps, each over an equal share of the column blocks, so no warp walks
// tens of thousands of column blocks alone.
constexpr int64_t TASK_ENTRIES = 4096;   // entries of a row block per merge task
constexpr int64_t TASK_MIN_CBS = 16;     // column blocks per task at least

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

// First position in ci[lo, hi) (ascending) whose column block is >= cb.
__device__ __forceinline__ int64_t first_at_or_after(const ConvParams &C, int64_t lo, int64_t hi, uint32_t cb)
{
    while (lo < hi) {
        const int64_t mid = lo + ((hi - lo) >> 1);
        if (((uint32_t)__ldg(C.ci + mid) >> 4) < cb) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// A lane's cursor over its row's entries in merge task t's column blocks;
// only after the rows were validated.  Sets *rb and the task's column-block
// range.
__device__ __forceinline__ RowCursor open_task(const ConvParams &C, int64_t t, int lane, int64_t *rb_out)
{
    const uint32_t rb = __ldg(C.t_rb + t);
    const uint32_t t0 = __ldg(C.rb_t0 + rb), nt = __ldg(C.rb_t0 + rb + 1) - t0, k = (uint32_t)t - t0;
    const uint32_t c_lo = (uint32_t)((uint64_t)C.nbc * k / nt), c_hi = (uint32_t)((uint64_t)C.nbc * (k + 1u) / nt);
    *rb_out = rb;
    RowCursor r{0, 0, NO_CB};
    const int64_t row = (int64_t)rb * BS + lane;
    if (lane < BS && row < C.m) {
        const int64_t a = __ldg(C.rp + row), b = __ldg(C.rp + row + 1);
        r.pos = k == 0u ? a : first_at_or_after(C, a, b, c_lo);
        r.end = k + 1u == nt ? b : first_at_or_after(C, r.pos, b, c_hi);
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

// Pass 1: validate the row pointers (before any entry is read) and the
// rows' columns (range, repeats, order); one warp per row.
__global__ void __launch_bounds__(CT) k_conv_validate(ConvParams C)
{
    if (blockIdx.x == 0 && threadIdx.x == 0 && (__ldg(C.rp) != 0 || __ldg(C.rp + C.m) != C.nnz))
        atomicOr(C.err, ERR_PTR);
    const int lane = threadIdx.x & 31;
    unsigned bad = 0;
    for (int64_t row = (int64_t)blockIdx.x * (CT / 32) + (threadIdx.x >> 5); row < C.m;
         row += (int64_t)gridDim.x * (CT / 32)) {
        const int64_t a = __ldg(C.rp + row), b = __ldg(C.rp + row + 1);
        if (a < 0 || b < a || b > C.nnz) {
            bad |= ERR_PTR;
            continue;
        }
        for (int64_t k = a + lane; k < b; k += 32) {
            const int32_t c = __ldg(C.ci + k);
            if (c < 0 || (int64_t)c >= C.n) bad |= ERR_RANGE;
            else if (k > a) {
                const int32_t p = __ldg(C.ci + k - 1);
                if (c == p) bad |= ERR_DUP;
                else if (c < p) bad |= ERR_ORDER;
            }
        }
    }
    bad = __reduce_or_sync(FULL, bad);
    if (bad && lane == 0) atomicOr(C.err, bad);
}

// Merge tasks per row block, from its entry count.
__global__ void k_task_counts(ConvParams C)
{
    for (int64_t rb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; rb < C.nbr; rb += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = __ldg(C.rp + min(C.m, (rb + 1) * BS)) - __ldg(C.rp + rb * BS);
        const int64_t cap = max((int64_t)1, C.nbc / TASK_MIN_CBS);
        C.rb_t0[rb] = (uint32_t)min(cap, max((int64_t)1, (e + TASK_ENTRIES - 1) / TASK_ENTRIES));
    }
}

__global__ void k_task_fill(ConvParams C)
{
    for (int64_t rb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; rb < C.nbr; rb += (int64_t)gridDim.x * blockDim.x)
        for (uint32_t t = C.rb_t0[rb]; t < C.rb_t0[rb + 1]; ++t) C.t_rb[t] = (uint32_t)rb;
}

// Pass 2: blocks of every merge task.
__global__ void __launch_bounds__(CT) k_conv_count(ConvParams C)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (CT / 32) + (threadIdx.x >> 5);
    if (t >= C.ntasks) return;
    int64_t rb;
    RowCursor r = open_task(C, t, lane, &rb);
    uint32_t nb = 0;
    for (;;) {
        int64_t s;
        uint32_t cnt;
        if (merge_step(C, r, &s, &cnt) == NO_CB) break;
        ++nb;
    }
    if (lane == 0) C.t_off[t] = nb;
}

// Row-block pointers from the tasks' first blocks.
__global__ void k_rb_ptr_from_tasks(ConvParams C)
{
    for (int64_t rb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; rb <= C.nbr; rb += (int64_t)gridDim.x * blockDim.x)
        C.rb_ptr[rb] = rb < C.nbr ? C.t_off[C.rb_t0[rb]] : (uint32_t)C.B;
}

// Statistics of the block of the current merge step, on every lane.
struct BlockStats {
    uint32_t nnz, maxr, maxc, cm;   // cm: column occupancy (bit c: column c holds an entry)
    uint32_t rmask;                 // this lane's row mask (bit c: entry in column c)
    uint32_t cmask_own;             // lanes 0-15: rows holding an entry in column `lane`
    uint32_t cc_own;                // lanes 0-15: entries in column `lane`
    uint32_t rbase;                 // row-major rank of this lane's first entry
};

// The per-column fields (maxc, cmask_own, cc_own: a 16 x 16 bit transpose)
// are formed only when `cols` (warp-uniform) asks for them.
__device__ __forceinline__ BlockStats block_stats(const ConvParams &C, int64_t s, uint32_t cnt, int lane, bool cols)
{
    BlockStats b{};
    for (uint32_t i = 0; i < cnt; ++i) b.rmask |= 1u << ((uint32_t)__ldg(C.ci + s + i) & 15u);
    b.nnz = __reduce_add_sync(FULL, cnt);
    b.maxr = __reduce_max_sync(FULL, cnt);
    b.cm = __reduce_or_sync(FULL, b.rmask);
    uint32_t maxc = 0;
    if (cols) {
        for (int c = 0; c < 16; ++c) {
            const uint32_t rows = __ballot_sync(FULL, (b.rmask >> c) & 1u) & 0xFFFFu;
            maxc = max(maxc, (uint32_t)__popc(rows));
            if (lane == c) { b.cmask_own = rows; b.cc_own = __popc(rows); }
        }
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

// Pass 3: the descriptor of every block.
__global__ void __launch_bounds__(CT) k_conv_desc(ConvParams C)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (CT / 32) + (threadIdx.x >> 5);
    if (t >= C.ntasks) return;
    int64_t rb;
    RowCursor r = open_task(C, t, lane, &rb);
    uint32_t p = C.t_off[t];
    const bool valued = C.va != nullptr;
    for (;; ++p) {
        int64_t s;
        uint32_t cnt;
        const uint32_t cb = merge_step(C, r, &s, &cnt);
        if (cb == NO_CB) break;
        // the column counts matter only for the skew rule (th0 <= nnz <= th1)
        const uint32_t nnz_w = __reduce_add_sync(FULL, cnt);
        const bool skew = C.force_format < 0 && (int)nnz_w >= C.th0 && (int)nnz_w <= C.th1;
        const BlockStats b = block_stats(C, s, cnt, lane, skew);
        const uint32_t fmt = classify_dev(C, (int)b.nnz, (int)b.maxr, (int)b.maxc);
        uint32_t meta;
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
        } else {
            meta = meta_pack(b.cm, fmt, b.nnz);
        }
        if (lane == 0 && p < (uint64_t)C.B) C.desc[p] = make_uint2(cb, meta);
    }
}

// Pass 4: encode every stored block's payload at its offset (the payload
// array is zero-filled first, so padding bytes stay 0).
__global__ void __launch_bounds__(CT) k_conv_encode(ConvParams C)
{
    __shared__ uint32_t s_cp[CT / 32][16], s_cm[CT / 32][16];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * (CT / 32) + w;
    if (t >= C.ntasks) return;
    int64_t rb;
    RowCursor r = open_task(C, t, lane, &rb);
    uint32_t p = C.t_off[t];
    const bool valued = C.va != nullptr;
    for (;; ++p) {
        int64_t s;
        uint32_t cnt;
        const uint32_t cb = merge_step(C, r, &s, &cnt);
        if (cb == NO_CB) break;
        const uint2 d = C.desc[p];
        if (meta_inline(d.y)) continue;
        const uint32_t fmt = meta_fmt(d.y);
        // column masks and pointers: Dense masks, ForceCSC and patched-CSR layouts
        const BlockStats b = block_stats(C, s, cnt, lane, fmt == FMT_DENSE || fmt == FMT_FCSC || fmt == FMT_PCSR);
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

// ---------------------------------------------------------------------------
// Scans.  Three passes over tiles of SCAN_TILE items: per-tile aggregates,
// one CTA scanning the aggregates, then each tile scanned from its prefix.
// An operation supplies the element type T, identity(), combine(a, b) (a
// before b), load(i), store(i, exclusive prefix, element) and finish(total).

constexpr int SCAN_T = 256, SCAN_V = 16, SCAN_TILE = SCAN_T * SCAN_V, SCAN_W = SCAN_T / 32;

template <class T>
__device__ __forceinline__ T shfl_up_any(const T &v, int o)
{
    static_assert(sizeof(T) % 4 == 0, "32-bit words");
    T r;
    const uint32_t *a = reinterpret_cast<const uint32_t *>(&v);
    uint32_t *b = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(T) / 4); ++k) b[k] = __shfl_up_sync(FULL, a[k], o);
    return r;
}

// Exclusive scan of one value per thread over the CTA; *total gets the
// combination of all of them.  s_w holds SCAN_W values.
template <class Op>
__device__ typename Op::T block_exclusive(typename Op::T v, typename Op::T *s_w, typename Op::T *total)
{
    using T = typename Op::T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T t = shfl_up_any(inc, o);
        if (lane >= o) inc = Op::combine(t, inc);
    }
    T ex = shfl_up_any(inc, 1);
    if (lane == 0) ex = Op::identity();
    if (lane == 31) s_w[warp] = inc;
    __syncthreads();
    if (threadIdx.x == 0) {
        T run = Op::identity();
        for (int w = 0; w < SCAN_W; ++w) {
            const T t = s_w[w];
            s_w[w] = run;
            run = Op::combine(run, t);
        }
        s_w[SCAN_W] = run;
    }
    __syncthreads();
    const T res = Op::combine(s_w[warp], ex);
    *total = s_w[SCAN_W];
    __syncthreads();
    return res;
}

template <class Op>
__global__ void __launch_bounds__(SCAN_T) k_scan_reduce(Op op, int64_t n, typename Op::T *agg)
{
    using T = typename Op::T;
    __shared__ T s_w[SCAN_W + 1];
    const int64_t base = (int64_t)blockIdx.x * SCAN_TILE + (int64_t)threadIdx.x * SCAN_V;
    T a = Op::identity();
    for (int k = 0; k < SCAN_V; ++k)
        if (base + k < n) a = Op::combine(a, op.load(base + k));
    T tot;
    block_exclusive<Op>(a, s_w, &tot);
    if (threadIdx.x == 0) agg[blockIdx.x] = tot;
}

template <class Op>
__global__ void __launch_bounds__(SCAN_T) k_scan_aggs(Op op, int64_t ntiles, typename Op::T *agg)
{
    using T = typename Op::T;
    __shared__ T s_w[SCAN_W + 1];
    T carry = Op::identity();
    for (int64_t b = 0; b < ntiles; b += SCAN_T) {
        const int64_t i = b + threadIdx.x;
        const T v = i < ntiles ? agg[i] : Op::identity();
        T tot;
        const T ex = block_exclusive<Op>(v, s_w, &tot);
        if (i < ntiles) agg[i] = Op::combine(carry, ex);
        carry = Op::combine(carry, tot);
    }
    if (threadIdx.x == 0) op.finish(carry);
}

template <class Op>
__global__ void __launch_bounds__(SCAN_T) k_scan_down(Op op, int64_t n, const typename Op::T *agg)
{
    using T = typename Op::T;
    __shared__ T s_w[SCAN_W + 1];
    const int64_t base = (int64_t)blockIdx.x * SCAN_TILE + (int64_t)threadIdx.x * SCAN_V;
    T v[SCAN_V];
    T a = Op::identity();
#pragma unroll
    for (int k = 0; k < SCAN_V; ++k) {
        v[k] = base + k < n ? op.load(base + k) : Op::identity();
        a = Op::combine(a, v[k]);
    }
    T tot;
    T run = Op::combine(agg[blockIdx.x], block_exclusive<Op>(a, s_w, &tot));
#pragma unroll
    for (int k = 0; k < SCAN_V; ++k)
        if (base + k < n) {
            op.store(base + k, run, v[k]);
            run = Op::combine(run, v[k]);
        }
}

// Exclusive prefix sums of n counts in place, the total stored at a[n] and
// (64-bit) at *total; totals of 2^32 or more set ERR_SIZE.
struct CountScan {
    using T = unsigned long long;
    uint32_t *a;
    int64_t n;
    unsigned long long *total;
    unsigned *err;
    __device__ static T identity() { return 0ull; }
    __device__ static T combine(T x, T y) { return x + y; }
    __device__ T load(int64_t i) const { return a[i]; }
    __device__ void store(int64_t i, T ex, T) const { a[i] = (uint32_t)ex; }
    __device__ void finish(T t) const
    {
        *total = t;
        if (t >= (1ull << 32)) atomicOr(err, ERR_SIZE);
        a[n] = (uint32_t)t;
    }
};

// Payload offsets: block p's payload starts where block p-1's ended,
// rounded up to DENSE_ALIGN_UNITS for a valued Dense block.  The running
// end offset after a range of blocks is a function x -> f(x) of the offset
// before it, of the form x + b or align(x + a) + b; these compose in closed
// form (align(align(x + a1) + b1 + a2) = align(x + a1) + align(b1 + a2)
// since align(x + a1) is a multiple of the alignment), so the offsets are a
// scan over that composition.
struct Shift {
    uint32_t al, pad;
    unsigned long long a, b;
};
__device__ __forceinline__ unsigned long long align_units(unsigned long long x)
{
    return (x + DENSE_ALIGN_UNITS - 1) / DENSE_ALIGN_UNITS * DENSE_ALIGN_UNITS;
}
struct OffsetScan {
    using T = Shift;
    const uint2 *desc;
    uint32_t *ref;
    bool valued;
    unsigned long long *total;
    unsigned *err;
    __device__ static T identity() { return Shift{0u, 0u, 0ull, 0ull}; }
    __device__ static T combine(const T &g, const T &h)
    {
        if (!h.al) return Shift{g.al, 0u, g.a, g.b + h.b};
        if (!g.al) return Shift{1u, 0u, g.b + h.a, h.b};
        return Shift{1u, 0u, g.a, align_units(g.b + h.a) + h.b};
    }
    __device__ T load(int64_t p) const
    {
        const uint32_t meta = desc[p].y;
        const bool al = valued && !meta_inline(meta) && meta_fmt(meta) == FMT_DENSE;
        return Shift{al ? 1u : 0u, 0u, 0ull, (unsigned long long)meta_units(meta, valued)};
    }
    __device__ static unsigned long long apply0(const T &f) { return f.al ? align_units(f.a) + f.b : f.b; }
    __device__ void store(int64_t p, const T &ex, const T &e) const
    {
        unsigned long long start = apply0(ex);
        if (e.al) start = align_units(start);
        if (start + e.b >= (1ull << 32)) atomicOr(err, ERR_SIZE);
        ref[p] = (uint32_t)start;
    }
    __device__ void finish(const T &t) const
    {
        *total = apply0(t);
        if (*total >= (1ull << 32)) atomicOr(err, ERR_SIZE);
    }
};

// ---------------------------------------------------------------------------
// Block-CSC view.

// Row block holding primary block p (the largest rb with rb_ptr[rb] <= p).
__device__ __forceinline__ uint32_t row_block_of(const uint32_t *rb_ptr, int64_t nbr, uint32_t p)
{
    uint32_t lo = 0, hi = (uint32_t)nbr;
    while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) >> 1;
        if (__ldg(rb_ptr + mid) <= p) lo = mid;
        else hi = mid;
    }
    return lo;
}

constexpr uint32_t SORT_CHUNK = 4096;   // blocks sorted at once in shared memory

struct CscParams {
    int64_t nbr, nbc, B;
    const uint32_t *rb_ptr;
    const uint2 *desc;
    const uint32_t *ref;
    uint32_t *cb_ptr;       // counts, then pointers (nbc + 1)
    uint32_t *cur;          // per column block: next free position
    uint32_t *pos;          // B: primary ids in CSC order (the csc_ref array until filled)
    uint32_t *tmp;          // B: chunk-sorted ranges
    uint32_t *lists;        // [nbc] ranges over 32 blocks, [nbc] ranges over SORT_CHUNK
    unsigned *nlists;       // their counts
    uint2 *csc_desc;
    unsigned *err;
};

__global__ void k_csc_count(CscParams P)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < P.B; p += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t c = P.desc[p].x & DESC_COL_MASK;
        if (c < (uint64_t)P.nbc) atomicAdd(P.cb_ptr + c, 1u);
        else atomicOr(P.err, ERR_INTERNAL);
    }
}

__global__ void k_csc_scatter(CscParams P)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < P.B; p += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t c = P.desc[p].x & DESC_COL_MASK;
        if (c >= (uint64_t)P.nbc) continue;
        const uint32_t q = atomicAdd(P.cur + c, 1u);
        if (q < P.cb_ptr[c + 1]) P.pos[q] = (uint32_t)p;
        else atomicOr(P.err, ERR_INTERNAL);
    }
}

// One warp per column block: ranges of up to 32 blocks are ranked in place
// (ids are distinct); longer ranges are listed for the CTA sorts.
__global__ void __launch_bounds__(CT) k_csc_small(CscParams P)
{
    const int lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * (CT / 32) + (threadIdx.x >> 5);
    if (c >= P.nbc) return;
    const uint32_t s = P.cb_ptr[c], len = P.cb_ptr[c + 1] - s;
    if (len <= 1u) return;
    if (len <= 32u) {
        const uint32_t v = (uint32_t)lane < len ? P.pos[s + lane] : 0xFFFFFFFFu;
        uint32_t rank = 0;
        for (int j = 0; j < 32; ++j) {
            const uint32_t t = __shfl_sync(FULL, v, j);
            rank += ((uint32_t)j < len && t < v) ? 1u : 0u;
        }
        __syncwarp();
        if ((uint32_t)lane < len) P.pos[s + rank] = v;
        return;
    }
    if (lane == 0) {
        P.lists[atomicAdd(P.nlists, 1u)] = (uint32_t)c;
        if (len > SORT_CHUNK) P.lists[P.nbc + atomicAdd(P.nlists + 1, 1u)] = (uint32_t)c;
    }
}

// Bitonic sort, ascending, of s[0..np) (np a power of two) by the CTA.
__device__ void bitonic_sort(uint32_t *s, uint32_t np)
{
    for (uint32_t k = 2; k <= np; k <<= 1)
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t i = threadIdx.x; i < np; i += blockDim.x) {
                const uint32_t l = i ^ j;
                if (l > i) {
                    const uint32_t a = s[i], b = s[l];
                    if ((a > b) == ((i & k) == 0u)) { s[i] = b; s[l] = a; }
                }
            }
            __syncthreads();
        }
}

// One CTA per listed range: each chunk of up to SORT_CHUNK blocks sorted in
// shared memory, in place when the range is one chunk, else into tmp.
__global__ void __launch_bounds__(CT) k_csc_sort(CscParams P)
{
    __shared__ uint32_t s_v[SORT_CHUNK];
    const uint32_t nl = *P.nlists;
    for (uint32_t e = blockIdx.x; e < nl; e += gridDim.x) {
        const uint32_t c = P.lists[e];
        const uint32_t s = P.cb_ptr[c], len = P.cb_ptr[c + 1] - s;
        uint32_t *dst = len > SORT_CHUNK ? P.tmp : P.pos;
        for (uint32_t c0 = 0; c0 < len; c0 += SORT_CHUNK) {
            const uint32_t cl = min(SORT_CHUNK, len - c0);
            uint32_t np = 2;
            while (np < cl) np <<= 1;
            for (uint32_t i = threadIdx.x; i < np; i += blockDim.x)
                s_v[i] = i < cl ? P.pos[s + c0 + i] : 0xFFFFFFFFu;
            __syncthreads();
            bitonic_sort(s_v, np);
            for (uint32_t i = threadIdx.x; i < cl; i += blockDim.x) dst[s + c0 + i] = s_v[i];
            __syncthreads();
        }
    }
}

// Ranges of several chunks: an id's final rank is its rank in its own
// sorted chunk plus the count of smaller ids in each other chunk.
__global__ void __launch_bounds__(CT) k_csc_merge(CscParams P)
{
    const uint32_t nh = P.nlists[1];
    for (uint32_t e = blockIdx.x; e < nh; e += gridDim.x) {
        const uint32_t c = P.lists[P.nbc + e];
        const uint32_t s = P.cb_ptr[c], len = P.cb_ptr[c + 1] - s;
        const uint32_t nch = (len + SORT_CHUNK - 1) / SORT_CHUNK;
        for (uint32_t i = threadIdx.x; i < len; i += blockDim.x) {
            const uint32_t v = P.tmp[s + i], own = i / SORT_CHUNK;
            uint32_t rank = i - own * SORT_CHUNK;
            for (uint32_t k = 0; k < nch; ++k) {
                if (k == own) continue;
                const uint32_t *ch = P.tmp + s + k * SORT_CHUNK;
                uint32_t lo = 0, hi = min(SORT_CHUNK, len - k * SORT_CHUNK);
                while (lo < hi) {
                    const uint32_t mid = (lo + hi) >> 1;
                    if (ch[mid] < v) lo = mid + 1;
                    else hi = mid;
                }
                rank += lo;
            }
            P.pos[s + rank] = v;
        }
    }
}

// CSC position q: {row block, meta} and the payload offset of its block.
__global__ void k_csc_fill(CscParams P)
{
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < P.B; q += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t p = P.pos[q];
        if (p >= (uint64_t)P.B) {
            atomicOr(P.err, ERR_INTERNAL);
            continue;
        }
        P.csc_desc[q] = make_uint2(row_block_of(P.rb_ptr, P.nbr, p), P.desc[p].y);
        P.pos[q] = __ldg(P.ref + p);
    }
}

// Rows of each row block that hold an entry.
__global__ void k_rb_rows(const int64_t *rp, int64_t m, int64_t nbr, uint16_t *rows)
{
    for (int64_t rb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; rb < nbr; rb += (int64_t)gridDim.x * blockDim.x) {
        uint32_t bits = 0;
        for (int r = 0; r < BS; ++r) {
            const int64_t i = rb * BS + r;
            if (i < m && __ldg(rp + i + 1) > __ldg(rp + i)) bits |= 1u << r;
        }
        rows[rb] = (uint16_t)bits;
    }
}

// Blocks and entries per format, and the total tile weight.
__global__ void k_format_counts(const uint2 *desc, int64_t B, unsigned long long *out)
{
    __shared__ unsigned long long s_c[2 * DBS_NUM_FORMATS + 1];
    if (threadIdx.x < 2 * DBS_NUM_FORMATS + 1) s_c[threadIdx.x] = 0;
    __syncthreads();
    unsigned long long nb[DBS_NUM_FORMATS] = {}, nz[DBS_NUM_FORMATS] = {}, w = 0;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < B; p += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t meta = desc[p].y, f = meta_fmt(meta);
        if (f >= (uint32_t)DBS_NUM_FORMATS) continue;
        nb[f] += 1;
        nz[f] += meta_nnz(meta);
        w += fmt_weight(f);
    }
    for (int f = 0; f < DBS_NUM_FORMATS; ++f) {
        if (nb[f]) atomicAdd(s_c + f, nb[f]);
        if (nz[f]) atomicAdd(s_c + DBS_NUM_FORMATS + f, nz[f]);
    }
    if (w) atomicAdd(s_c + 2 * DBS_NUM_FORMATS, w);
    __syncthreads();
    if (threadIdx.x < 2 * DBS_NUM_FORMATS + 1 && s_c[threadIdx.x]) atomicAdd(out + threadIdx.x, s_c[threadIdx.x]);
}

// ---------------------------------------------------------------------------
// Pull tiles (Section 3.3.2 segments, generalised as in the host builder: a
// tile closes once its weight reaches W or its count reaches the block cap,
// and before a block whose row block is R or more past the tile's first).

struct TileParams {
    int64_t nbr, B;
    uint32_t W, R;
    const uint32_t *rb_ptr;
    uint2 *desc;
    const uint32_t *ref;
    uint32_t *next;         // B: end of the tile starting at each block; then the tile starts
    uint4 *tiles;
    unsigned long long *count;
    unsigned *err;
};

constexpr int NEXT_SPAN = 32 + (int)TILE_MAX_BLOCKS;   // blocks a warp's 32 starts can reach

// One warp per 32 consecutive starts: block weights over the reachable
// window, their prefix sums, and per start the first block where the weight
// reaches W (a binary search; every weight is at least 1 and W <= 256).
__global__ void __launch_bounds__(CT) k_tile_next(TileParams P)
{
    __shared__ uint32_t s_pre[CT / 32][NEXT_SPAN];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = ((int64_t)blockIdx.x * (CT / 32) + warp) * 32;
    if (base >= P.B) return;
    uint32_t *pre = s_pre[warp];
    const int64_t kmax = min((int64_t)NEXT_SPAN, P.B - base);
    constexpr int PER = NEXT_SPAN / 32;
    uint32_t loc[PER], sum = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int64_t i = (int64_t)lane * PER + k;
        loc[k] = i < kmax ? fmt_weight(meta_fmt(P.desc[base + i].y)) : 0u;
        sum += loc[k];
    }
    uint32_t inc = sum;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += t;
    }
    uint32_t run = inc - sum;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        run += loc[k];
        pre[lane * PER + k] = run;
    }
    __syncwarp();
    const int64_t p = base + lane;
    if (p >= P.B) return;
    const uint32_t target = (lane ? pre[lane - 1] : 0u) + P.W;
    uint32_t lo = (uint32_t)lane, hi = (uint32_t)kmax;
    while (lo < hi) {
        const uint32_t mid = (lo + hi) >> 1;
        if (pre[mid] >= target) hi = mid;
        else lo = mid + 1;
    }
    int64_t e = lo < (uint32_t)kmax ? base + lo + 1 : P.B;
    e = min(e, p + (int64_t)TILE_MAX_BLOCKS - (int64_t)(p & 1));
    const uint32_t rb = row_block_of(P.rb_ptr, P.nbr, (uint32_t)p);
    e = min(e, (int64_t)P.rb_ptr[min((int64_t)rb + P.R, P.nbr)]);
    e = min(e, P.B);
    P.next[p] = (uint32_t)e;
}

constexpr int CHAIN_T = 1024;
constexpr uint32_t CHAIN_WIN = 12288;   // ends staged per window (a multiple of 4: 16-byte loads)
constexpr size_t CHAIN_SMEM = 4u * CHAIN_WIN * sizeof(uint32_t);   // two windows of ends, two of starts

// One CTA: the tile starts are the chain 0 -> next[0] -> ... < B.  The ends
// are staged in shared memory in fixed windows of CHAIN_WIN blocks, two
// buffers deep: while thread 0 walks window k (a walk leaves a window at
// most 256 blocks past its end, inside the next one), the other warps stage
// window k + 1 and copy window k - 1's starts, which the walk collects in
// shared memory, to next[t] with coalesced stores (t never exceeds the
// start, so those entries were staged and read already).
__global__ void __launch_bounds__(CHAIN_T) k_tile_chain(TileParams P)
{
    extern __shared__ __align__(16) uint32_t chain_smem[];
    uint32_t *s_next[2] = {chain_smem, chain_smem + CHAIN_WIN};
    uint32_t *s_st[2] = {chain_smem + 2 * CHAIN_WIN, chain_smem + 3 * CHAIN_WIN};
    __shared__ uint32_t s_p, s_t, s_n[2], s_t0[2];
    const uint32_t nwin = (uint32_t)((P.B + CHAIN_WIN - 1) / CHAIN_WIN);
    // window k into dst: 16-byte loads, all of a thread's in flight together
    auto stage = [&](uint32_t k, uint32_t *dst, uint32_t tid0, uint32_t nthr) {
        const int64_t w0 = (int64_t)k * CHAIN_WIN, wl = min((int64_t)CHAIN_WIN, P.B - w0);
        const uint4 *src4 = reinterpret_cast<const uint4 *>(P.next + w0);
        uint4 *dst4 = reinterpret_cast<uint4 *>(dst);
        const int64_t n4 = wl >> 2;
        constexpr int U = (int)(CHAIN_WIN / 4 / (CHAIN_T - 32)) + 1;
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = (int64_t)(threadIdx.x - tid0) + (int64_t)u * nthr;
            if (i < n4) v[u] = src4[i];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = (int64_t)(threadIdx.x - tid0) + (int64_t)u * nthr;
            if (i < n4) dst4[i] = v[u];
        }
        for (int64_t i = 4 * n4 + (threadIdx.x - tid0); i < wl; i += nthr) dst[i] = P.next[w0 + i];
    };
    auto flush = [&](uint32_t buf, uint32_t tid0, uint32_t nthr) {
        for (uint32_t i = threadIdx.x - tid0; i < s_n[buf]; i += nthr) P.next[s_t0[buf] + i] = s_st[buf][i];
    };
    if (threadIdx.x == 0) { s_p = 0; s_t = 0; s_n[0] = s_n[1] = 0; s_t0[0] = s_t0[1] = 0; }
    if (nwin) stage(0, s_next[0], 0, blockDim.x);
    __syncthreads();
    uint32_t k = 0;
    for (; k < nwin; ++k) {
        const uint32_t *cur = s_next[k & 1];
        if (threadIdx.x == 0) {
            const int64_t w0 = (int64_t)k * CHAIN_WIN, w1 = min(w0 + (int64_t)CHAIN_WIN, P.B);
            uint32_t p = s_p, n = 0;
            uint32_t *st = s_st[k & 1];
            while ((int64_t)p < w1) {
                const uint32_t e = cur[p - (uint32_t)w0];
                st[n++] = p;
                if (e <= p || (int64_t)e > P.B) {
                    atomicOr(P.err, ERR_INTERNAL);
                    p = (uint32_t)P.B;
                    break;
                }
                p = e;
            }
            s_t0[k & 1] = s_t;
            s_n[k & 1] = n;
            s_t += n;
            s_p = p;
        } else if (threadIdx.x >= 32) {
            if (k + 1 < nwin) stage(k + 1, s_next[(k + 1) & 1], 32, blockDim.x - 32);
            if (k > 0) flush((k - 1) & 1, 32, blockDim.x - 32);
        }
        __syncthreads();
        if ((int64_t)s_p >= P.B) break;
    }
    // the walk ends in window k: its starts are still in shared memory
    if (nwin) flush(min(k, nwin - 1) & 1, 0, blockDim.x);
    if (threadIdx.x == 0) *P.count = s_t;
}

// One thread per tile: its kernel form, and each block's local row block.
__global__ void k_tile_build(TileParams P, uint32_t T)
{
    for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        const uint32_t p0 = P.next[t], p1 = t + 1 < T ? P.next[t + 1] : (uint32_t)P.B;
        const uint32_t nb = p1 - p0;
        if (p1 <= p0 || (int64_t)p1 > P.B || (p0 & 1u) + nb > TILE_MAX_BLOCKS) {
            atomicOr(P.err, ERR_INTERNAL);
            continue;
        }
        const uint32_t rb0 = row_block_of(P.rb_ptr, P.nbr, p0), rbl = row_block_of(P.rb_ptr, P.nbr, p1 - 1);
        const uint32_t span = rbl - rb0 + 1u;
        if (span > TILE_MAX_SPAN || (int64_t)rb0 + span > P.nbr) {
            atomicOr(P.err, ERR_INTERNAL);
            continue;
        }
        uint32_t w = span | (nb << TILE_NBLK_SHIFT);
        if (P.rb_ptr[rb0] < p0) w |= TILE_FIRST_SHARED;
        if (P.rb_ptr[rb0 + span] > p1) w |= TILE_LAST_SHARED;
        P.tiles[t] = make_uint4(p0, P.ref[p0], rb0, w);
        uint32_t rb = rb0;
        for (uint32_t p = p0; p < p1; ++p) {
            while (P.rb_ptr[rb + 1] <= p) ++rb;
            P.desc[p].x |= (rb - rb0) << DESC_LRB_SHIFT;
        }
    }
}

// Counts the host reads between passes.
struct Small {
    unsigned err;
    unsigned nlists[2];
    unsigned pad;
    unsigned long long B, P, B_csc, T;
    unsigned long long fmt[2 * DBS_NUM_FORMATS + 1];   // blocks, entries per format; total weight
};

// The device allocations of one conversion: every one not handed to the
// matrix is released when this goes out of scope.
struct Slots {
    static constexpr int N = 24;
    void *p[N] = {};
    template <class T>
    bool alloc(T **q, size_t bytes)
    {
        *q = nullptr;
        for (int i = 0; i < N; ++i)
            if (!p[i]) {
                if (dev_malloc(q, std::max<size_t>(bytes, 16)) != cudaSuccess) { cudaGetLastError(); *q = nullptr; return false; }
                p[i] = *q;
                return true;
            }
        return false;
    }
    void release(void *q)
    {
        for (int i = 0; i < N; ++i)
            if (q && p[i] == q) { dev_free(q); p[i] = nullptr; }
    }
    void keep(void *q)
    {
        for (int i = 0; i < N; ++i)
            if (q && p[i] == q) p[i] = nullptr;
    }
    ~Slots()
    {
        for (int i = 0; i < N; ++i) dev_free(p[i]);
    }
};

unsigned grid_for(int64_t n, int sms)
{
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)sms * 32));
}

template <class Op>
bool run_scan(const Op &op, int64_t n, typename Op::T *agg, cudaStream_t s)
{
    const int64_t ntiles = (n + SCAN_TILE - 1) / SCAN_TILE;
    if (ntiles) k_scan_reduce<Op><<<(unsigned)ntiles, SCAN_T, 0, s>>>(op, n, agg);
    k_scan_aggs<Op><<<1, SCAN_T, 0, s>>>(op, ntiles, agg);
    if (ntiles) k_scan_down<Op><<<(unsigned)ntiles, SCAN_T, 0, s>>>(op, n, agg);
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace

namespace dbs {

dbs_status device_convert(int64_t m, int64_t n, int64_t nnz, const int64_t *d_rp, const int32_t *d_ci,
                          const float *d_va, const dbs_build_opts &o, cudaStream_t s, DeviceFormat *F,
                          bool *fallback)
{
    *fallback = false;
    *F = DeviceFormat{};
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    const int64_t nbr = (m + BS - 1) / BS, nbc = (n + BS - 1) / BS;
    Slots S;
    Small h{};
    Small *d_small = nullptr;
    auto oom = []() { return DBS_ERR_OOM; };
    auto cuda_fail = [&]() { cudaGetLastError(); return DBS_ERR_CUDA; };
    auto read_small = [&]() {
        return cudaMemcpyAsync(&h, d_small, sizeof(Small), cudaMemcpyDeviceToHost, s) == cudaSuccess &&
               cudaStreamSynchronize(s) == cudaSuccess;
    };
    ConvParams C{};
    C.m = m; C.n = n; C.nnz = nnz; C.nbr = nbr; C.nbc = nbc;
    C.rp = d_rp; C.ci = d_ci; C.va = d_va;
    C.th0 = o.th0; C.th1 = o.th1; C.th2 = o.th2; C.force_format = o.force_format;
    const bool valued = d_va != nullptr;

    // 1. validation; merge tasks; blocks per task; block-CSR pointers
    if (!S.alloc(&d_small, sizeof(Small)) || !S.alloc(&C.rb_ptr, sizeof(uint32_t) * (size_t)(nbr + 1)) ||
        !S.alloc(&C.rb_t0, sizeof(uint32_t) * (size_t)(nbr + 1))) return oom();
    if (cudaMemsetAsync(d_small, 0, sizeof(Small), s) != cudaSuccess ||
        cudaMemsetAsync(C.rb_ptr, 0, sizeof(uint32_t) * (size_t)(nbr + 1), s) != cudaSuccess ||
        cudaMemsetAsync(C.rb_t0, 0, sizeof(uint32_t) * (size_t)(nbr + 1), s) != cudaSuccess) return cuda_fail();
    C.err = &d_small->err;
    k_conv_validate<<<(unsigned)std::max<int64_t>(1, std::min<int64_t>((m + 7) / 8, (int64_t)sms * 64)), CT, 0, s>>>(C);
    if (cudaGetLastError() != cudaSuccess || !read_small()) return cuda_fail();
    if (h.err & (ERR_PTR | ERR_RANGE | ERR_DUP)) return DBS_ERR_INVALID_ARG;
    if (h.err & ERR_ORDER) { *fallback = true; return DBS_OK; }
    // scan partials: one per tile of the scanned array
    auto agg_bytes = [](int64_t len) { return sizeof(Shift) * (size_t)((len + SCAN_TILE - 1) / SCAN_TILE + 1); };
    char *d_agg = nullptr;
    if (!S.alloc(&d_agg, agg_bytes(nbr))) return oom();
    k_task_counts<<<grid_for(nbr, sms), 256, 0, s>>>(C);
    {
        CountScan op{C.rb_t0, nbr, &d_small->T, C.err};
        if (!run_scan(op, nbr, reinterpret_cast<unsigned long long *>(d_agg), s) || !read_small()) return cuda_fail();
    }
    const int64_t ntasks = (int64_t)h.T;
    C.ntasks = ntasks;
    if (!S.alloc(&C.t_rb, sizeof(uint32_t) * (size_t)ntasks) || !S.alloc(&C.t_off, sizeof(uint32_t) * (size_t)(ntasks + 1)))
        return oom();
    if (cudaMemsetAsync(C.t_off, 0, sizeof(uint32_t) * (size_t)(ntasks + 1), s) != cudaSuccess) return cuda_fail();
    k_task_fill<<<grid_for(nbr, sms), 256, 0, s>>>(C);
    const unsigned grid_t = (unsigned)((ntasks + CT / 32 - 1) / (CT / 32));
    if (grid_t) k_conv_count<<<grid_t, CT, 0, s>>>(C);
    S.release(d_agg);
    if (!S.alloc(&d_agg, agg_bytes(ntasks))) return oom();
    {
        CountScan op{C.t_off, ntasks, &d_small->B, C.err};
        if (!run_scan(op, ntasks, reinterpret_cast<unsigned long long *>(d_agg), s) || !read_small()) return cuda_fail();
    }
    if (h.err & ERR_SIZE) return DBS_ERR_UNSUPPORTED;
    const int64_t B = (int64_t)h.B;
    C.B = B;
    k_rb_ptr_from_tasks<<<grid_for(nbr + 1, sms), 256, 0, s>>>(C);

    // 2. descriptors, storage counts and payload offsets
    if (!S.alloc(&C.desc, sizeof(uint2) * (size_t)(B + 8)) || !S.alloc(&C.ref, sizeof(uint32_t) * (size_t)(B + 8)))
        return oom();
    if (cudaMemsetAsync(C.desc, 0, sizeof(uint2) * (size_t)(B + 8), s) != cudaSuccess ||
        cudaMemsetAsync(C.ref, 0, sizeof(uint32_t) * (size_t)(B + 8), s) != cudaSuccess) return cuda_fail();
    if (grid_t) k_conv_desc<<<grid_t, CT, 0, s>>>(C);
    k_format_counts<<<grid_for(B, sms), 256, 0, s>>>(C.desc, B, d_small->fmt);
    S.release(d_agg);
    if (!S.alloc(&d_agg, agg_bytes(std::max(B, nbc)))) return oom();
    {
        OffsetScan op{C.desc, C.ref, valued, &d_small->P, C.err};
        if (!run_scan(op, B, reinterpret_cast<Shift *>(d_agg), s) || !read_small()) return cuda_fail();
    }
    if (h.err & ERR_SIZE) return DBS_ERR_UNSUPPORTED;
    const int64_t P = (int64_t)h.P;

    // 3. payload
    if (!S.alloc(&C.payload, (size_t)P * 16)) return oom();
    if (cudaMemsetAsync(C.payload, 0, std::max<size_t>((size_t)P * 16, 16), s) != cudaSuccess) return cuda_fail();
    if (grid_t) k_conv_encode<<<grid_t, CT, 0, s>>>(C);
    if (cudaGetLastError() != cudaSuccess) return cuda_fail();
    S.release(C.rb_t0);
    S.release(C.t_rb);
    S.release(C.t_off);

    // 4. block-CSC view
    CscParams Q{};
    Q.nbr = nbr; Q.nbc = nbc; Q.B = B;
    Q.rb_ptr = C.rb_ptr; Q.desc = C.desc; Q.ref = C.ref;
    Q.nlists = d_small->nlists;
    Q.err = C.err;
    if (!S.alloc(&Q.cb_ptr, sizeof(uint32_t) * (size_t)(nbc + 1)) || !S.alloc(&Q.cur, sizeof(uint32_t) * (size_t)nbc) ||
        !S.alloc(&Q.lists, sizeof(uint32_t) * 2 * (size_t)nbc) || !S.alloc(&Q.csc_desc, sizeof(uint2) * (size_t)(B + 8)) ||
        !S.alloc(&Q.pos, sizeof(uint32_t) * (size_t)(B + 8)) || !S.alloc(&Q.tmp, sizeof(uint32_t) * (size_t)B))
        return oom();
    if (cudaMemsetAsync(Q.cb_ptr, 0, sizeof(uint32_t) * (size_t)(nbc + 1), s) != cudaSuccess ||
        cudaMemsetAsync(Q.csc_desc, 0, sizeof(uint2) * (size_t)(B + 8), s) != cudaSuccess ||
        cudaMemsetAsync(Q.pos, 0, sizeof(uint32_t) * (size_t)(B + 8), s) != cudaSuccess) return cuda_fail();
    k_csc_count<<<grid_for(B, sms), 256, 0, s>>>(Q);
    {
        CountScan op{Q.cb_ptr, nbc, &d_small->B_csc, C.err};
        if (!run_scan(op, nbc, reinterpret_cast<unsigned long long *>(d_agg), s)) return cuda_fail();
    }
    if (nbc && cudaMemcpyAsync(Q.cur, Q.cb_ptr, sizeof(uint32_t) * (size_t)nbc, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return cuda_fail();
    k_csc_scatter<<<grid_for(B, sms), 256, 0, s>>>(Q);
    if (nbc) k_csc_small<<<(unsigned)((nbc + CT / 32 - 1) / (CT / 32)), CT, 0, s>>>(Q);
    k_csc_sort<<<(unsigned)sms * 4, CT, 0, s>>>(Q);
    k_csc_merge<<<(unsigned)sms * 4, CT, 0, s>>>(Q);
    k_csc_fill<<<grid_for(B, sms), 256, 0, s>>>(Q);
    if (cudaGetLastError() != cudaSuccess) return cuda_fail();
    S.release(Q.cur);
    S.release(Q.lists);

    // 5. rows holding an entry, per row block
    uint16_t *d_rows = nullptr;
    if (!S.alloc(&d_rows, sizeof(uint16_t) * (size_t)(nbr + 2))) return oom();
    if (cudaMemsetAsync(d_rows, 0, sizeof(uint16_t) * (size_t)(nbr + 2), s) != cudaSuccess) return cuda_fail();
    k_rb_rows<<<grid_for(nbr, sms), 256, 0, s>>>(d_rp, m, nbr, d_rows);
    if (cudaGetLastError() != cudaSuccess || !read_small()) return cuda_fail();
    if (h.err || h.B_csc != (unsigned long long)B) return DBS_ERR_INTERNAL;

    // 6. pull tiles
    TileParams T{};
    T.nbr = nbr; T.B = B;
    T.W = tile_weight_cap(o, h.fmt[2 * DBS_NUM_FORMATS]);
    T.R = o.tile_max_row_blocks > 0 ? (uint32_t)o.tile_max_row_blocks : TILE_MAX_SPAN;
    T.rb_ptr = C.rb_ptr; T.desc = C.desc; T.ref = C.ref;
    T.next = Q.tmp;
    T.count = &d_small->T;
    T.err = C.err;
    const int64_t warps = (B + 31) / 32;
    if (warps) k_tile_next<<<(unsigned)((warps + CT / 32 - 1) / (CT / 32)), CT, 0, s>>>(T);
    if (cudaFuncSetAttribute(k_tile_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CHAIN_SMEM) != cudaSuccess)
        return cuda_fail();
    k_tile_chain<<<1, CHAIN_T, CHAIN_SMEM, s>>>(T);
    if (cudaGetLastError() != cudaSuccess || !read_small()) return cuda_fail();
    if (h.err) return DBS_ERR_INTERNAL;
    const int64_t NT = (int64_t)h.T;
    if (!S.alloc(&T.tiles, sizeof(uint4) * (size_t)NT)) return oom();
    k_tile_build<<<grid_for(NT, sms), 256, 0, s>>>(T, (uint32_t)NT);
    if (cudaGetLastError() != cudaSuccess || !read_small()) return cuda_fail();
    if (h.err) return DBS_ERR_INTERNAL;

    // hand the matrix's arrays over; the rest is released with S
    F->rb_ptr = C.rb_ptr; F->blk_desc = reinterpret_cast<U2 *>(C.desc); F->blk_ref = C.ref;
    F->cb_ptr = Q.cb_ptr; F->csc_desc = reinterpret_cast<U2 *>(Q.csc_desc); F->csc_ref = Q.pos;
    F->payload = reinterpret_cast<U4 *>(C.payload); F->tiles = reinterpret_cast<U4 *>(T.tiles); F->rb_rows = d_rows;
    for (void *q : {(void *)C.rb_ptr, (void *)C.desc, (void *)C.ref, (void *)Q.cb_ptr, (void *)Q.csc_desc, (void *)Q.pos,
                    (void *)C.payload, (void *)T.tiles, (void *)d_rows})
        S.keep(q);
    F->B = B; F->P = P; F->T = NT;
    for (int f = 0; f < DBS_NUM_FORMATS; ++f) {
        F->blocks_by_format[f] = (int64_t)h.fmt[f];
        F->nnz_by_format[f] = (int64_t)h.fmt[DBS_NUM_FORMATS + f];
    }
    return DBS_OK;
}

}  // namespace dbs
