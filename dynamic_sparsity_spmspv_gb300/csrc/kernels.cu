// CUDA kernels (sm_103a) and the execution part of the C ABI: workspace,
// SpMSpV with sparse or dense x, DB-BFS, statistics, self-test.
//
// DB-SpMSpV (Cong et al., ICPP '26):
//   4.1      vector metadata on the GPU: blk_x_mask per 16-element block and
//            the nonzero-block count, joined to the SpMSpV by a grid-level
//            barrier inside one launch (no host round trip);
//   3.3.1    high-level path: push iff N_nzblk / N_blk < th3, decided on the
//            device; low-level microkernel from block type and blk_x_mask;
//   3.3.2    push: matrix-block tasks flattened over the active column blocks
//            (a warp takes 32 to 256 CSC positions, sized per call); pull:
//            load-weighted tiles of consecutive primary blocks, one warp each;
//   3.3.3    hierarchical writeback: microkernel registers / warp shuffles ->
//            shared-memory row accumulators -> global;
//   Alg. 2-4 fp32 microkernels per (block, active column) pair: Dense over a
//            column-major block (only the active columns' 64-byte runs are
//            read), ForceCSC over a column's run, ForceCSR and patched CSR
//            by row lookups; patched CSR in column mode through
//            row_idx_csc2csr with the whole warp;
//   Alg. 5   Boolean reachability with the visited mask; here one lane per
//            block computes the found-row mask with bit operations;
//   4.2      DB-BFS: the level loop runs inside one cooperative launch;
//   4.3      DB-Decoding layer: one ordinary launch, one CTA per row block.
//
// Every device-side wait is a grid barrier with a time bound; on expiry the
// kernel latches DBS_ERR_TIMEOUT in the workspace and returns.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <new>

#include "internal.h"
#include "spmv_dev.h"

using namespace dbs;

namespace {

constexpr int NT = 256;              // threads per CTA
constexpr int NW = NT / 32;          // warps per CTA
constexpr uint32_t FULL = 0xFFFFFFFFu;
constexpr uint32_t CTILE = 2 * NT;   // row blocks per compaction tile (one mask word per thread)
constexpr int BFS_LEVEL_LOG = 64;    // BFS levels whose frontier, path and time are recorded

constexpr int MAX_GRID = 4096;       // cooperative grid size cap

struct Ctrl {
    unsigned long long bar[2][16];      // grid-barrier arrival counters by launch parity, one 128-byte line each
    unsigned int err;
    unsigned int path;
    unsigned int n_blk[3];      // nonzero vector blocks (N_nzblk) of the slot's vector
    unsigned int n_vis[3];      // matrix blocks in those column blocks (push work)
    unsigned int n_act[3];      // push list length of the slot
    unsigned int n_chunk[3];    // push task count of the slot
    unsigned int tile_next[3];  // pull tiles handed out dynamically (tail of the static order)
    unsigned int bfs_levels;
    unsigned int bfs_push_levels;
    unsigned int gen;           // launches on this control block; its parity picks the barrier counter
    unsigned long long x_active;
    unsigned long long visited;
    unsigned long long hits;
    unsigned long long touched;
    unsigned long long bytes;
    unsigned long long nzblk;
    unsigned long long y_nnz;
    unsigned long long reached;
    unsigned long long t_phase[4];   // device timestamps: start, metadata done, traversal done, end
    unsigned long long lv_t[BFS_LEVEL_LOG + 1];   // BFS: start time of each level (and of the exit)
    unsigned long long lv_u[BFS_LEVEL_LOG];       // BFS: end of each level's traversal
    unsigned int lv_nz[BFS_LEVEL_LOG];            // BFS: nonzero frontier blocks per level
    unsigned int lv_nv[BFS_LEVEL_LOG];            // BFS: matrix blocks in the frontier's column blocks
    unsigned int lv_path[BFS_LEVEL_LOG];          // BFS: 1 push, 2 pull per level
};

struct KParams {
    // matrix
    int32_t m, n, nbr, nbc;
    uint32_t B, T;
    int valued;
    const uint32_t *__restrict__ rb_ptr;
    const uint2 *__restrict__ blk_desc;
    const uint32_t *__restrict__ blk_ref;
    const uint32_t *__restrict__ cb_ptr;
    const uint2 *__restrict__ csc_desc;
    const uint32_t *__restrict__ csc_ref;
    const uint4 *__restrict__ payload;
    const uint4 *__restrict__ tiles;
    const unsigned short *__restrict__ rb_rows;   // rows holding an entry, per row block
    // call
    int path_force;
    const int32_t *x_idx;
    const float *x_val;
    long long x_nnz;
    const float *x_in;        // dense x (dense mode)
    float tau;                // decoding: activation magnitude threshold
    const float *xv;          // x values read by the microkernels
    const uint32_t *uvis32;   // caller's visited mask (Boolean SpMSpV), or NULL
    int32_t *y_idx;
    float *y_val;
    long long *y_nnz;
    float *y_dense;
    long long bfs_src;
    int32_t *levels;
    // workspace
    float *x_dense;
    uint32_t *xm32;           // sparse-x masks: zero between calls
    uint32_t *dxm32;          // dense-x masks: fully rewritten by every dense call
    uint32_t *act[3];
    uint4 *chunks[3];         // push tasks {q0, q1, column block, 0}
    float *y_acc;
    uint32_t *yrm32;
    unsigned long long *ctile_flag;   // per compaction tile: epoch << 34 | state << 32 | count or prefix
    uint32_t n_ctiles;
    uint32_t *bvis32;
    uint32_t *fm32[2];
    Ctrl *ctrl;
    double th3;
    double push_frac;
    // dense_spmv matrices: whether a kept CSR SpMV plan exists, and the
    // sampled x density at which dense-x calls use it
    int has_spmv;
    double spmv_frac;
    int local_pull_min;
    int stats;
    long long timeout_ns;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned ld_cg(const unsigned *p) { return __ldcg(p); }

// 16-bit block masks packed two per 32-bit word (block b in word b >> 1).
__device__ __forceinline__ uint32_t mask16(const uint32_t *w, uint32_t b)
{
    return (__ldcg(w + (b >> 1)) >> ((b & 1u) << 4)) & 0xFFFFu;
}
// Visited rows of row block b: a 16-bit load, so a caller's mask of exactly
// ceil(m / 16) half-words is never read past its end.
__device__ __forceinline__ uint32_t vis16(const uint32_t *v, uint32_t b)
{
    return __ldcg(reinterpret_cast<const unsigned short *>(v) + b);
}
__device__ __forceinline__ uint32_t or16(uint32_t *w, uint32_t b, uint32_t bits)
{
    uint32_t sh = (b & 1u) << 4;
    return (atomicOr(w + (b >> 1), bits << sh) >> sh) & 0xFFFFu;
}

// Bounded grid barrier.  Returns false (and every caller must return) when
// the wait timed out or another block latched an error.  Every launch owns
// one of two 64-bit arrival counters (by the parity of the launch count kept
// in the control block) and clears the other one for the launch after it.
// The count lives on the device, so a launch captured once in a CUDA graph
// and replayed any number of times stays correct.  Block b's k-th barrier adds 1 to the counter
// with a release (the block's writes, ordered before it by the block-wide
// barrier, become visible first) and waits, with acquire loads, until the
// counter reaches k * gridDim.x.  Arrival is fire-and-forget, so the last
// block to arrive releases everyone after one trip to L2.
__device__ __forceinline__ void red_release_add(unsigned long long *p, unsigned long long v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__shared__ unsigned s_bar_epoch;
__shared__ unsigned s_gen;   // this launch's number (the control block's count at entry)

// Start of every kernel that uses grid_sync (all threads call it).  Every
// block reads the launch count before its first barrier arrival, and block 0
// advances it only after that barrier, so all blocks see the same number.
__device__ __forceinline__ void grid_sync_init(const KParams &P)
{
    if (threadIdx.x == 0) {
        s_bar_epoch = 0u;
        s_gen = ld_cg(&P.ctrl->gen);
        if (blockIdx.x == 0) P.ctrl->bar[(s_gen & 1u) ^ 1u][0] = 0ull;
    }
    __syncthreads();
}
// Counter slot of a sparse-x or dense-x call: launches alternate slots.
__device__ __forceinline__ int launch_slot() { return (int)(s_gen & 1u); }
// Tag of this launch for the compaction flags: 1 .. 2^30 - 1, so flags left
// zero never match.
__device__ __forceinline__ unsigned long long launch_epoch() { return s_gen % 0x3FFFFFFFu + 1u; }
__device__ bool grid_sync(const KParams &P)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        Ctrl *c = P.ctrl;
        unsigned long long *cnt = &c->bar[s_gen & 1u][0];
        const unsigned long long target = (unsigned long long)(++s_bar_epoch) * gridDim.x;
        int ok = 1;
        red_release_add(cnt, 1ull);
        if (ld_acquire64(cnt) < target) {
            const unsigned long long t0 = globaltimer();
            while (ld_acquire64(cnt) < target) {
                if (ld_cg(&c->err) != 0u) { ok = 0; break; }
                if ((long long)(globaltimer() - t0) > P.timeout_ns) {
                    atomicCAS(&c->err, 0u, (unsigned)DBS_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        if (ok && ld_cg(&c->err) != 0u) ok = 0;
        if (ok && s_bar_epoch == 1u && blockIdx.x == 0) c->gen = s_gen + 1u;
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ void latch_error(const KParams &P, unsigned code)
{
    atomicCAS(&P.ctrl->err, 0u, code);
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(FULL, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Block-wide exclusive scan of one value per thread; returns the prefix and
// stores the total in *total.  All threads must call it.
template <int NWB = NW>
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t *total)
{
    __shared__ uint32_t s_w[NWB];
    __shared__ uint32_t s_tot;
    int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = warp_incl_scan(v, lane);
    if (lane == 31) s_w[w] = inc;
    __syncthreads();
    if (w == 0) {
        uint32_t x = lane < NWB ? s_w[lane] : 0u;
        uint32_t xi = warp_incl_scan(x, lane);
        if (lane < NWB) s_w[lane] = xi - x;
        if (lane == NWB - 1) s_tot = xi;
    }
    __syncthreads();
    uint32_t r = s_w[w] + inc - v;
    *total = s_tot;
    __syncthreads();
    return r;
}

// Push task size: CSC positions per warp task, a power of two in
// [PUSH_CHUNK_MIN, PUSH_CHUNK] giving about one task per warp for `work`
// matrix blocks, so a small push still spreads over the grid and a large one
// amortises each task's fixed cost.
__device__ __forceinline__ uint32_t push_chunk(unsigned long long work)
{
    const unsigned long long target = work / ((unsigned long long)gridDim.x * NW);
    uint32_t ch = PUSH_CHUNK_MIN;
    while (ch < PUSH_CHUNK && 2ull * ch <= target) ch <<= 1;
    return ch;
}

// Push list construction (Section 3.3.2: matrix-block tasks flattened over
// the active column blocks).  Every thread of the CTA calls this together;
// thread t appends column block cb if `want`.  The CTA reserves its list
// entries and its tasks (32 CSC positions each) with one atomic per counter
// and then writes the tasks with all its threads, so a column block with
// thousands of tasks does not serialise on one thread.
struct ListStage {
    uint32_t cb[2 * NT];
    uint32_t q0[2 * NT];
    uint32_t qe[2 * NT];
    uint32_t cstart[2 * NT + 1];
    uint32_t base_a, base_c;
};

// The plus-times pull and push drains keep their (block, column) pair lists
// in the list stage's memory, which is idle once the traversal starts: up to
// 32 queued blocks x 16 columns per warp.
constexpr uint32_t PAIRS_PER_ROUND = 32 * 16;
static_assert(sizeof(ListStage) >= NW * PAIRS_PER_ROUND * sizeof(uint16_t), "pair lists must fit the list stage");

__device__ void cta_append(const KParams &P, ListStage &L, int slot, bool want0, uint32_t cb0, bool want1,
                           uint32_t cb1, uint32_t ch)
{
    const int tid = threadIdx.x;
    uint32_t s0 = 0, e0 = 0, s1 = 0, e1 = 0;
    if (want0) { s0 = __ldg(P.cb_ptr + cb0); e0 = __ldg(P.cb_ptr + cb0 + 1); }
    if (want1) { s1 = __ldg(P.cb_ptr + cb1); e1 = __ldg(P.cb_ptr + cb1 + 1); }
    const uint32_t n0 = want0 ? (e0 - s0 + ch - 1) / ch : 0u, n1 = want1 ? (e1 - s1 + ch - 1) / ch : 0u;
    uint32_t tot_a, tot_c;
    const uint32_t oa = block_excl_scan((want0 ? 1u : 0u) + (want1 ? 1u : 0u), &tot_a);
    const uint32_t oc = block_excl_scan(n0 + n1, &tot_c);
    if (tot_a == 0u) return;
    if (tid == 0) {
        L.base_a = atomicAdd(&P.ctrl->n_act[slot], tot_a);
        L.base_c = tot_c ? atomicAdd(&P.ctrl->n_chunk[slot], tot_c) : 0u;
        L.cstart[tot_a] = tot_c;
    }
    if (want0) { L.cb[oa] = cb0; L.q0[oa] = s0; L.qe[oa] = e0; L.cstart[oa] = oc; }
    if (want1) {
        const uint32_t k = oa + (want0 ? 1u : 0u);
        L.cb[k] = cb1; L.q0[k] = s1; L.qe[k] = e1; L.cstart[k] = oc + n0;
    }
    __syncthreads();
    if (want0) P.act[slot][L.base_a + oa] = cb0;
    if (want1) P.act[slot][L.base_a + oa + (want0 ? 1u : 0u)] = cb1;
    for (uint32_t t = tid; t < tot_c; t += NT) {
        uint32_t lo = 0, hi = tot_a - 1u;       // last entry whose tasks start at or before t
        while (lo < hi) {
            const uint32_t mid = (lo + hi + 1u) >> 1;
            if (L.cstart[mid] <= t) lo = mid; else hi = mid - 1u;
        }
        const uint32_t q0 = L.q0[lo] + (t - L.cstart[lo]) * ch;
        P.chunks[slot][L.base_c + t] = make_uint4(q0, min(q0 + ch, L.qe[lo]), L.cb[lo], 0u);
    }
    __syncthreads();
}

// Sum of one value per thread over the CTA, added to *dst once per CTA.
template <class T>
__device__ __forceinline__ void cta_count(T *dst, uint32_t v)
{
    uint32_t tot;
    block_excl_scan(v, &tot);
    if (threadIdx.x == 0 && tot) atomicAdd(dst, (T)tot);
}

__device__ __forceinline__ void stamp(const KParams &P, int i)
{
    if (P.stats && blockIdx.x == 0 && threadIdx.x == 0) P.ctrl->t_phase[i] = globaltimer();
}

// ------------------------------------------------------------ microkernels
// fp32 warp microkernels: the whole warp works on one block with uniform
// arguments; on return lane l (and l + 16) holds row (l & 15)'s partial sum
// and whether that row met an active entry.

struct RowOut {
    float sum;
    uint32_t touched;
};

// One 16-byte load of read-only data that asks L2 to fetch 64 bytes on a
// miss (a Dense column is one aligned 64-byte run).
__device__ __forceinline__ float4 ldg_l2_64(const float4 *p)
{
    float4 v;
    asm("ld.global.nc.L2::64B.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// x values: a generic load, because push passes the vector block cached in
// shared memory and pull passes global memory written earlier in the launch
// (never read before that point, so no stale L1 line can exist).
__device__ __forceinline__ float xval(const float *xb, uint32_t c) { return xb[c]; }

// Patched CSR in column mode (Section 3.3.3, the local push paradigm of a
// patched block with few active columns): for each active column walk its
// row_idx_csc2csr bytes (row, offset within the row) and read the value from
// the row-ordered array; two columns per step, one per 16 lanes.
__device__ __forceinline__ RowOut mk_pcsr_col(const uint8_t *__restrict__ b, uint32_t nnz, uint32_t act,
                                              const float *xb, int lane, float *wacc, uint32_t *nread)
{
    if (lane < 16) wacc[lane] = 0.0f;
    __syncwarp();
    const float *vals = reinterpret_cast<const float *>(b + val_offset(FMT_PCSR, nnz));
    uint32_t a = act, rows = 0, cnt = 0;
    const uint32_t h = lane >> 4, l = lane & 15;
    while (a) {
        uint32_t c0 = __ffs(a) - 1u;
        a &= a - 1u;
        uint32_t c1 = a ? __ffs(a) - 1u : 16u;
        if (a) a &= a - 1u;
        uint32_t c = h ? c1 : c0;
        if (c < 16u) {
            uint32_t s = __ldg(b + OFF_PCOLPTR + c);
            uint32_t e = c == 15u ? nnz : (uint32_t)__ldg(b + OFF_PCOLPTR + c + 1);
            uint32_t k = s + l;
            if (k < e) {
                uint32_t code = __ldg(b + OFF_RCSC + k);
                uint32_t row = code >> 4, off = code & 15u;
                float v = __ldg(vals + __ldg(b + OFF_PTR + row) + off) * xval(xb, c);
                atomicAdd(&wacc[row], v);
                rows |= 1u << row;
                ++cnt;
            }
        }
    }
    __syncwarp();
    rows = __reduce_or_sync(FULL, rows);
    float s = wacc[lane & 15];
    __syncwarp();
    *nread = cnt;
    return RowOut{s, (rows >> (lane & 15)) & 1u};
}

// Whether a block needs the whole-warp patched-CSR column mode.
__device__ __forceinline__ bool needs_col_mode(const KParams &P, uint32_t meta, uint32_t act)
{
    return meta_fmt(meta) == FMT_PCSR && (int)__popc(act) < P.local_pull_min;
}

// The whole-warp microkernel of a patched-CSR block in column mode (Section
// 3.3.1: chosen by the block type and its active columns); *bytes gets the
// algorithmic bytes when statistics are on.
__device__ __forceinline__ RowOut mk_heavy(const KParams &P, const uint8_t *b, uint32_t meta, uint32_t act,
                                           const float *xb, int lane, float *wacc, uint32_t *bytes)
{
    uint32_t nr = 0;
    const RowOut o = mk_pcsr_col(b, meta_nnz(meta), act, xb, lane, wacc, &nr);
    if (P.stats) *bytes = 64u + 5u * __reduce_add_sync(FULL, nr);   // structure, then a code byte + value per entry
    return o;
}

// Column-pair microkernel (plus-times; Dense, ForceCSR, ForceCSC and patched
// CSR in row mode): one lane takes one active column c of one block and
// forms the products a_rc * x_c of every row r holding an entry in column c
// (acc[r], 0 for the other rows); returns those rows.  None of a pair's loads
// depends on another, so a warp has the payload reads of 32 pairs in flight
// together instead of walking a block's active columns one after another
// (Algorithms 2-4 restated per (block, column) pair).  ADD: the products are
// added to acc instead of replacing it.
template <bool ADD = false>
__device__ __forceinline__ uint32_t pair_products(const uint8_t *__restrict__ b, uint32_t fmt, uint32_t nnz, uint32_t c,
                                                  float xc, float (&acc)[16])
{
    const float *vals = reinterpret_cast<const float *>(b + val_offset(fmt, nnz));
    uint32_t rows = 0;
    if (fmt == FMT_DENSE) {
        // column c's 16 values are one aligned 64-byte run (absent entries
        // hold 0 and are excluded by the column mask, so no 0 * inf appears)
        rows = __ldg(reinterpret_cast<const uint16_t *>(b + dense_mask_off(true)) + c);
        const float4 *v4 = reinterpret_cast<const float4 *>(vals + c * 16u);
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 t = ldg_l2_64(v4 + q);
            v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) acc[r] = (ADD ? acc[r] : 0.0f) + (((rows >> r) & 1u) ? v[r] * xc : 0.0f);
    } else if (fmt == FMT_FCSC) {
        rows = __ldg(reinterpret_cast<const uint16_t *>(b + OFF_MASK) + c);
        const uint32_t cp = __ldg(b + OFF_PTR + c);
#pragma unroll
        for (int r = 0; r < 16; ++r)
            acc[r] = (ADD ? acc[r] : 0.0f) +
                     (((rows >> r) & 1u) ? __ldg(vals + cp + __popc(rows & ((1u << r) - 1u))) * xc : 0.0f);
    } else {
        // row layouts: row_ptr u8[16] at 0, row_mask u16[16] at 16
        const uint4 *b4 = reinterpret_cast<const uint4 *>(b);
        const uint4 rp = __ldg(b4), m0 = __ldg(b4 + 1), m1 = __ldg(b4 + 2);
        const uint32_t rpw[4] = {rp.x, rp.y, rp.z, rp.w};
        const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        const uint32_t below = (1u << c) - 1u;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const uint32_t rm = (mw[r >> 1] >> ((r & 1) * 16)) & 0xFFFFu;
            const uint32_t base = (rpw[r >> 2] >> ((r & 3) * 8)) & 0xFFu;
            const bool has = (rm >> c) & 1u;
            rows |= (has ? 1u : 0u) << r;
            acc[r] = (ADD ? acc[r] : 0.0f) + (has ? __ldg(vals + base + __popc(rm & below)) * xc : 0.0f);
        }
    }
    return rows;
}

// Sum over the warp of acc[r] from the lanes with `in` set (transpose
// reduction: each step halves the rows a lane keeps and adds its partner's
// share).  Returns row (lane >> 1) & 15's total on lanes 2r and 2r + 1.
__device__ __forceinline__ float warp_rows_sum(const float (&acc)[16], bool in, int lane)
{
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
    float v8[8], v4[4], v2[2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float lo = in ? acc[j] : 0.0f, hi = in ? acc[j + 8] : 0.0f;
        v8[j] = (b4 ? hi : lo) + __shfl_xor_sync(FULL, b4 ? lo : hi, 16);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) v4[j] = (b3 ? v8[j + 4] : v8[j]) + __shfl_xor_sync(FULL, b3 ? v8[j] : v8[j + 4], 8);
#pragma unroll
    for (int j = 0; j < 2; ++j) v2[j] = (b2 ? v4[j + 2] : v4[j]) + __shfl_xor_sync(FULL, b2 ? v4[j] : v4[j + 2], 4);
    float v = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(FULL, b1 ? v2[0] : v2[1], 2);
    return v + __shfl_xor_sync(FULL, v, 1);
}

// COO block, one lane: scan the packed coordinates (Section 3.3.3).  Adds the
// products through `add(row, value)` and returns the touched-row bits.  The
// entries go in groups of four, whose value and x loads are all issued
// before any product is formed.
template <class Add>
__device__ __forceinline__ uint32_t coo_lane(const uint8_t *__restrict__ b, uint32_t nnz, uint32_t act,
                                            const float *xb, bool valued, Add add)
{
    const float *vals = reinterpret_cast<const float *>(b + val_offset(FMT_COO, nnz));
    const uint4 *c4 = reinterpret_cast<const uint4 *>(b);
    uint32_t rows = 0, cur = 16u;
    float acc = 0.0f;
    for (uint32_t base = 0; base < nnz; base += 16u) {
        const uint4 v = __ldg(c4 + (base >> 4));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (uint32_t g = 0; g < 4u; ++g) {
            if (base + 4u * g >= nnz) break;
            float av[4], xx[4];
            uint32_t hit = 0;
#pragma unroll
            for (uint32_t j = 0; j < 4u; ++j) {
                const uint32_t e = (wv[g] >> (8u * j)) & 0xFFu, idx = base + 4u * g + j;
                const bool on = idx < nnz && ((act >> (e & 15u)) & 1u);
                hit |= (on ? 1u : 0u) << j;
                av[j] = on && valued ? __ldg(vals + idx) : 0.0f;
                xx[j] = on && valued ? xval(xb, e & 15u) : 0.0f;
            }
#pragma unroll
            for (uint32_t j = 0; j < 4u; ++j) {
                if (!((hit >> j) & 1u)) continue;
                const uint32_t r = ((wv[g] >> (8u * j)) >> 4) & 15u;
                rows |= 1u << r;
                // entries are in row-major order: a row's run of products is
                // summed first and handed to `add` once
                if (valued) {
                    const float p = av[j] * xx[j];
                    if (r == cur) {
                        acc += p;
                    } else {
                        if (cur < 16u) add(cur, acc);
                        cur = r;
                        acc = p;
                    }
                }
            }
        }
    }
    if (valued && cur < 16u) add(cur, acc);
    return rows;
}

// A valued COO block of at most three entries is one 16-byte unit:
// coordinate bytes 0-2, values from byte 4.  Adds the products of its active
// entries into yr (row r of the block at yr[r]) and returns their rows.
__device__ __forceinline__ uint32_t coo_unit(uint4 u, uint32_t nnz, uint32_t act, const float *xb, float *yr)
{
    const float v[3] = {__uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)};
    uint32_t rows = 0, cur = 16u;
    float acc = 0.0f;
#pragma unroll
    for (uint32_t j = 0; j < 3u; ++j) {
        const uint32_t e = (u.x >> (8u * j)) & 0xFFu, c = e & 15u, r = e >> 4;
        if (j < nnz && ((act >> c) & 1u)) {
            rows |= 1u << r;
            // entries are in row-major order: a row's products are summed
            // first and added to y once
            const float p = v[j] * xval(xb, c);
            if (r == cur) {
                acc += p;
            } else {
                if (cur < 16u) atomicAdd(yr + cur, acc);
                cur = r;
                acc = p;
            }
        }
    }
    if (cur < 16u) atomicAdd(yr + cur, acc);
    return rows;
}

// ------------------------------------------------------------- traversal

// Per-warp state of a pull task.  Plus-times keeps per-row partial sums;
// the Boolean variant does not.
template <int SR>
struct WarpPull {
    // Queued hits with a payload.  Boolean pull (kept across tiles, up to 31
    // carried over): qe = block id, qm = meta with the active columns in
    // its low 16 bits, qr = row block.  Plus-times pull: qe = act | fmt << 16 |
    // (nnz - 1) << 19 | lrb << 27, qm = column block, qr = payload offset.
    // Push: see push_tasks.
    uint32_t qe[TILE_MAX_BLOCKS + 32];
    uint32_t qm[TILE_MAX_BLOCKS + 32];
    uint32_t qr[TILE_MAX_BLOCKS + 32];
    uint32_t rm[TILE_MAX_SPAN];       // touched (Boolean: found) rows per row block
    uint32_t nq;                      // queued COO hits, from the front
    uint32_t nq2;                     // queued hits of the other formats, from the back
    float y[SR == 0 ? TILE_MAX_SPAN * 16 : 1];   // partial row sums (plus-times)
};

struct SmemBase {
    float wacc[NW][16];
    float wx[NW][16];
    unsigned long long st[4];   // visited, hits, touched, bytes
    ListStage L;
};

template <int SR>
struct SmemT : SmemBase {
    WarpPull<SR> wp[NW];
};

// Output rows staged per round by the compaction, in the warps' pull state
// (the row index of each output entry).
template <int SR>
constexpr uint32_t STAGE_ROWS = (uint32_t)(sizeof(WarpPull<SR>) * NW / 4u) & ~31u;

extern __shared__ __align__(128) unsigned char smem_raw[];

// Statistics: a warp sums its lanes' counts and one lane adds them to the
// CTA's shared counter (all lanes of the warp must call it).
__device__ __forceinline__ void stat_add(SmemBase &S, int i, unsigned long long v)
{
    const unsigned long long w = __reduce_add_sync(FULL, (unsigned)v);
    if ((threadIdx.x & 31) == 0 && w) atomicAdd(&S.st[i], w);
}

// Bit operations on a 16-bit column mask m held twice, mm = m | m << 16: a
// right funnel shift of (mm:mm) by a coordinate byte (row << 4 | col) wraps
// at 32 and so brings bit col of m to bit 0 whatever the row's low bit is.
__device__ __forceinline__ uint32_t dup16(uint32_t m) { return m | (m << 16); }
__device__ __forceinline__ uint32_t coord_found(uint32_t mm, uint32_t s)
{
    return (__funnelshift_r(mm, mm, s) & 1u) << ((s >> 4) & 15u);
}

// Rows of an inline block (its coordinate bytes in bits 0-23 of the meta
// word) reached from the active columns.
__device__ __forceinline__ uint32_t inline_found(uint32_t meta, uint32_t mm)
{
    return coord_found(mm, meta) | coord_found(mm, meta >> 8) | coord_found(mm, meta >> 16);
}

// inline_found without the row extraction: coordinate byte s's found bit
// goes to bit ((s >> 4) & 31), i.e. row or row + 16 depending on the low bit
// of the next byte; fold16 brings the two halves together once per run.
__device__ __forceinline__ uint32_t coord_found_w(uint32_t mm, uint32_t s)
{
    return __funnelshift_l(0u, __funnelshift_r(mm, mm, s) & 1u, s >> 4);
}
__device__ __forceinline__ uint32_t inline_found_w(uint32_t meta, uint32_t mm)
{
    return coord_found_w(mm, meta) | coord_found_w(mm, meta >> 8) | coord_found_w(mm, meta >> 16);
}
__device__ __forceinline__ uint32_t fold16(uint32_t f) { return (f | (f >> 16)) & 0xFFFFu; }

// Rows of a COO block reached from its active columns: 16 coordinates per
// 16-byte unit, the first `cnt` of them valid.
__device__ __forceinline__ uint32_t coo_found16(uint4 v, uint32_t mm, uint32_t cnt)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t f = 0;
#pragma unroll
    for (uint32_t j = 0; j < 16u; ++j) {
        const uint32_t b = coord_found(mm, w[j >> 2] >> (8u * (j & 3u)));
        f |= j < cnt ? b : 0u;
    }
    return f;
}
// Rows of a stored block reached from its active columns `act` (Algorithm 5
// semantics), given the first two 16-byte units that hold its pattern (see
// bool_load); longer COO blocks read the rest.
__device__ __forceinline__ uint32_t bool_found_units(uint32_t fmt, uint32_t nnz, uint32_t act, uint4 u0, uint4 u1,
                                                     const uint4 *b4)
{
    uint32_t f = 0;
    if (fmt == FMT_COO) {
        const uint32_t mm = dup16(act);
        f = coo_found16(u0, mm, nnz);
        if (nnz > 16u) f |= coo_found16(u1, mm, nnz - 16u);
        for (uint32_t base = 32; base < nnz; base += 16u) f |= coo_found16(__ldg(b4 + (base >> 4)), mm, nnz - base);
    } else {
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        if (fmt == FMT_DENSE || fmt == FMT_FCSC) {          // column masks: OR the active columns
#pragma unroll
            for (uint32_t c = 0; c < 16; ++c)
                f |= ((act >> c) & 1u) ? (w[c >> 1] >> ((c & 1u) << 4)) & 0xFFFFu : 0u;
        } else {                                            // row masks: rows meeting an active column
#pragma unroll
            for (uint32_t r = 0; r < 16; ++r)
                f |= ((w[r >> 1] >> ((r & 1u) << 4)) & act) ? 1u << r : 0u;
        }
    }
    return f;
}
// The two units bool_found_units starts from: COO coordinates 0-31, the
// Dense column masks (32 bytes at dense_mask_off), or the Force / patched
// masks (bytes 16-47).
__device__ __forceinline__ void bool_load(const uint4 *b4, uint32_t fmt, uint32_t nnz, bool valued, uint4 &u0,
                                          uint4 &u1)
{
    const uint32_t s = fmt == FMT_COO ? 0u : fmt == FMT_DENSE ? dense_mask_off(valued) / 16u : 1u;
    u0 = __ldg(b4 + s);
    u1 = (fmt != FMT_COO || nnz > 16u) ? __ldg(b4 + s + 1) : make_uint4(0u, 0u, 0u, 0u);
}

// Plus-times drain of a pull tile's queued hits (the queue layout of
// WarpPull for plus-times): COO hits one per lane, the other formats as
// (block, active column) pairs, patched-CSR blocks in column mode by the
// whole warp.  Row sums go to the warp's row accumulators W.y / W.rm.
template <bool ST>
__device__ __forceinline__ void pt_drain(const KParams &P, SmemT<0> &S, WarpPull<0> &W, int warp, int lane,
                                         uint32_t nq, const float *xv, uint32_t &c_bytes)
{
    const uint32_t nq2 = W.nq2;
    auto q_nnz = [](uint32_t e) { return ((e >> 19) & 0xFFu) + 1u; };
    // COO hits one per lane
    for (uint32_t i = lane; i < nq; i += 32) {
        const uint32_t e = W.qe[i], lrb = e >> 27, nnz = q_nnz(e);
        float *sy = &W.y[lrb * 16u];
        const uint8_t *b = reinterpret_cast<const uint8_t *>(P.payload + W.qr[i]);
        const uint32_t rows = coo_lane(b, nnz, e & 0xFFFFu, xv + (size_t)W.qm[i] * 16u, true,
                                       [&](uint32_t r, float v) { atomicAdd(&sy[r], v); });
        if (rows) atomicOr(&W.rm[lrb], rows);
        if (ST) c_bytes += 4u + val_offset(FMT_COO, nnz) + 4u * nnz;
    }
    __syncwarp();
    // the other formats: every (block, active column) pair is one
    // lane's work, in rounds of up to 32 queued blocks; the pairs' row
    // products are summed per row block by the warp.  Patched-CSR
    // blocks in column mode take the whole-warp microkernel after.
    uint16_t *pl = reinterpret_cast<uint16_t *>(&S.L) + warp * PAIRS_PER_ROUND;
    bool any_col_mode = false;
    for (uint32_t g0 = 0; g0 < nq2; g0 += 32) {
        uint32_t act = 0;
        if (g0 + lane < nq2) {
            const uint32_t e = W.qe[TILE_MAX_BLOCKS - 1u - g0 - lane], fmt = (e >> 16) & 7u;
            act = e & 0xFFFFu;
            if (fmt == FMT_PCSR && (int)__popc(act) < P.local_pull_min) { act = 0; any_col_mode = true; }
            if (ST && act) c_bytes += 4u + (fmt == FMT_DENSE ? 32u : 48u);
        }
        const uint32_t np = __popc(act), incl = warp_incl_scan(np, lane);
        const uint32_t tot = __shfl_sync(FULL, incl, 31);
        for (uint32_t o = incl - np; act; act &= act - 1u) pl[o++] = (uint16_t)((lane << 4) | (__ffs(act) - 1u));
        __syncwarp();
        for (uint32_t q0 = 0; q0 < tot; q0 += 32) {
            const bool in = q0 + lane < tot;
            float acc[16];
            uint32_t rows = 0, lrb = 0;
            if (in) {
                const uint32_t pe = pl[q0 + lane], c = pe & 15u;
                const uint32_t k = TILE_MAX_BLOCKS - 1u - g0 - (pe >> 4), e = W.qe[k], fmt = (e >> 16) & 7u;
                lrb = e >> 27;
                const float xc = xval(xv + (size_t)W.qm[k] * 16u, c);
                rows = pair_products(reinterpret_cast<const uint8_t *>(P.payload + W.qr[k]), fmt, q_nnz(e), c, xc,
                                     acc);
                if (ST) c_bytes += fmt == FMT_DENSE ? 64u : 4u * __popc(rows);
            } else {
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = 0.0f;
            }
            // one row block at a time (a tile's pairs mostly share one)
            for (uint32_t pend = __ballot_sync(FULL, in); pend;) {
                const uint32_t g = __shfl_sync(FULL, lrb, __ffs(pend) - 1);
                const bool mine = in && lrb == g;
                pend &= ~__ballot_sync(FULL, mine);
                const float sum = warp_rows_sum(acc, mine, lane);
                const uint32_t bits = __reduce_or_sync(FULL, mine ? rows : 0u), r = (lane >> 1) & 15u;
                if (!(lane & 1) && ((bits >> r) & 1u)) W.y[g * 16u + r] += sum;
                if (lane == 0 && bits) W.rm[g] |= bits;
                __syncwarp();
            }
        }
    }
    if (__any_sync(FULL, any_col_mode)) {
        for (uint32_t i = 0; i < nq2; ++i) {
            const uint32_t k = TILE_MAX_BLOCKS - 1u - i;
            const uint32_t e = W.qe[k], act = e & 0xFFFFu, lj = e >> 27;
            const uint32_t meta = meta_pack(act, (e >> 16) & 7u, q_nnz(e));
            if (!needs_col_mode(P, meta, act)) continue;
            const float *xj = xv + (size_t)W.qm[k] * 16u;
            uint32_t by = 0;
            RowOut o = mk_heavy(P, reinterpret_cast<const uint8_t *>(P.payload + W.qr[k]), meta, act, xj, lane,
                                S.wacc[warp], &by);
            if (lane < 16 && o.touched) W.y[lj * 16u + lane] += o.sum;
            const uint32_t bits = __ballot_sync(FULL, lane < 16 && o.touched) & 0xFFFFu;
            if (lane == 0) {
                if (bits) W.rm[lj] |= bits;
                if (ST) c_bytes += 4u + by;
            }
            __syncwarp();
        }
    }
}

// Pull (Section 3.3.2): every warp takes tiles of consecutive primary blocks
// (load-weighted segments of at most 256 blocks and 32 row blocks) and works
// through them without block-wide synchronisation.
//   * Each lane loads the descriptors of its eight blocks (li = k*32 + lane,
//     so every load instruction of the warp reads 256 contiguous bytes), then
//     issues all eight vector-mask lookups before using any of them.
//   * Inline blocks are resolved in registers and OR-ed into the row
//     accumulators; stored blocks that meet an active column are queued with
//     their meta word.
//   * Queued hits are drained one per lane (Boolean, COO) or by the whole
//     warp (Dense / Force / patched-CSR microkernels); the payload offset of
//     a hit comes from blk_ref.
// Row results gather in the warp's shared-memory accumulators and are written
// back once per row block (Section 3.3.3).
// SR 0 = plus-times, 1 = Boolean.  DOUT: dense output y.  With a visited
// mask, tiles whose rows are all visited are skipped.
// Mask lookups go through L1: the masks are read-only between two grid
// barriers, and every barrier ends with an acquire at GPU scope, after which
// plain loads observe all writes made before the barrier (the same guarantee
// that cooperative grid synchronisation gives).
template <int SR, bool DOUT, bool ST>
__device__ void pull_tiles(const KParams &P, SmemT<SR> &S, const uint32_t *xm, const uint32_t *vis,
                           uint32_t *out_rm, int tslot)
{
    constexpr int WK = 8;                       // blocks per lane per tile
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    WarpPull<SR> &W = S.wp[warp];
    const unsigned short *xm16 = reinterpret_cast<const unsigned short *>(xm);
    const float *xv = P.xv;
    const uint32_t nwarps = gridDim.x * NW;
    // Tiles [0, T0) are taken in a static strided order; the last six
    // rounds [T0, T) are handed out one tile at a time, so warps that drew
    // cheap tiles help finish the expensive ones.
    const uint32_t rounds = P.T / nwarps;
    const uint32_t T0 = rounds > 6u ? (rounds - 6u) * nwarps : 0u;
    unsigned *ctr = &P.ctrl->tile_next[tslot];
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    auto next_tile = [&](uint32_t t) -> uint32_t {
        if (t + nwarps < T0) return t + nwarps;
        const uint32_t v = lane == 0 ? T0 + atomicAdd(ctr, 1u) : 0u;
        return __shfl_sync(FULL, v, 0);
    };

    // visited rows of a tile's row blocks (lane i: row block rb0 + i); a tile
    // whose rows are all visited is skipped before its descriptors are read
    auto settle = [&](uint32_t &tt, uint4 &tdd, uint32_t &vr) {
        while (tt < P.T) {
            vr = lane < (int)(tdd.w & TILE_SPAN_MASK) ? vis16(vis, tdd.z + lane) : 0xFFFFu;
            if (!__all_sync(FULL, vr == 0xFFFFu)) return;
            tt = next_tile(tt);
            tdd = tt < P.T ? __ldg(P.tiles + tt) : z4;
        }
    };
    auto load_desc = [&](const uint4 &tdd, uint2 (&dd)[WK]) {
#pragma unroll
        for (int k = 0; k < WK; ++k) {
            const uint32_t li = (uint32_t)(k * 32 + lane);
            dd[k] = li < (tdd.w >> TILE_NBLK_SHIFT) ? __ldcs(P.blk_desc + tdd.x + li) : make_uint2(0u, 0u);
        }
    };

    // Software pipeline over a warp's tiles: the descriptors of the next tile
    // are loaded while the current one is looked up and processed.
    uint32_t t = blockIdx.x * NW + warp;
    if (t >= T0) {                                   // straight to the dynamic tail
        const uint32_t v = lane == 0 ? T0 + atomicAdd(ctr, 1u) : 0u;
        t = __shfl_sync(FULL, v, 0);
    }
    uint4 td = t < P.T ? __ldg(P.tiles + t) : z4;
    uint32_t vrow = 0;
    if (SR == 1 && vis) settle(t, td, vrow);
    uint2 d[WK];
    load_desc(td, d);
    while (t < P.T) {
        uint32_t c_vis = 0, c_hit = 0, c_touch = 0, c_bytes = 0;   // statistics of this tile
        uint32_t t_n = next_tile(t);
        uint4 td_n = t_n < P.T ? __ldg(P.tiles + t_n) : z4;
        const uint32_t rb0 = td.z, span = td.w & TILE_SPAN_MASK, nblk = td.w >> TILE_NBLK_SHIFT;
        const uint32_t p0 = td.x, edge = td.w;   // TILE_FIRST_SHARED / TILE_LAST_SHARED
        if (lane < (int)span) W.rm[lane] = 0u;
        if (SR == 0)
            for (uint32_t i = lane; i < span * 16u; i += 32) W.y[i] = 0.0f;
        if (lane == 0) { W.nq = 0u; W.nq2 = 0u; }
        uint32_t mm[WK / 2];   // the eight column-block masks, two per register
#pragma unroll
        for (int j = 0; j < WK / 2; ++j) {
            const uint32_t l0 = (uint32_t)(2 * j * 32 + lane), l1 = l0 + 32u;
            const uint32_t a = l0 < nblk ? (uint32_t)__ldca(xm16 + (d[2 * j].x & DESC_COL_MASK)) : 0u;
            const uint32_t b = l1 < nblk ? (uint32_t)__ldca(xm16 + (d[2 * j + 1].x & DESC_COL_MASK)) : 0u;
            mm[j] = a | (b << 16);
        }
        // plus-times: every block carries a payload, and pull runs when most
        // blocks are visited, so the payload offsets go out with the mask
        // lookups (one memory round trip for both)
        uint32_t rf[SR == 0 ? WK : 1];
        if (SR == 0) {
#pragma unroll
            for (int k = 0; k < WK; ++k) {
                const uint32_t li = (uint32_t)(k * 32 + lane);
                rf[k] = li < nblk ? __ldg(P.blk_ref + p0 + li) : 0u;
            }
        }
        uint32_t vrow_n = 0;
        if (SR == 1 && vis) settle(t_n, td_n, vrow_n);
        uint2 d_n[WK];
        if (SR == 1) load_desc(td_n, d_n);   // plus-times: after the queue (fewer live registers)
        __syncwarp();
#pragma unroll
        for (int k = 0; k < WK; ++k) {
            const uint32_t li = (uint32_t)(k * 32 + lane);
            const uint32_t m = (mm[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu;   // 0 past the tile's end
            const uint32_t meta = d[k].y, lrb = d[k].x >> DESC_LRB_SHIFT;
            if (ST && m) { ++c_vis; c_touch += meta_nnz(meta); }
            // both outcomes computed, one kept: no divergent branch per block
            const bool inl = SR == 1 && meta_inline(meta);
            if (SR == 1) {
                const uint32_t f = inl ? inline_found(meta, dup16(m)) : 0u;
                if (f) {
                    atomicOr(&W.rm[lrb], f);
                    if (ST) ++c_hit;
                }
            }
            const uint32_t a = inl ? 0u : m & meta & 0xFFFFu;
            if (a) {
                // COO hits from the front of the queue, the others from the
                // back, so drain rounds run one decoder each
                const uint32_t fmt = meta_fmt(meta);
                const bool back = fmt != FMT_COO;
                const uint32_t slot = back ? TILE_MAX_BLOCKS - 1u - atomicAdd(&W.nq2, 1u) : atomicAdd(&W.nq, 1u);
                if (SR == 1) {
                    W.qe[slot] = li | (lrb << 8) | (a << 16);
                    W.qm[slot] = meta;
                } else {
                    W.qe[slot] = a | (fmt << 16) | ((meta_nnz(meta) - 1u) << 19) | (lrb << 27);
                    W.qm[slot] = d[k].x & DESC_COL_MASK;
                    W.qr[slot] = rf[SR == 0 ? k : 0];
                }
                if (ST) ++c_hit;
            }
        }
        if (SR == 0) load_desc(td_n, d_n);
        __syncwarp();

        // payload-carrying hits
        const uint32_t nq = W.nq;
        if constexpr (SR == 1) {
            // COO hits (front of the queue), then the mask formats (back)
            for (uint32_t i = lane; i < nq; i += 32) {
                const uint32_t e = W.qe[i], nnz = meta_nnz(W.qm[i]);
                const uint4 *b = P.payload + __ldg(P.blk_ref + p0 + (e & 0xFFu));
                const uint4 u0 = __ldg(b);
                const uint4 u1 = nnz > 16u ? __ldg(b + 1) : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t r = bool_found_units(FMT_COO, nnz, e >> 16, u0, u1, b);
                if (r) atomicOr(&W.rm[(e >> 8) & 0xFFu], r);
                if (ST) c_bytes += 4u + nnz;
            }
            const uint32_t nq2 = W.nq2;
            for (uint32_t i = lane; i < nq2; i += 32) {
                const uint32_t k = TILE_MAX_BLOCKS - 1u - i;
                const uint32_t e = W.qe[k], meta = W.qm[k];
                const uint4 *b = P.payload + __ldg(P.blk_ref + p0 + (e & 0xFFu));
                const uint32_t fmt = meta_fmt(meta), nnz = meta_nnz(meta);
                uint4 u0, u1;
                bool_load(b, fmt, nnz, P.valued != 0, u0, u1);
                const uint32_t r = bool_found_units(fmt, nnz, e >> 16, u0, u1, b);
                if (r) atomicOr(&W.rm[(e >> 8) & 0xFFu], r);
                if (ST) c_bytes += 4u + 32u;
            }
        } else {
            pt_drain<ST>(P, S, W, warp, lane, nq, xv, c_bytes);
        }
        __syncwarp();

        // write the task's row blocks back: a row block entirely inside the
        // task is stored, one shared with a neighbouring task is added
        if (SR == 1) {
            if (lane < (int)span) {
                const uint32_t f = W.rm[lane] & ~vrow;
                if (f) or16(out_rm, rb0 + lane, f);
            }
        } else {
            for (uint32_t i = lane; i < span * 16u; i += 32) {
                const uint32_t lrb = i >> 4, r = i & 15u;
                if (!((W.rm[lrb] >> r) & 1u)) continue;
                const bool partial = (lrb == 0u && (edge & TILE_FIRST_SHARED)) ||
                                     (lrb == span - 1u && (edge & TILE_LAST_SHARED));
                float *dst = DOUT ? P.y_dense : P.y_acc;
                const size_t row = (size_t)(rb0 + lrb) * 16u + r;
                if (partial) atomicAdd(dst + row, W.y[i]);
                else dst[row] = W.y[i];
            }
            if (!DOUT && lane < (int)span && W.rm[lane]) or16(out_rm, rb0 + lane, W.rm[lane]);
        }
        if (ST) {
            if (lane == 0) c_bytes += 8u * nblk + 16u;
            stat_add(S, 0, c_vis);
            stat_add(S, 1, c_hit);
            stat_add(S, 2, c_touch);
            stat_add(S, 3, c_bytes);
        }
        __syncwarp();
        t = t_n;
        td = td_n;
        vrow = vrow_n;
#pragma unroll
        for (int k = 0; k < WK; ++k) d[k] = d_n[k];
    }
}

// Boolean pull (Sections 3.3.2 and 3.3.3, Algorithm 5 semantics), the
// path of Boolean SpMSpV and of DB-BFS pull levels.  Tiles as in
// pull_tiles, but each lane handles its eight blocks with as little work per
// block as the format allows: the descriptors arrive two per 16-byte load
// (lane l takes units u0 + 32j + l of the tile, u0 the unit holding p0), all
// eight vector-mask lookups go out together, an inline block's found rows
// come from its coordinate bytes in registers, and a lane ORs them into one
// register while its blocks stay in one row block (blocks are in row-block
// order), so shared memory sees one OR per row-block change instead of one
// per found block.  Stored blocks that meet an active column are queued
// across tiles and decoded in full rounds of 32 (one block per lane); the
// lanes' found rows are combined per row block (match and reduce) and
// OR-ed into the output, since a queued block's tile has been flushed by
// then.  Visited rows are not removed from those: every consumer of a
// Boolean pull's output applies the visited mask itself.
template <bool ST>
__device__ void pull_bool(const KParams &P, SmemT<1> &S, const uint32_t *xm, const uint32_t *vis,
                          uint32_t *out_rm, int tslot)
{
    constexpr int WU = 4;                       // 16-byte descriptor units per lane per tile
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    WarpPull<1> &W = S.wp[warp];
    const unsigned short *xm16 = reinterpret_cast<const unsigned short *>(xm);
    const uint4 *desc4 = reinterpret_cast<const uint4 *>(P.blk_desc);
    const uint32_t nwarps = gridDim.x * NW;
    const uint32_t rounds = P.T / nwarps;
    const uint32_t T0 = rounds > 6u ? (rounds - 6u) * nwarps : 0u;
    unsigned *ctr = &P.ctrl->tile_next[tslot];
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    auto next_tile = [&](uint32_t t) -> uint32_t {
        if (t + nwarps < T0) return t + nwarps;
        const uint32_t v = lane == 0 ? T0 + atomicAdd(ctr, 1u) : 0u;
        return __shfl_sync(FULL, v, 0);
    };
    // visited rows of a tile's row blocks; tiles whose rows are all visited
    // are skipped before their descriptors are read
    auto settle = [&](uint32_t &tt, uint4 &tdd, uint32_t &vr) {
        while (tt < P.T) {
            vr = lane < (int)(tdd.w & TILE_SPAN_MASK) ? vis16(vis, tdd.z + lane) : 0xFFFFu;
            if (!__all_sync(FULL, vr == 0xFFFFu)) return;
            tt = next_tile(tt);
            tdd = tt < P.T ? __ldg(P.tiles + tt) : z4;
        }
    };
    // units holding at least one block of the tile (block 2u < p0 + count);
    // the descriptor array has padding past B, so a unit's second block may
    // lie one past the last block.  A unit's block outside the tile (the one
    // before an odd p0, the one after the last block) is zeroed: column
    // block 0, local row block 0, a stored block with no columns, so it
    // finds nothing and the loop needs no range test per block.
    auto load_desc = [&](const uint4 &tdd, uint4 (&dd)[WU]) {
        const uint32_t u0 = tdd.x >> 1, end = tdd.x + (tdd.w >> TILE_NBLK_SHIFT);
#pragma unroll
        for (int j = 0; j < WU; ++j) {
            const uint32_t u = u0 + (uint32_t)(j * 32 + lane);
            dd[j] = 2u * u < end ? __ldcs(desc4 + u) : z4;
            if (2u * u < tdd.x) { dd[j].x = 0u; dd[j].y = 0u; }
            if (2u * u + 1u >= end) { dd[j].z = 0u; dd[j].w = 0u; }
        }
    };
    // queued entries [0, n) decoded, one per lane, their rows combined per
    // row block across the warp and OR-ed into the output
    auto drain = [&](uint32_t n, uint32_t &c_bytes) {
        for (uint32_t i0 = 0; i0 < n; i0 += 32) {
            const uint32_t i = i0 + (uint32_t)lane;
            uint32_t r = 0, rb = 0xFFFFFFFFu;
            if (i < n) {
                const uint32_t qm = W.qm[i], fmt = meta_fmt(qm), nnz = meta_nnz(qm);
                const uint4 *b = P.payload + __ldg(P.blk_ref + W.qe[i]);
                uint4 u0, u1;
                bool_load(b, fmt, nnz, P.valued != 0, u0, u1);
                r = bool_found_units(fmt, nnz, qm & 0xFFFFu, u0, u1, b);
                rb = W.qr[i];
                if (ST) c_bytes += 4u + (fmt == FMT_COO ? nnz : 32u);
            }
            const uint32_t grp = __match_any_sync(FULL, rb);
            const uint32_t rr = __reduce_or_sync(grp, r);
            if (rr && rb != 0xFFFFFFFFu && lane == __ffs(grp) - 1) or16(out_rm, rb, rr);
        }
    };

    uint32_t t = blockIdx.x * NW + warp;
    if (t >= T0) {
        const uint32_t v = lane == 0 ? T0 + atomicAdd(ctr, 1u) : 0u;
        t = __shfl_sync(FULL, v, 0);
    }
    if (lane == 0) W.nq = 0u;
    __syncwarp();
    uint4 td = t < P.T ? __ldg(P.tiles + t) : z4;
    uint32_t vrow = 0;
    if (vis) settle(t, td, vrow);
    uint4 d[WU];
    load_desc(td, d);
    while (t < P.T) {
        uint32_t c_vis = 0, c_hit = 0, c_touch = 0, c_bytes = 0;
        uint32_t t_n = next_tile(t);
        uint4 td_n = t_n < P.T ? __ldg(P.tiles + t_n) : z4;
        const uint32_t p0 = td.x, rb0 = td.z, span = td.w & TILE_SPAN_MASK, nblk = td.w >> TILE_NBLK_SHIFT;
        // block k of this lane (k = 2j + h) is tile block li = 2 (32 j + lane) + h - (p0 & 1)
        const int lbase = 2 * lane - (int)(p0 & 1u);
        if (lane < (int)span) W.rm[lane] = 0u;
        uint32_t mp[WU];   // the eight column-block masks, two per register
#pragma unroll
        for (int j = 0; j < WU; ++j) {
            const uint32_t a = (uint32_t)__ldca(xm16 + (d[j].x & DESC_COL_MASK));
            const uint32_t b = (uint32_t)__ldca(xm16 + (d[j].z & DESC_COL_MASK));
            mp[j] = a | (b << 16);
        }
        uint32_t vrow_n = 0;
        if (vis) settle(t_n, td_n, vrow_n);
        uint4 d_n[WU];
        load_desc(td_n, d_n);
        __syncwarp();

        // acc holds found rows at row or row + 16 (inline_found_w), folded
        // when a run ends
        uint32_t acc = 0, cur = 0;
#pragma unroll
        for (int k = 0; k < 2 * WU; ++k) {
            const int li = lbase + 64 * (k >> 1) + (k & 1);
            const uint32_t dx = (k & 1) ? d[k >> 1].z : d[k >> 1].x;
            const uint32_t meta = (k & 1) ? d[k >> 1].w : d[k >> 1].y;
            // the block's column mask held twice (both 16-bit halves)
            const uint32_t mm = __byte_perm(mp[k >> 1], 0u, (k & 1) ? 0x3232u : 0x1010u), lrb = dx >> DESC_LRB_SHIFT;
            const bool inl = meta_inline(meta);
            const uint32_t f = inl ? inline_found_w(meta, mm) : 0u;
            if (lrb != cur) {
                if (acc) atomicOr(&W.rm[cur], fold16(acc));
                acc = 0u;
                cur = lrb;
            }
            acc |= f;
            const uint32_t a = inl ? 0u : mm & meta & 0xFFFFu;
            if (a) {
                const uint32_t slot = atomicAdd(&W.nq, 1u);
                W.qe[slot] = p0 + (uint32_t)li;
                W.qm[slot] = (meta & 0xFFFF0000u) | a;
                W.qr[slot] = rb0 + lrb;
            }
            if (ST) {
                const bool valid = li >= 0 && li < (int)nblk;
                if (valid && (mm & 0xFFFFu)) { ++c_vis; c_touch += meta_nnz(meta); }
                if (f || a) ++c_hit;
            }
        }
        // the lanes' last runs: one OR for the warp when they share a row block
        const uint32_t c0 = __shfl_sync(FULL, cur, 0);
        if (__all_sync(FULL, cur == c0 || acc == 0u)) {
            const uint32_t r = fold16(__reduce_or_sync(FULL, acc));
            if (lane == 0 && r) atomicOr(&W.rm[c0], r);
        } else if (acc) {
            atomicOr(&W.rm[cur], fold16(acc));
        }
        __syncwarp();

        if (lane < (int)span) {
            const uint32_t f = W.rm[lane] & ~vrow;
            if (f) or16(out_rm, rb0 + lane, f);
        }
        // stored blocks meeting an active column, in full rounds; at most 31
        // stay queued, so the next tile's 256 fit
        const uint32_t nq = W.nq;
        if (nq >= 32u) {
            const uint32_t nfull = nq & ~31u, rem = nq - nfull;
            drain(nfull, c_bytes);
            uint32_t e0 = 0, e1 = 0, e2 = 0;
            if ((uint32_t)lane < rem) { e0 = W.qe[nfull + lane]; e1 = W.qm[nfull + lane]; e2 = W.qr[nfull + lane]; }
            __syncwarp();
            if ((uint32_t)lane < rem) { W.qe[lane] = e0; W.qm[lane] = e1; W.qr[lane] = e2; }
            if (lane == 0) W.nq = rem;
        }
        if (ST) {
            if (lane == 0) c_bytes += 8u * nblk + 16u;
            stat_add(S, 0, c_vis);
            stat_add(S, 1, c_hit);
            stat_add(S, 2, c_touch);
            stat_add(S, 3, c_bytes);
        }
        __syncwarp();
        t = t_n;
        td = td_n;
        vrow = vrow_n;
#pragma unroll
        for (int j = 0; j < WU; ++j) d[j] = d_n[j];
    }
    uint32_t c_bytes = 0;
    drain(W.nq, c_bytes);
    if (ST) stat_add(S, 3, c_bytes);
    __syncwarp();
}

// Push (Section 3.3.2): warps take tasks of up to 256 consecutive CSC
// positions of one active column block; the active vector block is cached
// in shared memory (Section 3.3.3).  Each lane loads the descriptors of its
// eight positions together.  Inline blocks are resolved at once and their
// found rows OR-ed into the output mask; stored blocks meeting an active
// column are queued and drained one per lane (Boolean, COO) or by the whole
// warp (Dense / Force / patched CSR), their payload reached through csc_ref.
// Rows are written back with atomics.  Boolean found rows are not masked by
// the visited rows here: the caller masks them once afterwards (a stored
// block whose rows are all visited is skipped in the drain).
template <int SR, bool DOUT, bool ST>
__device__ void push_tasks(const KParams &P, SmemT<SR> &S, const uint32_t *xm, const uint32_t *vis,
                           uint32_t *out_rm, int cslot, uint32_t ch)
{
    constexpr int WK = PUSH_CHUNK / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    WarpPull<SR> &W = S.wp[warp];
    const uint32_t nch = ld_cg(&P.ctrl->n_chunk[cslot]);
    const uint32_t gw = blockIdx.x * NW + warp, nwarps = gridDim.x * NW;
    float *wx = S.wx[warp];
    float *y = DOUT ? P.y_dense : P.y_acc;
    uint32_t c_vis = 0, c_hit = 0, c_touch = 0, c_bytes = 0;
    // Software pipeline over a warp's tasks: the next task's descriptors are
    // loaded while the current one is processed, and the task after that is
    // fetched a round earlier still.
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    auto load_desc = [&](const uint4 &tk, uint2 (&dd)[WK]) {
#pragma unroll
        for (int k = 0; k < WK; ++k) {
            const uint32_t q = tk.x + (uint32_t)(k * 32 + lane);
            dd[k] = q < tk.y ? __ldg(P.csc_desc + q) : make_uint2(0u, 0u);
        }
    };
    uint32_t ci = gw;
    uint4 tk = ci < nch ? __ldcg(P.chunks[cslot] + ci) : z4;
    uint4 tk_n = ci + nwarps < nch ? __ldcg(P.chunks[cslot] + ci + nwarps) : z4;
    uint2 d[WK];
    load_desc(tk, d);
    for (; ci < nch; ci += nwarps) {
        const uint32_t q0 = tk.x, q1 = tk.y, c = tk.z;
        const uint4 tk_nn = ci + 2u * nwarps < nch ? __ldcg(P.chunks[cslot] + ci + 2u * nwarps) : z4;
        uint2 d_n[WK];
        load_desc(tk_n, d_n);
        const uint32_t xmb = mask16(xm, c), mm = dup16(xmb);
        if (SR == 0 && lane < 16) {
            const size_t j = (size_t)c * 16u + lane;
            wx[lane] = j < (size_t)P.n ? __ldcg(P.xv + j) : 0.0f;
        }
        if (lane == 0) { W.nq = 0u; W.nq2 = 0u; }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < WK; ++k) {
            const uint32_t ql = (uint32_t)(k * 32 + lane);
            if (q0 + ql >= q1) continue;
            const uint32_t rb = d[k].x, meta = d[k].y;
            if (ST) { ++c_vis; c_touch += meta_nnz(meta); c_bytes += 8u; }
            if (SR == 1 && meta_inline(meta)) {
                const uint32_t f = inline_found(meta, mm);
                if (f) {
                    or16(out_rm, rb, f);
                    if (ST) ++c_hit;
                }
            } else {
                const uint32_t a = meta & xmb & 0xFFFFu;
                if (a) {
                    // plus-times: COO hits from the front, the others from the back
                    const bool back = SR == 0 && meta_fmt(meta) != FMT_COO;
                    const uint32_t slot = back ? TILE_MAX_BLOCKS - 1u - atomicAdd(&W.nq2, 1u) : atomicAdd(&W.nq, 1u);
                    W.qe[slot] = ql | (a << 16);
                    W.qm[slot] = meta;
                    W.qr[slot] = rb;
                    if (ST) ++c_hit;
                }
            }
        }
        __syncwarp();
        const uint32_t nq = W.nq;
        if (SR == 1) {
            for (uint32_t i = lane; i < nq; i += 32) {
                const uint32_t e = W.qe[i], meta = W.qm[i], rb = W.qr[i];
                const uint32_t ref = __ldg(P.csc_ref + q0 + (e & 0xFFFFu));
                const uint32_t vm = vis ? vis16(vis, rb) : 0u;
                if (vm == 0xFFFFu) continue;
                const uint4 *pb = P.payload + ref;
                const uint32_t fmt = meta_fmt(meta), nnz = meta_nnz(meta);
                uint4 u0, u1;
                bool_load(pb, fmt, nnz, P.valued != 0, u0, u1);
                const uint32_t f = bool_found_units(fmt, nnz, e >> 16, u0, u1, pb) & ~vm;
                if (f) or16(out_rm, rb, f);
                if (ST) c_bytes += 4u + (fmt == FMT_COO ? nnz : 32u);
            }
        } else {
            const uint32_t nq2 = W.nq2;
            // COO hits: payload offsets of all of them first (independent
            // loads, the offset replacing the position and the active
            // columns the meta word's column mask), then one block per lane,
            // two per lane at a time with both first payload units loaded
            // before either is decoded
            for (uint32_t i = lane; i < nq; i += 32) {
                const uint32_t e = W.qe[i];
                W.qe[i] = __ldg(P.csc_ref + q0 + (e & 0xFFFFu));
                W.qm[i] = (W.qm[i] & ~0xFFFFu) | (e >> 16);
            }
            __syncwarp();
            for (uint32_t i = lane; i < nq; i += 64) {
                const bool two = i + 32u < nq;
                const uint32_t ref[2] = {W.qe[i], two ? W.qe[i + 32u] : W.qe[i]};
                const uint32_t mt[2] = {W.qm[i], two ? W.qm[i + 32u] : 0u};
                const uint32_t rbk[2] = {W.qr[i], two ? W.qr[i + 32u] : 0u};
                const uint4 u[2] = {__ldg(P.payload + ref[0]), __ldg(P.payload + ref[1])};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !two) break;
                    const uint32_t nnz = meta_nnz(mt[h]), act = mt[h] & 0xFFFFu;
                    float *yr = y + (size_t)rbk[h] * 16u;
                    const uint32_t rows =
                        nnz <= 3u ? coo_unit(u[h], nnz, act, wx, yr)
                                  : coo_lane(reinterpret_cast<const uint8_t *>(P.payload + ref[h]), nnz, act, wx, true,
                                             [&](uint32_t r, float v) { atomicAdd(yr + r, v); });
                    if (!DOUT && rows) or16(out_rm, rbk[h], rows);
                    if (ST) c_bytes += 4u + val_offset(FMT_COO, nnz) + 4u * nnz;
                }
            }
            // the other hits: payload offsets first (independent loads; the
            // offset replaces the position and the active columns replace
            // the meta word's column mask), then one block per lane, 32 at
            // a time: the lane adds up the row products of the block's
            // active columns in registers and adds each touched row to y
            // once (every block lies in its own row block).  A patched-CSR
            // block in column mode takes the whole warp after.
            for (uint32_t i = lane; i < nq2; i += 32) {
                const uint32_t k = TILE_MAX_BLOCKS - 1u - i;
                const uint32_t e = W.qe[k];
                W.qe[k] = __ldg(P.csc_ref + q0 + (e & 0xFFFFu));
                W.qm[k] = (W.qm[k] & ~0xFFFFu) | (e >> 16);
            }
            __syncwarp();
            bool any_col_mode = false;
            for (uint32_t i = lane; i < nq2; i += 32) {
                const uint32_t k = TILE_MAX_BLOCKS - 1u - i;
                const uint32_t meta = W.qm[k], act = meta & 0xFFFFu, rb = W.qr[k];
                if (needs_col_mode(P, meta, act)) { any_col_mode = true; continue; }
                const uint32_t fmt = meta_fmt(meta), nnz = meta_nnz(meta);
                const uint8_t *b = reinterpret_cast<const uint8_t *>(P.payload + W.qe[k]);
                float acc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = 0.0f;
                uint32_t rows = 0;
                for (uint32_t a = act; a; a &= a - 1u) {
                    const uint32_t c = __ffs(a) - 1u;
                    const uint32_t rc = pair_products<true>(b, fmt, nnz, c, wx[c], acc);
                    rows |= rc;
                    if (ST) c_bytes += fmt == FMT_DENSE ? 64u : 4u * __popc(rc);
                }
                float *yr = y + (size_t)rb * 16u;
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    if ((rows >> r) & 1u) atomicAdd(yr + r, acc[r]);
                if (!DOUT && rows) or16(out_rm, rb, rows);
                if (ST) c_bytes += 4u + (fmt == FMT_DENSE ? 32u : 48u);
            }
            if (__any_sync(FULL, any_col_mode)) {
                for (uint32_t i = 0; i < nq2; ++i) {
                    const uint32_t k = TILE_MAX_BLOCKS - 1u - i;
                    const uint32_t mj = W.qm[k], rj = W.qr[k];
                    if (!needs_col_mode(P, mj, mj & 0xFFFFu)) continue;
                    uint32_t by = 0;
                    RowOut o = mk_heavy(P, reinterpret_cast<const uint8_t *>(P.payload + W.qe[k]), mj, mj & 0xFFFFu, wx,
                                        lane, S.wacc[warp], &by);
                    if (lane < 16 && o.touched) atomicAdd(y + (size_t)rj * 16u + lane, o.sum);
                    const uint32_t bits = __ballot_sync(FULL, lane < 16 && o.touched) & 0xFFFFu;
                    if (lane == 0) {
                        if (!DOUT && bits) or16(out_rm, rj, bits);
                        if (ST) c_bytes += 4u + by;
                    }
                    __syncwarp();
                }
            }
        }
        __syncwarp();
        tk = tk_n;
        tk_n = tk_nn;
#pragma unroll
        for (int k = 0; k < WK; ++k) d[k] = d_n[k];
    }
    if (ST) {
        stat_add(S, 0, c_vis);
        stat_add(S, 1, c_hit);
        stat_add(S, 2, c_touch);
        stat_add(S, 3, c_bytes);
    }
}

// Section 3.3.1: push iff xb_sparsity = N_nzblk / N_blk < th3.  With
// push_frac > 0 the same decision is taken on the work each path implies:
// push visits the n_vis matrix blocks of the active column blocks, pull scans
// all B blocks, and push wins while n_vis < push_frac * B.
__device__ __forceinline__ bool choose_push(const KParams &P, uint32_t n_act, uint32_t n_vis)
{
    if (P.path_force == DBS_PATH_PUSH) return true;
    if (P.path_force == DBS_PATH_PULL) return false;
    if (P.nbc == 0 || P.B == 0) return true;
    if (P.push_frac > 0.0) return (double)n_vis < P.push_frac * (double)P.B;
    return (double)n_act / (double)P.nbc < P.th3;
}

// Blocks in column block cb (its block-CSC length).
__device__ __forceinline__ uint32_t cb_len(const KParams &P, uint32_t cb)
{
    return __ldg(P.cb_ptr + cb + 1) - __ldg(P.cb_ptr + cb);
}

__device__ __forceinline__ void stats_begin(SmemBase &S)
{
    if (threadIdx.x < 4) S.st[threadIdx.x] = 0ull;
}
__device__ __forceinline__ void stats_flush(const KParams &P, SmemBase &S)
{
    __syncthreads();
    if (P.stats && threadIdx.x == 0) {
        if (S.st[0]) atomicAdd(&P.ctrl->visited, S.st[0]);
        if (S.st[1]) atomicAdd(&P.ctrl->hits, S.st[1]);
        if (S.st[2]) atomicAdd(&P.ctrl->touched, S.st[2]);
        if (S.st[3]) atomicAdd(&P.ctrl->bytes, S.st[3]);
    }
}

__device__ __forceinline__ void reset_stats(const KParams &P)
{
    Ctrl *c = P.ctrl;
    c->x_active = 0; c->visited = 0; c->hits = 0; c->touched = 0; c->bytes = 0;
    c->nzblk = 0; c->y_nnz = 0; c->reached = 0;
    for (int i = 0; i < 4; ++i) c->t_phase[i] = 0;
}

// ------------------------------------------------------------- kernels

// One SpMSpV with a sparse x (index list + values) and a sparse output.
// Phases: metadata | [push list] | traversal | compaction counts | writes.
template <int SR, bool ST>
__global__ void __launch_bounds__(NT, 4) k_spmspv_sparse(KParams P)
{
    SmemT<SR> &S = *reinterpret_cast<SmemT<SR> *>(smem_raw);
    grid_sync_init(P);
    if (ld_cg(&P.ctrl->err) != 0u) return;
    const int tid = threadIdx.x;
    const size_t gtid = (size_t)blockIdx.x * NT + tid, gsz = (size_t)gridDim.x * NT;
    const int slot = launch_slot();
    stats_begin(S);
    if (blockIdx.x == 0 && tid == 0 && ST) reset_stats(P);
    stamp(P, 0);

    // Phase 1 (Section 4.1): scatter x and set the blk_x_mask bits.  Lanes
    // hitting the same mask word merge their bits and one of them issues the
    // atomic; a block whose half of the word was empty is new and counted.
    // Counts are added to the global total once per CTA.  When push is
    // likely (x has at most nbc / 4 entries, or push is forced) the new
    // blocks also form the push list right here, which saves a pass and a
    // grid barrier; pull ignores the list.
    const int lane = tid & 31;
    const bool early_list = P.path_force == DBS_PATH_PUSH ||
                            (P.path_force == DBS_PATH_AUTO && (unsigned long long)P.x_nnz * 4ull <= (unsigned long long)P.nbc);
    // task size of an early list, from the expected work (entries x mean blocks per column block)
    const uint32_t ch_early = push_chunk((unsigned long long)min((long long)P.x_nnz, (long long)P.nbc) *
                                         (P.nbc ? ((unsigned long long)P.B + P.nbc - 1) / P.nbc : 1ull));
    uint32_t first = 0, act_cnt = 0, work = 0;
    for (size_t base = (size_t)blockIdx.x * NT; base < (size_t)P.x_nnz; base += gsz) {
        const size_t e = base + tid;
        uint32_t j = 0;
        bool new_lo = false, new_hi = false;
        bool active = false;
        if (e < (size_t)P.x_nnz) {
            j = (uint32_t)__ldg(P.x_idx + e);
            if (j >= (uint32_t)P.n) {                 // also catches negative indices
                latch_error(P, DBS_ERR_INVALID_ARG);
            } else {
                const float v = P.x_val ? __ldg(P.x_val + e) : 1.0f;
                active = v != 0.0f;
                if (active && SR == 0) P.x_dense[j] = v;
            }
        }
        const uint32_t am = __ballot_sync(FULL, active);
        if (active) {
            ++act_cnt;
            const uint32_t word = j >> 5;
            const uint32_t peers = __match_any_sync(am, word);
            const uint32_t bits = __reduce_or_sync(peers, 1u << (j & 31u));
            if (lane == __ffs(peers) - 1) {
                const uint32_t old = atomicOr(P.xm32 + word, bits);
                new_lo = (bits & 0xFFFFu) && !(old & 0xFFFFu);
                new_hi = (bits >> 16) && !(old >> 16);
                if (new_lo) { ++first; work += cb_len(P, 2u * word); }
                if (new_hi) { ++first; work += cb_len(P, 2u * word + 1u); }
            }
        }
        if (early_list) {
            cta_append(P, S.L, slot, new_lo, 2u * (j >> 5), new_hi, 2u * (j >> 5) + 1u, ch_early);
        }
    }
    cta_count(&P.ctrl->n_blk[slot], first);
    cta_count(&P.ctrl->n_vis[slot], work);
    if (ST) cta_count(&P.ctrl->x_active, act_cnt);
    if (!grid_sync(P)) return;
    stamp(P, 1);

    // Phase 2 (Section 3.3.1): device-side path choice, then traversal.
    const uint32_t n_nz = ld_cg(&P.ctrl->n_blk[slot]);
    const bool push = choose_push(P, n_nz, ld_cg(&P.ctrl->n_vis[slot]));
    if (push) {
        const uint32_t ch = early_list ? ch_early : push_chunk(ld_cg(&P.ctrl->n_vis[slot]));
        if (!early_list) {
            // push list: each nonzero vector block is appended by the x entry
            // holding its lowest set mask bit (indices are unique)
            for (size_t base = (size_t)blockIdx.x * NT; base < (size_t)P.x_nnz; base += gsz) {
                const size_t e = base + tid;
                bool want = false;
                uint32_t j = 0;
                if (e < (size_t)P.x_nnz) {
                    j = (uint32_t)__ldg(P.x_idx + e);
                    if (j < (uint32_t)P.n) {
                        const uint32_t mb = mask16(P.xm32, j >> 4);
                        want = (mb & (0u - mb)) == (1u << (j & 15u));
                    }
                }
                cta_append(P, S.L, slot, want, j >> 4, false, 0u, ch);
            }
            if (!grid_sync(P)) return;
        }
        push_tasks<SR, false, ST>(P, S, P.xm32, P.uvis32, P.yrm32, slot, ch);
    } else {
        if constexpr (SR == 1) pull_bool<ST>(P, S, P.xm32, P.uvis32, P.yrm32, slot);
        else pull_tiles<0, false, ST>(P, S, P.xm32, nullptr, P.yrm32, slot);
    }
    stats_flush(P, S);
    if (!grid_sync(P)) return;
    stamp(P, 2);

    // Phase 3: clear x, reset counters, compact the output.
    for (size_t e = gtid; e < (size_t)P.x_nnz; e += gsz) {
        const uint32_t j = (uint32_t)__ldg(P.x_idx + e);
        if (j >= (uint32_t)P.n) continue;
        if (SR == 0) P.x_dense[j] = 0.0f;
        P.xm32[j >> 5] = 0u;
    }
    // Rows found by push may include visited ones: the caller's mask is
    // applied here, per word of two row blocks.
    auto unvisited = [&](size_t w) -> uint32_t {
        if (SR != 1 || !P.uvis32) return FULL;
        const uint32_t lo = 2u * w < (size_t)P.nbr ? vis16(P.uvis32, (uint32_t)(2u * w)) : 0u;
        const uint32_t hi = 2u * w + 1u < (size_t)P.nbr ? vis16(P.uvis32, (uint32_t)(2u * w + 1u)) : 0u;
        return ~(lo | (hi << 16));
    };
    if (blockIdx.x == 0 && tid == 0) {
        Ctrl *c = P.ctrl;
        c->path = push ? 1u : 2u;
        if (ST) c->nzblk = n_nz;
        // counters of both slots are clean for the next call, whichever slot it uses
        for (int k = 0; k < 2; ++k) {
            c->n_blk[k] = 0u; c->n_vis[k] = 0u; c->n_act[k] = 0u; c->n_chunk[k] = 0u; c->tile_next[k] = 0u;
        }
    }

    // Ascending output (Section 2.1 "then compaction") in one pass: block b
    // takes compaction tiles b, b + gridDim.x, ... in order; a tile publishes
    // its row count, adds up its predecessors' published counts back to the
    // first published prefix (waits bounded), publishes its own prefix and
    // writes its rows.  A tile waits only on lower tiles, which belong to
    // earlier rounds or to lower blocks of the same round, and every block
    // of the cooperative launch is resident, so the waits end.  The
    // accumulator and the row masks are cleared for the next call on the way.
    __shared__ uint32_t s_base;
    uint32_t *stage_idx = reinterpret_cast<uint32_t *>(&S.wp[0]);
    for (uint32_t ct = blockIdx.x; ct < P.n_ctiles; ct += gridDim.x) {
        const size_t wi = (size_t)ct * NT + tid;
        const uint32_t raw = __ldcg(P.yrm32 + wi);
        uint32_t bits = raw ? raw & unvisited(wi) : 0u;
        uint32_t tile_tot;
        const uint32_t off = block_excl_scan(__popc(bits), &tile_tot);
        if (tid < 32) {
            // warp 0 looks back over windows of 32 predecessors (lane l reads
            // tile j - l) until one has published its prefix
            const int lane = tid;
            const unsigned long long epoch = launch_epoch(), tag = epoch << 34;
            if (lane == 0) st_release64(P.ctile_flag + ct, tag | (1ull << 32) | tile_tot);   // count published
            uint32_t base = 0;
            bool ok = true;
            const unsigned long long t0 = globaltimer();
            for (int j = (int)ct - 1; j >= 0 && ok; j -= 32) {
                const int idx = j - lane;
                unsigned long long f = 0;
                if (idx >= 0) {
                    while (((f = ld_acquire64(P.ctile_flag + idx)) >> 34) != epoch) {
                        if ((long long)(globaltimer() - t0) > P.timeout_ns) { ok = false; break; }
                    }
                }
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                const uint32_t pm = __ballot_sync(FULL, idx >= 0 && ((f >> 32) & 2ull));   // prefixes
                const int stop = pm ? __ffs(pm) - 1 : 31;
                base += __reduce_add_sync(FULL, (lane <= stop && idx >= 0) ? (uint32_t)f : 0u);
                if (pm) break;
            }
            if (!ok && lane == 0) atomicCAS(&P.ctrl->err, 0u, (unsigned)DBS_ERR_TIMEOUT);
            if (lane == 0) {
                st_release64(P.ctile_flag + ct, tag | (2ull << 32) | (base + tile_tot));      // prefix published
                s_base = ok ? base : 0xFFFFFFFFu;
            }
        }
        __syncthreads();
        const uint32_t base = s_base;
        if (base == 0xFFFFFFFFu) return;
        if (raw) P.yrm32[wi] = 0u;
        // The tile's rows go to shared memory first (the warps' pull state
        // is free by now), in rounds of R, and out to y with coalesced
        // stores.
        for (uint32_t r0 = 0; r0 < tile_tot; r0 += STAGE_ROWS<SR>) {
            const uint32_t r1 = min(tile_tot, r0 + STAGE_ROWS<SR>);
            if (off < r1 && off + __popc(bits) > r0) {
                uint32_t b = bits, o = off;
                while (b) {
                    const uint32_t k = __ffs(b) - 1u;
                    b &= b - 1u;
                    if (o >= r0 && o < r1) stage_idx[o - r0] = (uint32_t)(2u * wi + (k >> 4)) * 16u + (k & 15u);
                    ++o;
                }
            }
            __syncthreads();
            // all threads gather the values (rows ascend within the tile, so
            // the accumulator reads are nearly contiguous) and store
            for (uint32_t i = tid; i < r1 - r0; i += NT) {
                const uint32_t row = stage_idx[i];
                P.y_idx[base + r0 + i] = (int32_t)row;
                if (SR == 0) {
                    P.y_val[base + r0 + i] = __ldcg(P.y_acc + row);
                    P.y_acc[row] = 0.0f;
                }
            }
            __syncthreads();
        }
        if (ct == P.n_ctiles - 1 && tid == 0) {
            *P.y_nnz = (long long)(base + tile_tot);
            if (ST) P.ctrl->y_nnz = base + tile_tot;
        }
        __syncthreads();
    }
    if (P.n_ctiles == 0 && blockIdx.x == 0 && tid == 0) *P.y_nnz = 0;
    stamp(P, 3);
}

// One SpMSpV with a dense x and a dense y (Section 4.3, DB-Decoding): the
// vector masks come from warp ballots (Section 4.1).  Counter slot P.slot is
// used by this call; the other slot is reset for the next call.
template <bool ST>
__global__ void __launch_bounds__(NT, 4) k_spmspv_dense(KParams P)
{
    SmemT<0> &S = *reinterpret_cast<SmemT<0> *>(smem_raw);
    // a dense x was handed to the kept CSR SpMV launched just before (the
    // paper's Limitations): the same sample decides, so nothing is left
    // here.  (Leaving before the barrier set-up is safe: the launch count is
    // not advanced, so the next launch uses the counters this one would have.)
    if (P.has_spmv && P.path_force == DBS_PATH_AUTO && dbs::spmvd::dense_x_sample(P.x_in, P.n, P.spmv_frac)) return;
    grid_sync_init(P);
    if (ld_cg(&P.ctrl->err) != 0u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t gtid = (size_t)blockIdx.x * NT + tid, gsz = (size_t)gridDim.x * NT;
    const int slot = launch_slot();
    stats_begin(S);
    if (blockIdx.x == 0 && tid == 0 && ST) reset_stats(P);
    stamp(P, 0);
    for (size_t i = gtid; i < (size_t)P.m; i += gsz) P.y_dense[i] = 0.0f;

    // Phase 1: each warp reads 32 x values, ballots their nonzero pattern and
    // splits it into the two 16-bit block masks; nonzero blocks are counted
    // per warp, per CTA, and added to the global count once per CTA.
    const uint32_t nwords = (uint32_t)((P.n + 31) / 32);
    uint32_t nb = 0, act_cnt = 0, work = 0;
    for (uint32_t w = blockIdx.x * NW + warp; w < nwords; w += gridDim.x * NW) {
        const size_t j = (size_t)w * 32u + lane;
        const float v = j < (size_t)P.n ? __ldg(P.x_in + j) : 0.0f;
        const uint32_t bal = __ballot_sync(FULL, v != 0.0f);
        if (lane == 0) {
            P.dxm32[w] = bal;
            if (bal & 0xFFFFu) { ++nb; work += cb_len(P, 2u * w); }
            if (bal >> 16) { ++nb; work += cb_len(P, 2u * w + 1u); }
            act_cnt += __popc(bal);
        }
    }
    cta_count(&P.ctrl->n_blk[slot], nb);
    cta_count(&P.ctrl->n_vis[slot], work);
    if (ST) cta_count(&P.ctrl->x_active, act_cnt);
    if (!grid_sync(P)) return;
    stamp(P, 1);

    const uint32_t n_nz = ld_cg(&P.ctrl->n_blk[slot]);
    const bool push = choose_push(P, n_nz, ld_cg(&P.ctrl->n_vis[slot]));
    if (push) {
        const uint32_t ch = push_chunk(ld_cg(&P.ctrl->n_vis[slot]));
        for (uint32_t base = blockIdx.x * NT; base < nwords; base += gridDim.x * NT) {
            const uint32_t w = base + tid;
            const uint32_t bal = w < nwords ? __ldcg(P.dxm32 + w) : 0u;
            cta_append(P, S.L, slot, (bal & 0xFFFFu) != 0u, 2u * w, (bal >> 16) != 0u, 2u * w + 1u, ch);
        }
        if (!grid_sync(P)) return;
        push_tasks<0, true, ST>(P, S, P.dxm32, nullptr, nullptr, slot, ch);
    } else {
        pull_tiles<0, true, ST>(P, S, P.dxm32, nullptr, nullptr, slot);
    }
    stamp(P, 2);
    stats_flush(P, S);
    if (blockIdx.x == 0 && tid == 0) {
        Ctrl *c = P.ctrl;
        const int o = slot ^ 1;
        c->n_blk[o] = 0u;
        c->n_vis[o] = 0u;
        c->n_act[o] = 0u;
        c->n_chunk[o] = 0u;
        c->tile_next[o] = 0u;
        c->path = push ? 1u : 2u;
        if (ST) c->nzblk = n_nz;
    }
    stamp(P, 3);
}

// DB-BFS (Section 4.2): the frontier is the vector-block mask; each level is
// next = (A or.and frontier) and not visited, on the path chosen from the
// frontier's nonzero-block ratio.  After a level's traversal one scan over
// the next-frontier words updates visited and levels, clears the old
// frontier and counts the new one's nonzero blocks; a level that takes the
// push path first builds its task list from the frontier words.  Counters
// rotate over three slots: two grid barriers per pull level, three per push.
template <bool ST>
__global__ void __launch_bounds__(NT, 4) k_bfs(KParams P)
{
    SmemT<1> &S = *reinterpret_cast<SmemT<1> *>(smem_raw);
    grid_sync_init(P);
    if (ld_cg(&P.ctrl->err) != 0u) return;
    const int tid = threadIdx.x;
    const size_t gtid = (size_t)blockIdx.x * NT + tid, gsz = (size_t)gridDim.x * NT;
    stats_begin(S);
    const uint32_t nwords = (uint32_t)((P.nbc + 1) / 2);
    for (size_t v = gtid; v < (size_t)P.n; v += gsz) P.levels[v] = -1;
    for (size_t w = gtid; w < nwords; w += gsz) {
        // rows that hold no entry can never be reached (nor can rows beyond
        // m): they start out visited, so tiles of reached and unreachable
        // rows are skipped as soon as the reachable ones are all visited
        const uint32_t lo = 2u * w < (size_t)P.nbr ? (uint32_t)__ldg(P.rb_rows + 2u * w) : 0u;
        const uint32_t hi = 2u * w + 1u < (size_t)P.nbr ? (uint32_t)__ldg(P.rb_rows + 2u * w + 1u) : 0u;
        P.bvis32[w] = ~(lo | (hi << 16));
        P.fm32[0][w] = 0u;
        P.fm32[1][w] = 0u;
    }
    if (blockIdx.x == 0 && tid == 0) {
        Ctrl *c = P.ctrl;
        for (int k = 0; k < 3; ++k) {
            c->n_blk[k] = 0u; c->n_vis[k] = 0u; c->n_act[k] = 0u; c->n_chunk[k] = 0u; c->tile_next[k] = 0u;
        }
        reset_stats(P);
        c->bfs_levels = 0u;
        c->bfs_push_levels = 0u;
    }
    stamp(P, 0);
    if (!grid_sync(P)) return;
    {   // level 0: the source; its push list has one block
        const uint32_t s = (uint32_t)P.bfs_src;
        if (blockIdx.x == 0 && tid == 0) {
            P.levels[s] = 0;
            or16(P.fm32[0], s >> 4, 1u << (s & 15u));
            or16(P.bvis32, s >> 4, 1u << (s & 15u));
            P.ctrl->n_blk[0] = 1u;
            P.ctrl->n_vis[0] = cb_len(P, s >> 4);
        }
        if (blockIdx.x == 0) cta_append(P, S.L, 0, tid == 0, s >> 4, false, 0u, push_chunk(cb_len(P, s >> 4)));
    }
    if (!grid_sync(P)) return;
    stamp(P, 1);

    unsigned long long nz_sum = 0;
    uint32_t push_levels = 0, L = 1;
    for (;; ++L) {
        const int cur = (int)((L - 1) % 3), nxt = (int)(L % 3), old = (int)((L + 1) % 3);
        uint32_t *fcur = P.fm32[(L - 1) & 1], *fnext = P.fm32[L & 1];
        const uint32_t n_nz = ld_cg(&P.ctrl->n_blk[cur]);
        if (blockIdx.x == 0 && tid == 0 && L - 1u < (uint32_t)BFS_LEVEL_LOG) P.ctrl->lv_t[L - 1u] = globaltimer();
        if (n_nz == 0u) break;
        nz_sum += n_nz;
        const bool push = choose_push(P, n_nz, ld_cg(&P.ctrl->n_vis[cur]));
        push_levels += push;
        if (blockIdx.x == 0 && tid == 0 && L - 1u < (uint32_t)BFS_LEVEL_LOG) {
            P.ctrl->lv_nz[L - 1u] = n_nz;
            P.ctrl->lv_nv[L - 1u] = ld_cg(&P.ctrl->n_vis[cur]);
            P.ctrl->lv_path[L - 1u] = push ? 1u : 2u;
        }
        if (push) {
            // push list of the frontier, built only for push levels (few
            // blocks; level 1's was built with the source)
            const uint32_t ch = push_chunk(ld_cg(&P.ctrl->n_vis[cur]));
            if (L > 1u) {
                for (uint32_t base = blockIdx.x * NT; base < nwords; base += gridDim.x * NT) {
                    const uint32_t w = base + tid;
                    const uint32_t fm = w < nwords ? __ldcg(fcur + w) : 0u;
                    cta_append(P, S.L, cur, (fm & 0xFFFFu) != 0u, 2u * w, (fm >> 16) != 0u, 2u * w + 1u, ch);
                }
                if (!grid_sync(P)) return;
            }
            push_tasks<1, false, ST>(P, S, fcur, P.bvis32, fnext, cur, ch);
        } else {
            pull_bool<ST>(P, S, fcur, P.bvis32, fnext, cur);
        }
        if (!grid_sync(P)) return;
        if (blockIdx.x == 0 && tid == 0 && L - 1u < (uint32_t)BFS_LEVEL_LOG) P.ctrl->lv_u[L - 1u] = globaltimer();

        // level update over all frontier words (one thread per word)
        uint32_t nb = 0, reached = 0, work = 0;
        for (uint32_t w = blockIdx.x * NT + tid; w < nwords; w += gridDim.x * NT) {
            const uint32_t raw = __ldcg(fnext + w);
            if (__ldcg(fcur + w)) fcur[w] = 0u;
            // push leaves visited rows among the found ones: keep the new rows
            const uint32_t vw = raw ? __ldcg(P.bvis32 + w) : 0u;
            const uint32_t nm = raw & ~vw;
            if (nm != raw) fnext[w] = nm;
            if (nm) {
                P.bvis32[w] = vw | nm;
                reached += __popc(nm);
                if (nm & 0xFFFFu) { ++nb; work += cb_len(P, 2u * w); }
                if (nm >> 16) { ++nb; work += cb_len(P, 2u * w + 1u); }
                uint32_t bits = nm;
                while (bits) {
                    const uint32_t k = __ffs(bits) - 1u;
                    bits &= bits - 1u;
                    P.levels[(2u * w + (k >> 4)) * 16u + (k & 15u)] = (int32_t)L;
                }
            }
        }
        cta_count(&P.ctrl->n_blk[nxt], nb);
        cta_count(&P.ctrl->n_vis[nxt], work);
        if (ST) cta_count(&P.ctrl->reached, reached);
        if (blockIdx.x == 0 && tid == 0) {
            Ctrl *c = P.ctrl;
            c->n_blk[old] = 0u;
            c->n_vis[old] = 0u;
            c->n_act[old] = 0u;
            c->n_chunk[old] = 0u;
            c->tile_next[old] = 0u;
        }
        if (!grid_sync(P)) return;
    }
    stamp(P, 2);
    stats_flush(P, S);
    if (blockIdx.x == 0 && tid == 0) {
        Ctrl *c = P.ctrl;
        // Every block has passed the last barrier and reads only n_blk[cur],
        // which is already 0: all slots can be cleared for the next call.
        for (int k = 0; k < 3; ++k) {
            c->n_blk[k] = 0u; c->n_vis[k] = 0u; c->n_act[k] = 0u; c->n_chunk[k] = 0u; c->tile_next[k] = 0u;
        }
        c->bfs_levels = L - 1u;   // the loop stops when frontier L-1 is empty
        c->bfs_push_levels = push_levels;
        c->path = 0u;
        c->nzblk = nz_sum;
        if (ST) c->reached += 1;   // the source
    }
    stamp(P, 3);
}

// DB-Decoding layer (Section 4.3; the mask generation of Section 4.1 moved
// into the traversal): y = A x' with x'_j = x_j where |x_j| > tau (NaN is
// kept) and 0 elsewhere -- magnitude thresholding of the activation -- on
// the pull path, in one ordinary launch.  A block of threads owns one row
// block at a time: each thread takes blocks of it (three at a time, their
// loads issued together), forms each block's activation mask from the 16 x
// values of its column block, and adds the products of every (block, active
// column) pair into its own 16 row sums; one reduction over the block then
// gives the row block's 16 results, stored once (rows without an active
// entry get 0).  No partial sum leaves the block, so no atomic, counter or
// fence is needed, and no metadata pass or device-wide barrier precedes the
// traversal.
__device__ __forceinline__ uint32_t act_mask(const float *__restrict__ x, uint32_t col, int n, float tau)
{
    const size_t j0 = (size_t)col * 16u;
    uint32_t m = 0;
    if (j0 + 16u <= (size_t)n) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x + j0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = __ldg(x4 + q);
            m |= (!(fabsf(v.x) <= tau) ? 1u : 0u) << (4 * q);
            m |= (!(fabsf(v.y) <= tau) ? 1u : 0u) << (4 * q + 1);
            m |= (!(fabsf(v.z) <= tau) ? 1u : 0u) << (4 * q + 2);
            m |= (!(fabsf(v.w) <= tau) ? 1u : 0u) << (4 * q + 3);
        }
    } else {
        for (uint32_t c = 0; c < 16u; ++c)
            if (j0 + c < (size_t)n && !(fabsf(__ldg(x + j0 + c)) <= tau)) m |= 1u << c;
    }
    return m;
}

constexpr int DEC_NT = 512; // threads per row block
constexpr int DEC_NW = DEC_NT / 32;
constexpr int DEC_K = 2;    // blocks per thread per round of a row block
constexpr int DEC_SLOTS = DEC_NT * DEC_K;

// The CTA owns one row block.  Per round of up to DEC_SLOTS blocks: each
// thread loads its blocks' descriptors and forms their activation masks;
// COO blocks are done by the thread at once, the other blocks' (block,
// active column) pairs are listed in shared memory and shared out evenly,
// so the round ends after about pairs / DEC_NT column reads per thread
// whatever the mix of active columns per block.  Every pair adds into the
// same 16 rows, kept in registers until the row block's reduction.
__global__ void __launch_bounds__(DEC_NT, 2) k_decode(KParams P)
{
    constexpr int NT = DEC_NT, NW = DEC_NW;
    __shared__ float s_part[NW][16];
    __shared__ uint32_t s_ref[DEC_SLOTS], s_meta[DEC_SLOTS], s_col[DEC_SLOTS];
    __shared__ uint16_t s_pair[DEC_SLOTS * 16];   // slot << 4 | column
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float tau = P.tau;
    const float *__restrict__ x = P.x_in;
    for (uint32_t rb = blockIdx.x; rb < (uint32_t)P.nbr; rb += gridDim.x) {
        const uint32_t p0 = __ldg(P.rb_ptr + rb), p1 = __ldg(P.rb_ptr + rb + 1);
        float acc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) acc[r] = 0.0f;
        for (uint32_t base = p0; base < p1; base += DEC_SLOTS) {
            uint2 d[DEC_K];
            uint32_t ref[DEC_K], am[DEC_K];
#pragma unroll
            for (int k = 0; k < DEC_K; ++k) {
                const uint32_t p = base + (uint32_t)(k * NT + tid);
                d[k] = p < p1 ? __ldg(P.blk_desc + p) : make_uint2(0u, 0u);
                ref[k] = p < p1 ? __ldg(P.blk_ref + p) : 0u;
            }
            uint32_t np = 0;
#pragma unroll
            for (int k = 0; k < DEC_K; ++k) {
                am[k] = base + (uint32_t)(k * NT + tid) < p1
                            ? act_mask(x, d[k].x & DESC_COL_MASK, P.n, tau) & d[k].y & 0xFFFFu : 0u;
                const uint32_t meta = d[k].y, col = d[k].x & DESC_COL_MASK;
                if (am[k] && meta_fmt(meta) == FMT_COO) {
                    coo_lane(reinterpret_cast<const uint8_t *>(P.payload + ref[k]), meta_nnz(meta), am[k],
                             x + (size_t)col * 16u, true, [&](uint32_t r, float v) {
#pragma unroll
                                 for (int rr = 0; rr < 16; ++rr) acc[rr] += (uint32_t)rr == r ? v : 0.0f;
                             });
                    am[k] = 0u;
                }
                if (am[k]) {
                    const uint32_t slot = (uint32_t)(k * NT + tid);
                    s_ref[slot] = ref[k];
                    s_meta[slot] = meta;
                    s_col[slot] = col;
                    np += __popc(am[k]);
                }
            }
            uint32_t tot;
            uint32_t o = block_excl_scan<NW>(np, &tot);
#pragma unroll
            for (int k = 0; k < DEC_K; ++k)
                for (uint32_t a = am[k]; a; a &= a - 1u)
                    s_pair[o++] = (uint16_t)(((uint32_t)(k * NT + tid) << 4) | (__ffs(a) - 1u));
            __syncthreads();
            // two pairs per step, their loads issued together
            for (uint32_t i = tid; i < tot; i += 2 * NT) {
                const uint32_t e0 = s_pair[i], s0 = e0 >> 4, c0 = e0 & 15u, m0 = s_meta[s0];
                const bool two = i + NT < tot;
                const uint32_t e1 = two ? s_pair[i + NT] : e0, s1 = e1 >> 4, c1 = e1 & 15u, m1 = s_meta[s1];
                const float x0 = __ldg(x + (size_t)s_col[s0] * 16u + c0), x1 = __ldg(x + (size_t)s_col[s1] * 16u + c1);
                pair_products<true>(reinterpret_cast<const uint8_t *>(P.payload + s_ref[s0]), meta_fmt(m0),
                                    meta_nnz(m0), c0, x0, acc);
                if (two)
                    pair_products<true>(reinterpret_cast<const uint8_t *>(P.payload + s_ref[s1]), meta_fmt(m1),
                                        meta_nnz(m1), c1, x1, acc);
            }
            __syncthreads();
        }
        // row sums over the block: warp transpose reduction, then the warps
        const float v = warp_rows_sum(acc, true, lane);
        if (!(lane & 1)) s_part[warp][(lane >> 1) & 15] = v;
        __syncthreads();
        if (tid < 16) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < NW; ++w) sum += s_part[w][tid];
            const size_t row = (size_t)rb * 16u + tid;
            if (row < (size_t)P.m) P.y_dense[row] = sum;
        }
        __syncthreads();
    }
}

// Withholds block 0 from the barrier so every other block's wait expires.
__global__ void __launch_bounds__(NT, 5) k_selftest_wait(KParams P)
{
    grid_sync_init(P);
    if (blockIdx.x == 0) return;
    grid_sync(P);
}

}  // namespace

// ------------------------------------------------------------------ host

struct dbs_workspace {
    const dbs_matrix *A = nullptr;
    int device = -1;
    int sms = 0;
    int grid_sparse[2][2] = {{0, 0}, {0, 0}};   // [semiring][statistics]
    int grid_dense[2] = {0, 0}, grid_bfs[2] = {0, 0};
    bool decode_ok = false;
    dbs_exec_opts opts{};
    float *x_dense = nullptr;
    uint32_t *xm32 = nullptr;
    uint32_t *dxm32 = nullptr;
    uint32_t *act[3] = {nullptr, nullptr, nullptr};
    uint4 *chunks[3] = {nullptr, nullptr, nullptr};
    float *y_acc = nullptr;
    uint32_t *yrm32 = nullptr;
    unsigned long long *ctile_flag = nullptr;
    uint32_t n_ctiles = 0;
    uint32_t *bvis32 = nullptr;
    uint32_t *fm32[2] = {nullptr, nullptr};
    float *spmv_part = nullptr;       // dense_spmv matrices: split rows' partial sums
    uint32_t *spmv_cnt = nullptr;     // and chunk counters (zero between calls)
    Ctrl *ctrl = nullptr;
    bool last_was_bfs = false;
};

namespace {

void ws_free(dbs_workspace *w)
{
    dbs::dev_free(w->x_dense); dbs::dev_free(w->xm32); dbs::dev_free(w->dxm32); dbs::dev_free(w->y_acc); dbs::dev_free(w->yrm32);
    dbs::dev_free(w->ctile_flag); dbs::dev_free(w->bvis32); dbs::dev_free(w->fm32[0]); dbs::dev_free(w->fm32[1]);
    dbs::dev_free(w->ctrl); dbs::dev_free(w->spmv_part); dbs::dev_free(w->spmv_cnt);
    for (int s = 0; s < 3; ++s) { dbs::dev_free(w->act[s]); dbs::dev_free(w->chunks[s]); }
}

template <class T>
bool dalloc(T **p, size_t count)
{
    size_t bytes = std::max<size_t>(count * sizeof(T), 16);
    if (dev_malloc(p, bytes) != cudaSuccess) { cudaGetLastError(); *p = nullptr; return false; }
    if (cudaMemset(*p, 0, bytes) != cudaSuccess) { cudaGetLastError(); return false; }
    return true;
}

KParams make_params(const dbs_matrix *A, dbs_workspace *w)
{
    KParams P{};
    P.m = (int32_t)A->m; P.n = (int32_t)A->n; P.nbr = (int32_t)A->nbr; P.nbc = (int32_t)A->nbc;
    P.B = (uint32_t)A->B; P.T = (uint32_t)A->T; P.valued = A->valued;
    P.rb_ptr = A->d_rb_ptr;
    P.blk_desc = reinterpret_cast<const uint2 *>(A->d_blk_desc);
    P.blk_ref = A->d_blk_ref;
    P.cb_ptr = A->d_cb_ptr;
    P.csc_desc = reinterpret_cast<const uint2 *>(A->d_csc_desc);
    P.csc_ref = A->d_csc_ref;
    P.payload = reinterpret_cast<const uint4 *>(A->d_payload);
    P.tiles = reinterpret_cast<const uint4 *>(A->d_tiles);
    P.rb_rows = A->d_rb_rows;
    P.x_dense = w->x_dense; P.xm32 = w->xm32; P.dxm32 = w->dxm32;
    for (int s = 0; s < 3; ++s) { P.act[s] = w->act[s]; P.chunks[s] = w->chunks[s]; }
    P.y_acc = w->y_acc; P.yrm32 = w->yrm32; P.ctile_flag = w->ctile_flag; P.n_ctiles = w->n_ctiles;
    P.bvis32 = w->bvis32; P.fm32[0] = w->fm32[0]; P.fm32[1] = w->fm32[1];
    P.ctrl = w->ctrl;
    P.th3 = w->opts.th3;
    P.push_frac = w->opts.push_work_frac;
    P.has_spmv = A->plan ? 1 : 0;
    P.spmv_frac = w->opts.spmv_x_frac;
    P.local_pull_min = w->opts.local_pull_min;
    P.stats = w->opts.collect_stats;
    P.timeout_ns = w->opts.wait_timeout_ns;
    return P;
}

constexpr size_t SMEM0 = sizeof(SmemT<0>), SMEM1 = sizeof(SmemT<1>);   // dynamic shared memory per CTA

dbs_status launch(const void *fn, int grid, KParams &P, cudaStream_t s, size_t smem)
{
    void *args[] = {&P};
    cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(NT), args, smem, s);
    if (e != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    return DBS_OK;
}

// A workspace launch (the launch count that picks the barrier counter and
// the counter slot is kept on the device).
dbs_status launch_ws(dbs_workspace *, const void *fn, int grid, KParams &P, cudaStream_t s, size_t smem)
{
    return launch(fn, grid, P, s, smem);
}

int coop_grid(const void *fn, int sms, size_t smem)
{
    int nb = 0;
    if (smem > 48u * 1024u &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, NT, smem) != cudaSuccess) { cudaGetLastError(); return 0; }
    return std::min(nb * sms, MAX_GRID);
}

dbs_status check_ready(const dbs_matrix *A, dbs_workspace *w)
{
    if (!A || !w || w->A != A || !A->on_device) return DBS_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    if (dev != w->device) return DBS_ERR_INVALID_ARG;
    return DBS_OK;
}

}  // namespace

extern "C" {

void dbs_exec_opts_default(dbs_exec_opts *o)
{
    if (!o) return;
    o->th3 = 0.01;
    // GB300 default: decide on the implied work.  Forced-path sweeps on
    // R-MAT scale 20 (SpMSpV and BFS levels) put the crossover near
    // n_vis / B = 0.45 (push 1.6x faster at 0.14 and 1.1x at 0.25, pull
    // 1.06x faster at 0.61 and 1.35x at 0.81); 0 selects the paper's th3 rule.
    o->push_work_frac = 0.45;
    // patched CSR always in row mode on GB300: its two dependent loads beat
    // the column mode's four even at ~2 active columns per block (LLM weight)
    o->local_pull_min = 0;
    o->collect_stats = 0;
    o->wait_timeout_ns = 2000000000LL;
    // dense-x calls on dense_spmv matrices: SpMV from this sampled density
    // (on GB300 the CSR SpMV already beats the blocked pull at 10 % on the
    // FEM, LLM and R-MAT matrices: 134 vs 220, 48 vs 52, 113 vs 255 us)
    o->spmv_x_frac = 0.08;
}

dbs_status dbs_workspace_create(const dbs_matrix *A, dbs_workspace **out)
{
    if (!A || !out || !A->on_device) return DBS_ERR_INVALID_ARG;
    dbs_workspace *w = alloc_fault() ? nullptr : new (std::nothrow) dbs_workspace();
    if (!w) return DBS_ERR_OOM;
    w->A = A;
    dbs_exec_opts_default(&w->opts);
    if (cudaGetDevice(&w->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&w->sms, cudaDevAttrMultiProcessorCount, w->device) != cudaSuccess) {
        cudaGetLastError();
        delete w;
        return DBS_ERR_CUDA;
    }
    const size_t nbc = (size_t)A->nbc, nbr = (size_t)A->nbr;
    const size_t chunk_cap = (size_t)A->B / PUSH_CHUNK_MIN + nbc + 1;   // tasks of the smallest size
    w->n_ctiles = (uint32_t)((nbr + CTILE - 1) / CTILE);
    const size_t yrm_words = std::max<size_t>(1, (size_t)w->n_ctiles) * CTILE / 2 + 8;
    bool ok = dalloc(&w->x_dense, nbc * 16 + 16) && dalloc(&w->xm32, nbc / 2 + 8) &&
              dalloc(&w->dxm32, nbc / 2 + 8) &&
              dalloc(&w->y_acc, nbr * 16 + 16) && dalloc(&w->yrm32, yrm_words) &&
              dalloc(&w->ctile_flag, (size_t)w->n_ctiles + 1) &&
              dalloc(&w->bvis32, nbr / 2 + 8) &&
              dalloc(&w->fm32[0], nbc / 2 + 8) && dalloc(&w->fm32[1], nbc / 2 + 8) && dalloc(&w->ctrl, 1);
    for (int s = 0; s < 3 && ok; ++s) ok = dalloc(&w->act[s], nbc + 1) && dalloc(&w->chunks[s], chunk_cap);
    if (ok && A->plan) ok = dalloc(&w->spmv_part, A->plan->max_chunks) && dalloc(&w->spmv_cnt, A->plan->max_split);
    if (!ok) { ws_free(w); delete w; return DBS_ERR_OOM; }
    w->grid_sparse[0][0] = coop_grid((const void *)k_spmspv_sparse<0, false>, w->sms, SMEM0);
    w->grid_sparse[0][1] = coop_grid((const void *)k_spmspv_sparse<0, true>, w->sms, SMEM0);
    w->grid_sparse[1][0] = coop_grid((const void *)k_spmspv_sparse<1, false>, w->sms, SMEM1);
    w->grid_sparse[1][1] = coop_grid((const void *)k_spmspv_sparse<1, true>, w->sms, SMEM1);
    w->grid_dense[0] = coop_grid((const void *)k_spmspv_dense<false>, w->sms, SMEM0);
    w->grid_dense[1] = coop_grid((const void *)k_spmspv_dense<true>, w->sms, SMEM0);
    w->grid_bfs[0] = coop_grid((const void *)k_bfs<false>, w->sms, SMEM1);
    w->grid_bfs[1] = coop_grid((const void *)k_bfs<true>, w->sms, SMEM1);
    {
        int nb = 0;
        w->decode_ok = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, (const void *)k_decode, DEC_NT, 0) ==
                           cudaSuccess && nb > 0;
        cudaGetLastError();
    }
    bool grids_ok = true;
    for (int a = 0; a < 2; ++a)
        grids_ok = grids_ok && w->grid_sparse[0][a] && w->grid_sparse[1][a] && w->grid_dense[a] && w->grid_bfs[a];
    grids_ok = grids_ok && w->decode_ok;
    if (!grids_ok) {
        ws_free(w);
        delete w;
        return DBS_ERR_CUDA;
    }
    *out = w;
    return DBS_OK;
}

dbs_status dbs_workspace_destroy(dbs_workspace *w)
{
    if (!w) return DBS_OK;
    ws_free(w);
    delete w;
    return DBS_OK;
}

dbs_status dbs_workspace_set_opts(dbs_workspace *w, const dbs_exec_opts *o)
{
    if (!w || !o) return DBS_ERR_INVALID_ARG;
    if (!(o->th3 >= 0.0) || !(o->push_work_frac >= 0.0) || o->local_pull_min < 0 || o->wait_timeout_ns <= 0 ||
        !(o->spmv_x_frac >= 0.0))
        return DBS_ERR_INVALID_ARG;
    w->opts = *o;
    return DBS_OK;
}

dbs_status dbs_workspace_check(dbs_workspace *w, void *stream)
{
    if (!w) return DBS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    Ctrl c;
    if (cudaMemcpy(&c, w->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    if (c.err == 0u) return DBS_OK;
    // A failed call can leave barrier, counters and scratch half-updated:
    // reset all of them.
    const dbs_matrix *A = w->A;
    bool ok = cudaMemset(w->ctrl, 0, sizeof(Ctrl)) == cudaSuccess &&
              cudaMemset(w->x_dense, 0, ((size_t)A->nbc * 16 + 16) * sizeof(float)) == cudaSuccess &&
              cudaMemset(w->xm32, 0, ((size_t)A->nbc / 2 + 8) * 4) == cudaSuccess &&
              cudaMemset(w->y_acc, 0, ((size_t)A->nbr * 16 + 16) * sizeof(float)) == cudaSuccess &&
              cudaMemset(w->yrm32, 0, (std::max<size_t>(1, w->n_ctiles) * CTILE / 2 + 8) * 4) == cudaSuccess &&
              cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) { cudaGetLastError(); return DBS_ERR_CUDA; }
    return (dbs_status)c.err;
}

dbs_status dbs_spmspv(const dbs_matrix *A, dbs_semiring sr, const int32_t *x_idx, const float *x_val,
                      int64_t x_nnz, const uint16_t *visited_mask, int32_t *y_idx, float *y_val,
                      int64_t *y_nnz, dbs_path path, dbs_workspace *w, void *stream)
{
    dbs_status st = check_ready(A, w);
    if (st != DBS_OK) return st;
    if (sr != DBS_PLUS_TIMES_F32 && sr != DBS_OR_AND_BOOL) return DBS_ERR_INVALID_ARG;
    if (path < DBS_PATH_AUTO || path > DBS_PATH_PULL) return DBS_ERR_INVALID_ARG;
    if (x_nnz < 0 || x_nnz > A->n || (x_nnz > 0 && !x_idx) || !y_idx || !y_nnz) return DBS_ERR_INVALID_ARG;
    if (sr == DBS_PLUS_TIMES_F32) {
        if (!A->valued) return DBS_ERR_UNSUPPORTED;
        if ((x_nnz > 0 && !x_val) || !y_val || visited_mask) return DBS_ERR_INVALID_ARG;
    }
    if (reinterpret_cast<uintptr_t>(visited_mask) & 3u) return DBS_ERR_INVALID_ARG;
    KParams P = make_params(A, w);
    P.path_force = (int)path;
    P.x_idx = x_idx;
    P.x_val = x_val;
    P.x_nnz = x_nnz;
    P.xv = w->x_dense;
    P.uvis32 = reinterpret_cast<const uint32_t *>(visited_mask);
    P.y_idx = y_idx;
    P.y_val = y_val;
    P.y_nnz = reinterpret_cast<long long *>(y_nnz);
    const int st_on = P.stats ? 1 : 0, sri = sr == DBS_PLUS_TIMES_F32 ? 0 : 1;
    const void *fns[2][2] = {{(const void *)k_spmspv_sparse<0, false>, (const void *)k_spmspv_sparse<0, true>},
                             {(const void *)k_spmspv_sparse<1, false>, (const void *)k_spmspv_sparse<1, true>}};
    const void *fn = fns[sri][st_on];
    w->last_was_bfs = false;
    // A call whose expected push work (x entries times the mean column-block
    // length) is below two tasks of 256 blocks per SM runs on one block per
    // SM: its grid barriers and block start-up cost less, and the work fits.
    // (A larger bound made calls that turn out to pull, or push with many
    // payload hits, slower.)
    int grid = w->grid_sparse[sri][st_on];
    const long long nbc = A->nbc > 0 ? A->nbc : 1;
    const long long work = (long long)x_nnz * ((A->B + nbc - 1) / nbc);
    if (path != DBS_PATH_PULL && work < 2LL * 256LL * w->sms) grid = std::min(grid, w->sms);
    return launch_ws(w, fn, grid, P, (cudaStream_t)stream, sr == DBS_PLUS_TIMES_F32 ? SMEM0 : SMEM1);
}

dbs_status dbs_spmspv_dense(const dbs_matrix *A, const float *x, float *y, dbs_path path, dbs_workspace *w,
                            void *stream)
{
    dbs_status st = check_ready(A, w);
    if (st != DBS_OK) return st;
    if (!A->valued) return DBS_ERR_UNSUPPORTED;
    if ((A->n > 0 && !x) || (A->m > 0 && !y) || path < DBS_PATH_AUTO || path > DBS_PATH_SPMV ||
        (path == DBS_PATH_SPMV && !A->plan))
        return DBS_ERR_INVALID_ARG;
    KParams P = make_params(A, w);
    P.path_force = (int)path;
    P.x_in = x;
    P.xv = x;
    P.y_dense = y;
    w->last_was_bfs = false;
    if (A->plan && (path == DBS_PATH_AUTO || path == DBS_PATH_SPMV)) {
        // the kept CSR SpMV first: forced, or gated by the sampled density of x
        st = spmv_launch_dense(A->plan, w->spmv_part, w->spmv_cnt, x, y, w->opts.spmv_x_frac, path == DBS_PATH_AUTO,
                               &w->ctrl->path, (cudaStream_t)stream);
        if (st != DBS_OK || path == DBS_PATH_SPMV) return st;
    }
    return P.stats ? launch_ws(w, (const void *)k_spmspv_dense<true>, w->grid_dense[1], P, (cudaStream_t)stream, SMEM0)
                   : launch_ws(w, (const void *)k_spmspv_dense<false>, w->grid_dense[0], P, (cudaStream_t)stream, SMEM0);
}

dbs_status dbs_decode_layer(const dbs_matrix *A, const float *x, float tau, float *y, dbs_workspace *w, void *stream)
{
    dbs_status st = check_ready(A, w);
    if (st != DBS_OK) return st;
    if (!A->valued) return DBS_ERR_UNSUPPORTED;
    if ((A->n > 0 && !x) || (A->m > 0 && !y) || !(tau >= 0.0f) || (reinterpret_cast<uintptr_t>(x) & 15u))
        return DBS_ERR_INVALID_ARG;
    if (A->m == 0) return DBS_OK;
    KParams P = make_params(A, w);
    P.path_force = DBS_PATH_PULL;
    P.x_in = x;
    P.xv = x;
    P.tau = tau;
    P.y_dense = y;
    // one block per row block, up to two blocks per SM (the rest loop)
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(A->nbr, 2 * (int64_t)w->sms));
    k_decode<<<grid, DEC_NT, 0, (cudaStream_t)stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return DBS_ERR_CUDA;
    return DBS_OK;
}

dbs_status dbs_bfs(const dbs_matrix *A, int64_t src, int32_t *levels, int32_t *nlevels_host, dbs_path path,
                   dbs_workspace *w, void *stream)
{
    dbs_status st = check_ready(A, w);
    if (st != DBS_OK) return st;
    if (A->m != A->n || src < 0 || src >= A->n || !levels || path < DBS_PATH_AUTO || path > DBS_PATH_PULL)
        return DBS_ERR_INVALID_ARG;
    KParams P = make_params(A, w);
    P.path_force = (int)path;
    P.bfs_src = src;
    P.levels = levels;
    cudaStream_t s = (cudaStream_t)stream;
    // Counter slots: a dense-x call leaves its own slot dirty and clears the
    // other, which the next launch (the count advanced by one) uses;
    // sparse-x and BFS calls leave every slot clear.
    w->last_was_bfs = true;
    st = P.stats ? launch_ws(w, (const void *)k_bfs<true>, w->grid_bfs[1], P, s, SMEM1)
                 : launch_ws(w, (const void *)k_bfs<false>, w->grid_bfs[0], P, s, SMEM1);
    if (st != DBS_OK || !nlevels_host) return st;
    Ctrl c;
    if (cudaMemcpyAsync(&c, w->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    if (c.err) return (dbs_status)c.err;
    *nlevels_host = (int32_t)c.bfs_levels;
    return DBS_OK;
}

dbs_status dbs_last_stats(dbs_workspace *w, void *stream, dbs_stats *out)
{
    if (!w || !out) return DBS_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    Ctrl c;
    if (cudaMemcpy(&c, w->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    *out = dbs_stats{};
    out->path = (int32_t)c.path;
    out->status = (int32_t)c.err;
    out->n_nzblk = (int64_t)c.nzblk;
    out->n_blk = w->A->nbc;
    out->x_active = (int64_t)c.x_active;
    out->visited_blocks = (int64_t)c.visited;
    out->hit_blocks = (int64_t)c.hits;
    out->touched_nnz = (int64_t)c.touched;
    out->bytes_alg = (int64_t)c.bytes;
    out->y_nnz = w->last_was_bfs ? (int64_t)c.reached : (int64_t)c.y_nnz;
    out->bfs_levels = (int32_t)c.bfs_levels;
    out->bfs_push_levels = (int32_t)c.bfs_push_levels;
    for (int i = 0; i < 3; ++i)
        out->phase_ns[i] = c.t_phase[i + 1] >= c.t_phase[i] ? (int64_t)(c.t_phase[i + 1] - c.t_phase[i]) : 0;
    return DBS_OK;
}

dbs_status dbs_bfs_level_stats(dbs_workspace *w, void *stream, int32_t max_levels, int64_t *frontier_blocks,
                               int64_t *push_work, int32_t *path, int64_t *level_ns, int64_t *traversal_ns)
{
    if (!w || max_levels < 0) return DBS_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    Ctrl c;
    if (cudaMemcpy(&c, w->ctrl, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    if (!w->last_was_bfs) return DBS_ERR_INVALID_ARG;
    const int n = std::min<int>(std::min<int>(max_levels, BFS_LEVEL_LOG), (int)c.bfs_levels);
    for (int l = 0; l < n; ++l) {
        if (frontier_blocks) frontier_blocks[l] = c.lv_nz[l];
        if (push_work) push_work[l] = c.lv_nv[l];
        if (path) path[l] = (int32_t)c.lv_path[l];
        if (level_ns) level_ns[l] = c.lv_t[l + 1] >= c.lv_t[l] ? (int64_t)(c.lv_t[l + 1] - c.lv_t[l]) : 0;
        if (traversal_ns) traversal_ns[l] = c.lv_u[l] >= c.lv_t[l] ? (int64_t)(c.lv_u[l] - c.lv_t[l]) : 0;
    }
    return DBS_OK;
}

dbs_status dbs_selftest_wait_timeout(dbs_workspace *w, void *stream)
{
    if (!w) return DBS_ERR_INVALID_ARG;
    KParams P = make_params(w->A, w);
    int grid = std::min(coop_grid((const void *)k_selftest_wait, w->sms, 0), 2 * w->sms);
    if (grid < 2) return DBS_ERR_UNSUPPORTED;
    return launch_ws(w, (const void *)k_selftest_wait, grid, P, (cudaStream_t)stream, 0);
}

}  // extern "C"

// ------------------------------------------------- allocation-free entry
//
// dbs_spmspv_dense_noalloc runs the dense-x SpMSpV kernel on the pull path
// with its scratch (the control block with the grid-barrier state and
// counters, and the vector-block mask words) in the fixed device array
// below instead of a workspace.  It is meant for callers that must not
// allocate GPU memory after start-up: cudaMalloc can synchronise the device
// and its failures surface at arbitrary times, which real-time serving loops
// and callers running under a fixed, pre-reserved memory budget cannot
// accept.  The array lives as long as the library is loaded on every device
// that loads it.

namespace {

constexpr int64_t NOALLOC_MAX_N = int64_t(1) << 22;                  // columns of A
constexpr size_t NOALLOC_MASK_WORDS = (size_t)NOALLOC_MAX_N / 32 + 8;  // 2 block masks per word
constexpr size_t NOALLOC_CTRL_BYTES = (sizeof(Ctrl) + 255) / 256 * 256;
constexpr size_t NOALLOC_BYTES = NOALLOC_CTRL_BYTES + NOALLOC_MASK_WORDS * sizeof(uint32_t);

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

struct NoAllocDevice {
    bool ready = false;
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
    int grid = 0;
};
constexpr int NOALLOC_MAX_DEVICES = 64;
NoAllocDevice g_noalloc_dev[NOALLOC_MAX_DEVICES];

// Once per device, with that device current: resolve the array's device
// address (in host code its name is only a stand-in) and the cooperative
// grid size.  No memory is allocated.
dbs_status noalloc_setup(int dev)
{
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (d.ready) return DBS_OK;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    const int grid = coop_grid((const void *)k_spmspv_dense<false>, sms, SMEM0);
    if (grid <= 0) return DBS_ERR_CUDA;
    d.scratch = static_cast<unsigned char *>(ptr);
    d.grid = grid;
    d.ready = true;
    return DBS_OK;
}

}  // namespace

extern "C" dbs_status dbs_spmspv_dense_noalloc_check(void *stream)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES || !g_noalloc_dev[dev].ready) return DBS_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    unsigned err = 0;
    if (cudaMemcpyFromSymbol(&err, g_noalloc_scratch, sizeof(unsigned), offsetof(Ctrl, err), cudaMemcpyDeviceToHost) !=
        cudaSuccess) {
        cudaGetLastError();
        return DBS_ERR_CUDA;
    }
    return (dbs_status)err;
}

extern "C" dbs_status dbs_spmspv_dense_noalloc(const dbs_matrix *A, const float *x, float *y, void *stream)
{
    if (!A || !A->on_device || !A->valued) return A && !A->valued ? DBS_ERR_UNSUPPORTED : DBS_ERR_INVALID_ARG;
    if ((A->n > 0 && !x) || (A->m > 0 && !y)) return DBS_ERR_INVALID_ARG;
    if (A->n > NOALLOC_MAX_N) return DBS_ERR_INVALID_ARG;      // beyond the fixed scratch
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    if (dev != A->device || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return DBS_ERR_INVALID_ARG;
    dbs_status st = noalloc_setup(dev);
    if (st != DBS_OK) return st;
    NoAllocDevice &d = g_noalloc_dev[dev];
    cudaStream_t s = (cudaStream_t)stream;
    // barrier state and counters must start at zero; the mask words are
    // fully rewritten by the kernel
    if (cudaMemsetAsync(d.scratch, 0, sizeof(Ctrl), s) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }

    KParams P{};
    P.m = (int32_t)A->m; P.n = (int32_t)A->n; P.nbr = (int32_t)A->nbr; P.nbc = (int32_t)A->nbc;
    P.B = (uint32_t)A->B; P.T = (uint32_t)A->T; P.valued = A->valued;
    P.rb_ptr = A->d_rb_ptr;
    P.blk_desc = reinterpret_cast<const uint2 *>(A->d_blk_desc);
    P.blk_ref = A->d_blk_ref;
    P.cb_ptr = A->d_cb_ptr;
    P.csc_desc = reinterpret_cast<const uint2 *>(A->d_csc_desc);
    P.csc_ref = A->d_csc_ref;
    P.payload = reinterpret_cast<const uint4 *>(A->d_payload);
    P.tiles = reinterpret_cast<const uint4 *>(A->d_tiles);
    P.rb_rows = A->d_rb_rows;
    P.ctrl = reinterpret_cast<Ctrl *>(d.scratch);
    P.dxm32 = reinterpret_cast<uint32_t *>(d.scratch + NOALLOC_CTRL_BYTES);
    P.path_force = DBS_PATH_PULL;          // the pull path needs no task lists
    P.x_in = x;
    P.xv = x;
    P.y_dense = y;
    dbs_exec_opts o;
    dbs_exec_opts_default(&o);
    P.th3 = o.th3;
    P.push_frac = o.push_work_frac;
    P.local_pull_min = o.local_pull_min;
    P.stats = 0;
    P.timeout_ns = o.wait_timeout_ns;
    return launch((const void *)k_spmspv_dense<false>, d.grid, P, s, SMEM0);
}
