// Host-side builder of the blocked dual-view matrix and the matrix part of the
// C ABI (build / destroy / info / export).
//
// DB-SpMSpV (Cong et al., ICPP '26):
//   Section 3.2.1 - 16x16 blocking, block-CSR + block-CSC views over one
//                   payload, low-level format by density (th0, th1) and
//                   directional skew (th2), patched CSR with row_idx_csc2csr;
//   Section 3.3.2 - load-weighted pull segments (Dense 4, Force/CSR 2, COO 1);
//   Section 5.5   - conversion is offline and reused across calls.
// The conversion runs once per matrix, on the host threads with one upload
// to HBM, or with device_convert on the GPU (build_gpu.cu); every later call
// runs on the GPU.  All device memory of the library is allocated here
// (dev_malloc / dev_free), which lets a build report its peak.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <unordered_map>

#include "internal.h"

using namespace dbs;

namespace {

struct Entry {
    uint64_t key;   // (col block << 8) | (local row << 4) | local col
    float val;
};

// One contiguous range of row blocks converted by one worker.
struct Chunk {
    int64_t rb0 = 0, rb1 = 0;
    std::vector<uint32_t> rb_count;   // blocks per row block
    std::vector<U2> desc;             // {col block, meta}
    std::vector<uint32_t> units;      // payload units per block
    std::vector<U4> payload;
    int error = DBS_OK;
};

inline int popc16(uint32_t v) { return __builtin_popcount(v & 0xFFFFu); }

// Low-level format class of one block (Section 3.2.1):
//   nnz < th0 -> COO, nnz > th1 -> Dense, otherwise the skew rule
//   skew_a = max_l n_l(a) / (nnz / 16 + eps); ForceCSC if skew_r / skew_c > th2,
//   ForceCSR if skew_c / skew_r > th2, patched CSR otherwise.
uint32_t classify(int nnz, int maxr, int maxc, const dbs_build_opts &o)
{
    if (nnz < o.th0) return FMT_COO;
    if (nnz > o.th1) return FMT_DENSE;
    const double eps = 1e-9;
    double skew_r = (double)maxr / ((double)nnz / (double)BS + eps);
    double skew_c = (double)maxc / ((double)nnz / (double)BS + eps);
    if (skew_r / skew_c > o.th2) return FMT_FCSC;
    if (skew_c / skew_r > o.th2) return FMT_FCSR;
    return FMT_PCSR;
}

// Encode one block's entries (sorted row-major: local row, then local col)
// into `out` (payload units, zero-initialized by the caller).
void encode_block(uint32_t fmt, const uint8_t *lr, const uint8_t *lc, const float *v, int nnz,
                  bool valued, uint8_t *out)
{
    const uint32_t voff = val_offset(fmt, (uint32_t)nnz);
    float *vals = reinterpret_cast<float *>(out + voff);
    int rcount[16] = {0}, ccount[16] = {0};
    for (int k = 0; k < nnz; ++k) { rcount[lr[k]]++; ccount[lc[k]]++; }
    int rptr[17] = {0}, cptr[17] = {0};
    for (int i = 0; i < 16; ++i) { rptr[i + 1] = rptr[i] + rcount[i]; cptr[i + 1] = cptr[i] + ccount[i]; }
    uint16_t rmask[16] = {0}, cmask[16] = {0};
    for (int k = 0; k < nnz; ++k) {
        rmask[lr[k]] |= (uint16_t)(1u << lc[k]);
        cmask[lc[k]] |= (uint16_t)(1u << lr[k]);
    }
    switch (fmt) {
    case FMT_COO:
        for (int k = 0; k < nnz; ++k) {
            out[k] = (uint8_t)((lr[k] << 4) | lc[k]);
            if (valued) vals[k] = v[k];
        }
        break;
    case FMT_DENSE:
        std::memcpy(out + dense_mask_off(valued), cmask, 32);
        if (valued)
            for (int k = 0; k < nnz; ++k) vals[lc[k] * 16 + lr[k]] = v[k];
        break;
    case FMT_FCSR:
        for (int i = 0; i < 16; ++i) out[OFF_PTR + i] = (uint8_t)rptr[i];
        std::memcpy(out + OFF_MASK, rmask, 32);
        if (valued)
            for (int k = 0; k < nnz; ++k) vals[k] = v[k];   // row-major = row order
        break;
    case FMT_FCSC: {
        for (int i = 0; i < 16; ++i) out[OFF_PTR + i] = (uint8_t)cptr[i];
        std::memcpy(out + OFF_MASK, cmask, 32);
        int fill[16] = {0};
        if (valued)
            for (int k = 0; k < nnz; ++k) vals[cptr[lc[k]] + fill[lc[k]]++] = v[k];
        break;
    }
    case FMT_PCSR: {
        for (int i = 0; i < 16; ++i) out[OFF_PTR + i] = (uint8_t)rptr[i];
        std::memcpy(out + OFF_MASK, rmask, 32);
        for (int i = 0; i < 16; ++i) out[OFF_PCOLPTR + i] = (uint8_t)cptr[i];
        int fill[16] = {0};
        for (int k = 0; k < nnz; ++k) {
            int off = k - rptr[lr[k]];                     // position inside its row
            out[OFF_RCSC + cptr[lc[k]] + fill[lc[k]]++] = (uint8_t)((lr[k] << 4) | off);
            if (valued) vals[k] = v[k];
        }
        break;
    }
    }
}

void convert_chunk(Chunk &ch, int64_t m, int64_t n, const int64_t *rp, const int32_t *ci,
                   const float *va, const dbs_build_opts &o, std::vector<Entry> &ents)
{
    const bool valued = va != nullptr;
    ch.rb_count.assign((size_t)(ch.rb1 - ch.rb0), 0);
    uint8_t lr[256], lc[256];
    float vv[256];
    for (int64_t rb = ch.rb0; rb < ch.rb1; ++rb) {
        int64_t r0 = rb * BS, r1 = std::min<int64_t>(m, r0 + BS);
        ents.clear();
        for (int64_t i = r0; i < r1; ++i) {
            for (int64_t k = rp[i]; k < rp[i + 1]; ++k) {
                int64_t c = ci[k];
                if (c < 0 || c >= n) { ch.error = DBS_ERR_INVALID_ARG; return; }
                uint64_t key = ((uint64_t)(c >> 4) << 8) | ((uint64_t)(i - r0) << 4) | (uint64_t)(c & 15);
                ents.push_back(Entry{key, valued ? va[k] : 0.0f});
            }
        }
        std::sort(ents.begin(), ents.end(), [](const Entry &a, const Entry &b) { return a.key < b.key; });
        size_t s = 0;
        while (s < ents.size()) {
            uint64_t cb = ents[s].key >> 8;
            size_t e = s;
            while (e < ents.size() && (ents[e].key >> 8) == cb) ++e;
            int nnz = (int)(e - s);
            int rc[16] = {0}, cc[16] = {0};
            uint32_t cm = 0;
            for (size_t t = s; t < e; ++t) {
                if (t > s && ents[t].key == ents[t - 1].key) { ch.error = DBS_ERR_INVALID_ARG; return; }
                lr[t - s] = (uint8_t)((ents[t].key >> 4) & 15);
                lc[t - s] = (uint8_t)(ents[t].key & 15);
                vv[t - s] = ents[t].val;
                rc[lr[t - s]]++;
                cc[lc[t - s]]++;
                cm |= 1u << lc[t - s];
            }
            int maxr = *std::max_element(rc, rc + 16), maxc = *std::max_element(cc, cc + 16);
            uint32_t fmt = o.force_format >= 0 ? (uint32_t)o.force_format : classify(nnz, maxr, maxc, o);
            if (fmt == FMT_COO && !valued && (uint32_t)nnz <= INLINE_MAX_NNZ) {
                // pattern-only COO block small enough to live in its meta word
                uint8_t coords[3];
                for (int k = 0; k < nnz; ++k) coords[k] = (uint8_t)((lr[k] << 4) | lc[k]);
                ch.desc.push_back(U2{(uint32_t)cb, meta_pack_inline(coords, (uint32_t)nnz)});
                ch.units.push_back(0);
                ch.rb_count[(size_t)(rb - ch.rb0)]++;
                s = e;
                continue;
            }
            uint32_t units = payload_units(fmt, (uint32_t)nnz, valued);
            size_t base = ch.payload.size();
            ch.payload.resize(base + units, U4{0, 0, 0, 0});
            encode_block(fmt, lr, lc, vv, nnz, valued, reinterpret_cast<uint8_t *>(&ch.payload[base]));
            ch.desc.push_back(U2{(uint32_t)cb, meta_pack(cm, fmt, (uint32_t)nnz)});
            ch.units.push_back(units);
            ch.rb_count[(size_t)(rb - ch.rb0)]++;
            s = e;
        }
    }
}

// Allocation-failure injection (dbs_debug_fail_alloc): the countdown to the
// allocation attempt that fails; -1 when off.
std::atomic<int64_t> g_fail_countdown{-1};

// Sizes of the live device allocations (dev_free), and the calling thread's
// build watch.
std::mutex g_alloc_mu;
std::unordered_map<void *, size_t> &alloc_sizes()
{
    static std::unordered_map<void *, size_t> sizes;
    return sizes;
}
thread_local MemWatch *t_watch = nullptr;

int num_sms_or_default()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
        return sms;
    cudaGetLastError();
    return 152;
}

// Pull tiles (Section 3.3.2, generalised): consecutive primary blocks are
// grouped until the accumulated weight reaches `W`; a tile never spans more
// than `R` row blocks.  With W = 16 and R = 1 these are exactly the paper's
// load-weighted row-block segments.
void build_tiles(const std::vector<uint32_t> &rb_ptr, const std::vector<U2> &desc, int64_t nbr,
                 uint32_t W, uint32_t R, std::vector<U4> &tiles)
{
    tiles.clear();
    uint32_t p0 = 0, rb0 = 0, w = 0, count = 0;
    auto close = [&](uint32_t p1, uint32_t rb_last) {
        tiles.push_back(U4{p0, p1, rb0, rb_last - rb0 + 1});
        count = 0;
        w = 0;
    };
    uint32_t last_rb = 0;
    for (int64_t rb = 0; rb < nbr; ++rb) {
        for (uint32_t p = rb_ptr[(size_t)rb]; p < rb_ptr[(size_t)rb + 1]; ++p) {
            if (count > 0 && (uint32_t)rb - rb0 + 1 > R) close(p, last_rb);
            if (count == 0) { p0 = p; rb0 = (uint32_t)rb; }
            w += fmt_weight(meta_fmt(desc[p].y));
            ++count;
            last_rb = (uint32_t)rb;
            if (w >= W || count + (p0 & 1u) >= TILE_MAX_BLOCKS) close(p + 1, last_rb);
        }
    }
    if (count > 0) close(rb_ptr[(size_t)nbr], last_rb);
}

template <class T>
dbs_status upload(const std::vector<T> &h, T **d, size_t min_elems, cudaStream_t s)
{
    size_t cnt = std::max(h.size(), min_elems);
    size_t bytes = std::max<size_t>(cnt * sizeof(T), 16);
    if (dev_malloc(d, bytes) != cudaSuccess) { cudaGetLastError(); *d = nullptr; return DBS_ERR_OOM; }
    if (cudaMemsetAsync(*d, 0, bytes, s) != cudaSuccess) return DBS_ERR_CUDA;
    if (!h.empty() && cudaMemcpyAsync(*d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DBS_ERR_CUDA;
    return DBS_OK;
}

void free_device(dbs_matrix *A)
{
    if (A->plan) dbs_spmv_plan_destroy(A->plan);
    dev_free(A->d_csr_rp); dev_free(A->d_csr_ci); dev_free(A->d_csr_va);
    A->plan = nullptr; A->d_csr_rp = nullptr; A->d_csr_ci = nullptr; A->d_csr_va = nullptr;
    dev_free(A->d_rb_ptr); dev_free(A->d_blk_desc); dev_free(A->d_blk_ref); dev_free(A->d_cb_ptr);
    dev_free(A->d_csc_desc); dev_free(A->d_csc_ref); dev_free(A->d_payload); dev_free(A->d_tiles);
    dev_free(A->d_rb_rows);
    A->d_rb_ptr = nullptr; A->d_blk_desc = nullptr; A->d_blk_ref = nullptr; A->d_cb_ptr = nullptr;
    A->d_csc_desc = nullptr; A->d_csc_ref = nullptr; A->d_payload = nullptr; A->d_tiles = nullptr;
    A->d_rb_rows = nullptr;
}

template <class T>
bool copy_from_device(std::vector<T> &h, const T *d, size_t cnt)
{
    h.resize(cnt);
    if (cnt == 0) return true;
    return cudaMemcpy(h.data(), d, cnt * sizeof(T), cudaMemcpyDeviceToHost) == cudaSuccess;
}

// A host view of the format: the kept copy, or a download of the device one.
dbs_status host_view(const dbs_matrix *A, HostFormat &tmp, const HostFormat **out)
{
    if (A->host) { *out = A->host; return DBS_OK; }
    if (!A->on_device) return DBS_ERR_INVALID_ARG;
    bool ok = copy_from_device(tmp.rb_ptr, A->d_rb_ptr, (size_t)A->nbr + 1) &&
              copy_from_device(tmp.blk_desc, A->d_blk_desc, (size_t)A->B) &&
              copy_from_device(tmp.blk_ref, A->d_blk_ref, (size_t)A->B) &&
              copy_from_device(tmp.cb_ptr, A->d_cb_ptr, (size_t)A->nbc + 1) &&
              copy_from_device(tmp.csc_desc, A->d_csc_desc, (size_t)A->B) &&
              copy_from_device(tmp.csc_ref, A->d_csc_ref, (size_t)A->B) &&
              copy_from_device(tmp.payload, A->d_payload, (size_t)A->P) &&
              copy_from_device(tmp.tiles, A->d_tiles, (size_t)A->T);
    if (!ok) { cudaGetLastError(); return DBS_ERR_CUDA; }
    *out = &tmp;
    return DBS_OK;
}

// The host conversion (Section 3.2.1) on the builder's threads, then one
// upload unless host_only.  Inputs are host arrays, or device arrays
// downloaded first.
dbs_status host_convert(dbs_matrix *A, const int64_t *row_ptr, const int32_t *col_idx, const float *vals,
                        bool inputs_on_device, const dbs_build_opts &o, cudaStream_t s)
{
    const int64_t m = A->m, n = A->n, nnz = A->nnz, nbr = A->nbr, nbc = A->nbc;
    HostFormat &H = *A->host;
    std::vector<int64_t> h_rp;
    std::vector<int32_t> h_ci;
    std::vector<float> h_va;
    const int64_t *rp = row_ptr;
    const int32_t *ci = col_idx;
    const float *va = vals;
    try {
        if (inputs_on_device) {
            host_alloc_point();
            h_rp.resize((size_t)m + 1);
            if (cudaMemcpy(h_rp.data(), row_ptr, sizeof(int64_t) * ((size_t)m + 1), cudaMemcpyDeviceToHost) != cudaSuccess) {
                cudaGetLastError();
                return DBS_ERR_CUDA;
            }
            rp = h_rp.data();
        }
    } catch (const std::bad_alloc &) {
        return DBS_ERR_OOM;
    }
    if (rp[0] != 0 || rp[m] != nnz) return DBS_ERR_INVALID_ARG;
    for (int64_t i = 0; i < m; ++i)
        if (rp[i + 1] < rp[i]) return DBS_ERR_INVALID_ARG;
    if (inputs_on_device) {
        try {
            h_ci.resize((size_t)nnz);
            if (vals) h_va.resize((size_t)nnz);
        } catch (const std::bad_alloc &) {
            return DBS_ERR_OOM;
        }
        if ((nnz && cudaMemcpy(h_ci.data(), col_idx, sizeof(int32_t) * (size_t)nnz, cudaMemcpyDeviceToHost) != cudaSuccess) ||
            (vals && nnz && cudaMemcpy(h_va.data(), vals, sizeof(float) * (size_t)nnz, cudaMemcpyDeviceToHost) != cudaSuccess)) {
            cudaGetLastError();
            return DBS_ERR_CUDA;
        }
        ci = h_ci.data();
        va = vals ? h_va.data() : nullptr;
    }

    try {
      {
        // 1. Row-block chunks converted in parallel.
        int nthreads = o.num_threads > 0 ? o.num_threads : (int)std::max(1u, std::thread::hardware_concurrency());
        const int64_t chunk_rb = std::max<int64_t>(1, std::min<int64_t>(4096, nbr / (int64_t)(8 * nthreads) + 1));
        std::vector<Chunk> chunks((size_t)((nbr + chunk_rb - 1) / chunk_rb));
        for (size_t c = 0; c < chunks.size(); ++c) {
            chunks[c].rb0 = (int64_t)c * chunk_rb;
            chunks[c].rb1 = std::min(nbr, chunks[c].rb0 + chunk_rb);
        }
        std::atomic<size_t> next{0};
        std::atomic<bool> oom{false};
        auto worker = [&]() {
            std::vector<Entry> ents;
            try {
                host_alloc_point();
                for (size_t c; (c = next.fetch_add(1)) < chunks.size();)
                    convert_chunk(chunks[c], m, n, rp, ci, va, o, ents);
            } catch (const std::bad_alloc &) {
                oom = true;
            }
        };
        std::vector<std::thread> pool;
        for (int t = 1; t < nthreads && (size_t)t < chunks.size(); ++t) pool.emplace_back(worker);
        worker();
        for (auto &t : pool) t.join();
        if (oom) return DBS_ERR_OOM;
        for (auto &c : chunks)
            if (c.error != DBS_OK) return (dbs_status)c.error;

        // 2. Concatenate: primary block order, payload offsets (a valued
        // Dense block starts on a 64-byte boundary).
        const bool valued_m = va != nullptr;
        auto aligned = [&](const U2 &d) { return valued_m && !meta_inline(d.y) && meta_fmt(d.y) == FMT_DENSE; };
        auto align_up = [](int64_t u) { return (u + DENSE_ALIGN_UNITS - 1) / DENSE_ALIGN_UNITS * DENSE_ALIGN_UNITS; };
        int64_t B = 0, P = 0;
        for (auto &c : chunks) {
            B += (int64_t)c.desc.size();
            for (size_t i = 0; i < c.units.size(); ++i) {
                if (aligned(c.desc[i])) P = align_up(P);
                P += c.units[i];
            }
        }
        if (B >= (int64_t(1) << 32) || P >= (int64_t(1) << 32)) return DBS_ERR_UNSUPPORTED;
        A->B = B; A->P = P;
        host_alloc_point();
        H.rb_ptr.resize((size_t)nbr + 1);
        H.blk_desc.resize((size_t)B);
        H.blk_ref.resize((size_t)B);
        H.payload.resize((size_t)P);
        {
            uint32_t pb = 0, pu = 0;
            H.rb_ptr[0] = 0;
            for (auto &c : chunks) {
                for (size_t i = 0; i < c.rb_count.size(); ++i)
                    H.rb_ptr[(size_t)c.rb0 + i + 1] = H.rb_ptr[(size_t)c.rb0 + i] + c.rb_count[i];
                std::copy(c.desc.begin(), c.desc.end(), H.blk_desc.begin() + pb);
                size_t lo = 0;
                for (size_t i = 0; i < c.units.size(); ++i) {
                    if (aligned(c.desc[i])) pu = (uint32_t)align_up(pu);
                    std::copy(c.payload.begin() + lo, c.payload.begin() + lo + c.units[i], H.payload.begin() + pu);
                    H.blk_ref[pb + i] = pu;
                    pu += c.units[i];
                    lo += c.units[i];
                }
                pb += (uint32_t)c.desc.size();
                std::vector<U2>().swap(c.desc);
                std::vector<U4>().swap(c.payload);
            }
        }
      }
      const int64_t B = A->B;

        // 3. Block-CSC view: counting sort of primary blocks by column block;
        //    row blocks stay ascending within a column block.
        host_alloc_point();
        H.cb_ptr.assign((size_t)nbc + 1, 0);
        for (int64_t p = 0; p < B; ++p) H.cb_ptr[H.blk_desc[(size_t)p].x + 1]++;
        for (int64_t c = 0; c < nbc; ++c) H.cb_ptr[(size_t)c + 1] += H.cb_ptr[(size_t)c];
        H.csc_desc.resize((size_t)B);
        H.csc_ref.resize((size_t)B);
        {
            std::vector<uint32_t> fill(H.cb_ptr.begin(), H.cb_ptr.end() - 1);
            for (int64_t rb = 0; rb < nbr; ++rb)
                for (uint32_t p = H.rb_ptr[(size_t)rb]; p < H.rb_ptr[(size_t)rb + 1]; ++p) {
                    uint32_t q = fill[H.blk_desc[p].x]++;
                    H.csc_desc[q] = U2{(uint32_t)rb, H.blk_desc[p].y};
                    H.csc_ref[q] = H.blk_ref[p];
                }
        }

        // Rows that hold an entry, per row block (a row without one can
        // never be reached or touched).
        H.rb_rows.assign((size_t)nbr, 0);
        for (int64_t i = 0; i < m; ++i)
            if (rp[i + 1] > rp[i]) H.rb_rows[(size_t)(i / BS)] |= (uint16_t)(1u << (i % BS));

        // 4. Pull tiles.
        uint64_t total_w = 0;
        for (int64_t p = 0; p < B; ++p) total_w += fmt_weight(meta_fmt(H.blk_desc[(size_t)p].y));
        const uint32_t W = tile_weight_cap(o, total_w);
        uint32_t R = o.tile_max_row_blocks > 0 ? (uint32_t)o.tile_max_row_blocks : TILE_MAX_SPAN;
        host_alloc_point();
        build_tiles(H.rb_ptr, H.blk_desc, nbr, W, R, H.tiles);
        A->T = (int64_t)H.tiles.size();
        for (size_t i = 0; i < H.tiles.size(); ++i) {
            // local row block of each block into blk_desc.x bits 27-31; flags
            // for row blocks shared with the neighbouring tiles
            U4 &tl = H.tiles[i];
            uint32_t rb = tl.z;
            for (uint32_t p = tl.x; p < tl.y; ++p) {
                while (H.rb_ptr[rb + 1] <= p) ++rb;
                H.blk_desc[p].x |= (rb - tl.z) << DESC_LRB_SHIFT;
            }
            if (H.rb_ptr[tl.z] < tl.x) tl.w |= TILE_FIRST_SHARED;
            if (H.rb_ptr[tl.z + (tl.w & TILE_SPAN_MASK)] > tl.y) tl.w |= TILE_LAST_SHARED;
            // kernel form: the block count joins w, the payload offset of
            // the first block replaces the end index
            tl.w |= (tl.y - tl.x) << TILE_NBLK_SHIFT;
            tl.y = tl.x < (uint32_t)B ? H.blk_ref[tl.x] : 0u;
        }
        // the pull kernel's copy and queue bounds rely on these
        {
            uint64_t next = 0;
            for (const U4 &tl : H.tiles) {
                const uint32_t nb = tl.w >> TILE_NBLK_SHIFT, span = tl.w & TILE_SPAN_MASK;
                if (tl.x != next || nb == 0 || (tl.x & 1u) + nb > TILE_MAX_BLOCKS || span == 0 ||
                    span > TILE_MAX_SPAN || (int64_t)tl.z + span > nbr)
                    return DBS_ERR_INTERNAL;
                next += nb;
            }
            if (next != (uint64_t)B) return DBS_ERR_INTERNAL;
        }
    } catch (const std::bad_alloc &) {
        return DBS_ERR_OOM;
    }


    dbs_matrix_info &I = A->info;
    for (int64_t p = 0; p < A->B; ++p) {
        uint32_t meta = H.blk_desc[(size_t)p].y;
        I.blocks_by_format[meta_fmt(meta)] += 1;
        I.nnz_by_format[meta_fmt(meta)] += meta_nnz(meta);
    }

    // Upload.
    if (!o.host_only) {
        if (cudaGetDevice(&A->device) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
        dbs_status st;
        if ((st = upload(H.rb_ptr, &A->d_rb_ptr, 1, s)) != DBS_OK) return st;
        // blk_desc is padded with 8 zero entries so vector loads may run past B.
        if ((st = upload(H.blk_desc, &A->d_blk_desc, (size_t)A->B + 8, s)) != DBS_OK) return st;
        if ((st = upload(H.blk_ref, &A->d_blk_ref, (size_t)A->B + 8, s)) != DBS_OK) return st;
        if ((st = upload(H.cb_ptr, &A->d_cb_ptr, 1, s)) != DBS_OK) return st;
        if ((st = upload(H.csc_desc, &A->d_csc_desc, (size_t)A->B + 8, s)) != DBS_OK) return st;
        if ((st = upload(H.csc_ref, &A->d_csc_ref, (size_t)A->B + 8, s)) != DBS_OK) return st;
        if ((st = upload(H.payload, &A->d_payload, 1, s)) != DBS_OK) return st;
        if ((st = upload(H.tiles, &A->d_tiles, 1, s)) != DBS_OK) return st;
        if ((st = upload(H.rb_rows, &A->d_rb_rows, (size_t)nbr + 2, s)) != DBS_OK) return st;
        if (cudaStreamSynchronize(s) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
        A->on_device = true;
    }
    return DBS_OK;
}

}  // namespace

bool dbs::alloc_fault()
{
    int64_t v = g_fail_countdown.load(std::memory_order_relaxed);
    while (v >= 0)
        if (g_fail_countdown.compare_exchange_weak(v, v - 1)) return v == 0;
    return false;
}

void dbs::host_alloc_point()
{
    if (alloc_fault()) throw std::bad_alloc();
}

cudaError_t dbs::dev_malloc_bytes(void **p, size_t bytes)
{
    *p = nullptr;
    if (alloc_fault()) return cudaErrorMemoryAllocation;
    void *q = nullptr;
    const cudaError_t e = cudaMalloc(&q, bytes);
    if (e != cudaSuccess) return e;
    try {
        std::lock_guard<std::mutex> g(g_alloc_mu);
        alloc_sizes()[q] = bytes;
    } catch (...) {
        cudaFree(q);
        return cudaErrorMemoryAllocation;
    }
    if (t_watch) {
        t_watch->live += (int64_t)bytes;
        t_watch->peak = std::max(t_watch->peak, t_watch->live);
    }
    *p = q;
    return cudaSuccess;
}

void dbs::dev_free(void *p)
{
    if (!p) return;
    size_t bytes = 0;
    {
        std::lock_guard<std::mutex> g(g_alloc_mu);
        auto &sizes = alloc_sizes();
        auto it = sizes.find(p);
        if (it != sizes.end()) {
            bytes = it->second;
            sizes.erase(it);
        }
    }
    cudaFree(p);
    if (t_watch) t_watch->live -= (int64_t)bytes;
}

void dbs::mem_watch(MemWatch *w) { t_watch = w; }

uint32_t dbs::tile_weight_cap(const dbs_build_opts &o, uint64_t total_weight)
{
    uint32_t W = (uint32_t)o.tile_weight;
    if (W == 0) {
        // about 64 tiles per SM, within [16, TILE_MAX_BLOCKS]
        const uint64_t target = (uint64_t)num_sms_or_default() * 64u;
        W = (uint32_t)std::min<uint64_t>(TILE_MAX_BLOCKS, std::max<uint64_t>(16, (total_weight + target - 1) / target));
    }
    return std::min<uint32_t>(W, TILE_MAX_BLOCKS);
}

extern "C" {

dbs_status dbs_debug_fail_alloc(int64_t k, int64_t *previous)
{
    const int64_t prev = g_fail_countdown.exchange(k < 0 ? -1 : k);
    if (previous) *previous = prev;
    return DBS_OK;
}

void dbs_build_opts_default(dbs_build_opts *o)
{
    if (!o) return;
    o->th0 = 32;
    o->th1 = 128;
    o->th2 = 2.0;
    o->force_format = DBS_FMT_AUTO;
    o->tile_weight = 0;
    o->tile_max_row_blocks = 0;
    o->keep_host = 0;
    o->host_only = 0;
    o->num_threads = 0;
    o->device_convert = 0;
    o->dense_spmv = 0;
}

const char *dbs_status_string(dbs_status s)
{
    switch (s) {
    case DBS_OK: return "DBS_OK";
    case DBS_ERR_INVALID_ARG: return "DBS_ERR_INVALID_ARG";
    case DBS_ERR_OOM: return "DBS_ERR_OOM";
    case DBS_ERR_CUDA: return "DBS_ERR_CUDA";
    case DBS_ERR_TIMEOUT: return "DBS_ERR_TIMEOUT";
    case DBS_ERR_UNSUPPORTED: return "DBS_ERR_UNSUPPORTED";
    case DBS_ERR_INTERNAL: return "DBS_ERR_INTERNAL";
    }
    return "DBS_ERR_UNKNOWN";
}

const char *dbs_version(void) { return "dbspmspv 0.1 sm_103a"; }

dbs_status dbs_matrix_build_csr(int64_t m, int64_t n, int64_t nnz, const int64_t *row_ptr,
                                const int32_t *col_idx, const float *vals, int inputs_on_device,
                                const dbs_build_opts *opts_in, void *stream, dbs_matrix **out)
{
    if (!out || !row_ptr || (nnz > 0 && !col_idx)) return DBS_ERR_INVALID_ARG;
    if (m < 0 || n < 0 || m >= (int64_t(1) << 31) || n >= (int64_t(1) << 31) || nnz < 0)
        return DBS_ERR_INVALID_ARG;
    dbs_build_opts o;
    if (opts_in) o = *opts_in; else dbs_build_opts_default(&o);
    if (o.th0 < 0 || o.th1 < 0 || !(o.th2 > 0.0) || o.force_format < -1 || o.force_format >= DBS_NUM_FORMATS ||
        o.tile_weight < 0 || o.tile_max_row_blocks < 0 || o.tile_max_row_blocks > (int)TILE_MAX_SPAN ||
        o.num_threads < 0 || o.dense_spmv < 0 || o.dense_spmv > 1)
        return DBS_ERR_INVALID_ARG;
    if (inputs_on_device && o.host_only) return DBS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    auto t_start = std::chrono::steady_clock::now();
    // the build's own device allocations, for build_peak_bytes
    MemWatch watch;
    mem_watch(&watch);
    struct Unwatch {
        ~Unwatch() { mem_watch(nullptr); }
    } unwatch;

    const int64_t nbr = (m + BS - 1) / BS, nbc = (n + BS - 1) / BS;
    const bool valued = vals != nullptr;
    dbs_matrix *A = nullptr;
    try {
        host_alloc_point();
        A = new dbs_matrix();
        A->host = new HostFormat();
    } catch (const std::bad_alloc &) {
        delete A;
        return DBS_ERR_OOM;
    }
    A->m = m; A->n = n; A->nnz = nnz; A->nbr = nbr; A->nbc = nbc; A->valued = valued;
    HostFormat &H = *A->host;
    dbs_matrix_info &I = A->info;
    auto fail = [&](dbs_status st) { free_device(A); delete A->host; delete A; return st; };

    bool on_gpu = inputs_on_device && o.device_convert;
    if (on_gpu) {
        // the whole conversion on the device (Section 3.2.1 without a sort)
        DeviceFormat D;
        bool fallback = false;
        const dbs_status st = device_convert(m, n, nnz, row_ptr, col_idx, vals, o, s, &D, &fallback);
        if (st != DBS_OK) return fail(st);
        if (fallback) {
            on_gpu = false;                 // a row's columns are not ascending: host conversion
        } else {
            if (cudaGetDevice(&A->device) != cudaSuccess) {
                cudaGetLastError();
                for (void *q : {(void *)D.rb_ptr, (void *)D.blk_desc, (void *)D.blk_ref, (void *)D.cb_ptr,
                                (void *)D.csc_desc, (void *)D.csc_ref, (void *)D.payload, (void *)D.tiles,
                                (void *)D.rb_rows})
                    dev_free(q);
                return fail(DBS_ERR_CUDA);
            }
            A->d_rb_ptr = D.rb_ptr; A->d_blk_desc = D.blk_desc; A->d_blk_ref = D.blk_ref; A->d_cb_ptr = D.cb_ptr;
            A->d_csc_desc = D.csc_desc; A->d_csc_ref = D.csc_ref; A->d_payload = D.payload; A->d_tiles = D.tiles;
            A->d_rb_rows = D.rb_rows;
            A->B = D.B; A->P = D.P; A->T = D.T;
            A->on_device = true;
            for (int f = 0; f < DBS_NUM_FORMATS; ++f) {
                I.blocks_by_format[f] = D.blocks_by_format[f];
                I.nnz_by_format[f] = D.nnz_by_format[f];
            }
        }
    }

    if (!on_gpu) {
        dbs_status st = host_convert(A, row_ptr, col_idx, vals, inputs_on_device != 0, o, s);
        if (st != DBS_OK) return fail(st);
    }

    // Info (Table 4 style storage report).
    I.m = m; I.n = n; I.nnz = nnz; I.nbr = nbr; I.nbc = nbc; I.nblocks = A->B;
    I.ntiles = A->T;
    I.payload_bytes = A->P * 16;
    I.view_bytes = (nbr + 1) * 4 + A->B * 8 + A->B * 4 + (nbc + 1) * 4 + A->B * 8 + A->B * 4 + A->T * 16 +
                   nbr * 2;   // + per row block: rows holding entries
    I.total_bytes = I.payload_bytes + I.view_bytes;
    I.csr_bytes = (m + 1) * 4 + nnz * 4 + (valued ? nnz * 4 : 0);
    I.csr_csc_bytes = I.csr_bytes + (n + 1) * 4 + nnz * 4 + (valued ? nnz * 4 : 0);
    I.valued = valued ? 1 : 0;

    if (A->on_device && o.dense_spmv && valued) {
        // the input CSR, kept on the device for dense-x calls, and its plan
        const size_t rb = sizeof(int64_t) * ((size_t)m + 1), cb = sizeof(int32_t) * (size_t)std::max<int64_t>(nnz, 1),
                     vb = sizeof(float) * (size_t)std::max<int64_t>(nnz, 1);
        if (dev_malloc(&A->d_csr_rp, rb) != cudaSuccess || dev_malloc(&A->d_csr_ci, cb) != cudaSuccess ||
            dev_malloc(&A->d_csr_va, vb) != cudaSuccess) {
            cudaGetLastError();
            return fail(DBS_ERR_OOM);
        }
        if (cudaMemcpy(A->d_csr_rp, row_ptr, rb, cudaMemcpyDefault) != cudaSuccess ||
            (nnz && cudaMemcpy(A->d_csr_ci, col_idx, sizeof(int32_t) * (size_t)nnz, cudaMemcpyDefault) != cudaSuccess) ||
            (nnz && cudaMemcpy(A->d_csr_va, vals, sizeof(float) * (size_t)nnz, cudaMemcpyDefault) != cudaSuccess)) {
            cudaGetLastError();
            return fail(DBS_ERR_CUDA);
        }
        dbs_status st2 = dbs_spmv_plan_create(m, n, nnz, A->d_csr_rp, A->d_csr_ci, A->d_csr_va, stream, &A->plan);
        if (st2 != DBS_OK) { A->plan = nullptr; return fail(st2); }
        I.spmv_bytes = (int64_t)(rb + (size_t)nnz * 8) + spmv_plan_bytes(A->plan);
    }
    I.on_device = A->on_device ? 1 : 0;
    if (on_gpu && o.keep_host) {
        // the host copy of a device conversion: every array downloaded
        bool ok = false;
        try {
            host_alloc_point();
            ok = copy_from_device(H.rb_ptr, A->d_rb_ptr, (size_t)nbr + 1) &&
                 copy_from_device(H.blk_desc, A->d_blk_desc, (size_t)A->B) &&
                 copy_from_device(H.blk_ref, A->d_blk_ref, (size_t)A->B) &&
                 copy_from_device(H.cb_ptr, A->d_cb_ptr, (size_t)nbc + 1) &&
                 copy_from_device(H.csc_desc, A->d_csc_desc, (size_t)A->B) &&
                 copy_from_device(H.csc_ref, A->d_csc_ref, (size_t)A->B) &&
                 copy_from_device(H.payload, A->d_payload, (size_t)A->P) &&
                 copy_from_device(H.tiles, A->d_tiles, (size_t)A->T) &&
                 copy_from_device(H.rb_rows, A->d_rb_rows, (size_t)nbr);
        } catch (const std::bad_alloc &) {
            return fail(DBS_ERR_OOM);
        }
        if (!ok) { cudaGetLastError(); return fail(DBS_ERR_CUDA); }
    }
    if (!o.keep_host && !o.host_only) { delete A->host; A->host = nullptr; }
    I.build_peak_bytes = watch.peak;
    I.build_seconds = std::chrono::duration<double>(std::chrono::steady_clock::now() - t_start).count();
    *out = A;
    return DBS_OK;
}

dbs_status dbs_matrix_destroy(dbs_matrix *A)
{
    if (!A) return DBS_OK;
    free_device(A);
    delete A->host;
    delete A;
    return DBS_OK;
}

dbs_status dbs_matrix_info_get(const dbs_matrix *A, dbs_matrix_info *out)
{
    if (!A || !out) return DBS_ERR_INVALID_ARG;
    *out = A->info;
    return DBS_OK;
}

dbs_status dbs_matrix_export_views(const dbs_matrix *A, int64_t *blk_row_ptr, int64_t *blk_col_idx,
                                   int64_t *blk_col_ptr, int64_t *blk_row_idx, int64_t *blk_csc2csr,
                                   int32_t *blk_nnz, int32_t *blk_format)
{
    if (!A) return DBS_ERR_INVALID_ARG;
    HostFormat tmp;
    const HostFormat *H = nullptr;
    try {
        dbs_status st = host_view(A, tmp, &H);
        if (st != DBS_OK) return st;
        if (blk_row_ptr) for (int64_t i = 0; i <= A->nbr; ++i) blk_row_ptr[i] = H->rb_ptr[(size_t)i];
        if (blk_col_ptr) for (int64_t i = 0; i <= A->nbc; ++i) blk_col_ptr[i] = H->cb_ptr[(size_t)i];
        for (int64_t p = 0; p < A->B; ++p) {
            if (blk_col_idx) blk_col_idx[p] = H->blk_desc[(size_t)p].x & DESC_COL_MASK;
            if (blk_nnz) blk_nnz[p] = (int32_t)meta_nnz(H->blk_desc[(size_t)p].y);
            if (blk_format) blk_format[p] = (int32_t)meta_fmt(H->blk_desc[(size_t)p].y);
            if (blk_row_idx) blk_row_idx[p] = H->csc_desc[(size_t)p].x;
        }
        if (blk_csc2csr) {
            // The CSC position q of column block c holding row block r maps to
            // the primary block (r, c): search row block r's column indices.
            for (int64_t c = 0; c < A->nbc; ++c)
                for (uint32_t q = H->cb_ptr[(size_t)c]; q < H->cb_ptr[(size_t)c + 1]; ++q) {
                    const uint32_t r = H->csc_desc[q].x;
                    auto b0 = H->blk_desc.begin() + H->rb_ptr[r], b1 = H->blk_desc.begin() + H->rb_ptr[r + 1];
                    auto it = std::lower_bound(b0, b1, (uint32_t)c,
                                               [](const U2 &d, uint32_t v) { return (d.x & DESC_COL_MASK) < v; });
                    if (it == b1 || (it->x & DESC_COL_MASK) != (uint32_t)c) return DBS_ERR_INTERNAL;
                    const size_t p = (size_t)(it - H->blk_desc.begin());
                    if (H->csc_ref[q] != H->blk_ref[p] || H->csc_desc[q].y != it->y) return DBS_ERR_INTERNAL;
                    blk_csc2csr[q] = (int64_t)p;
                }
        }
    } catch (const std::bad_alloc &) {
        return DBS_ERR_OOM;
    }
    return DBS_OK;
}

dbs_status dbs_matrix_export_raw(const dbs_matrix *A, int32_t which, void *dst, int64_t capacity, int64_t *bytes)
{
    if (!A || !bytes || which < 0 || which >= DBS_RAW_COUNT) return DBS_ERR_INVALID_ARG;
    const size_t B = (size_t)A->B, nbr = (size_t)A->nbr, nbc = (size_t)A->nbc;
    const HostFormat *H = A->host;
    const void *dsrc = nullptr, *hsrc = nullptr;
    size_t size = 0;
    switch (which) {
    case DBS_RAW_RB_PTR: size = (nbr + 1) * 4; dsrc = A->d_rb_ptr; hsrc = H ? H->rb_ptr.data() : nullptr; break;
    case DBS_RAW_BLK_DESC: size = B * 8; dsrc = A->d_blk_desc; hsrc = H ? H->blk_desc.data() : nullptr; break;
    case DBS_RAW_BLK_REF: size = B * 4; dsrc = A->d_blk_ref; hsrc = H ? H->blk_ref.data() : nullptr; break;
    case DBS_RAW_CB_PTR: size = (nbc + 1) * 4; dsrc = A->d_cb_ptr; hsrc = H ? H->cb_ptr.data() : nullptr; break;
    case DBS_RAW_CSC_DESC: size = B * 8; dsrc = A->d_csc_desc; hsrc = H ? H->csc_desc.data() : nullptr; break;
    case DBS_RAW_CSC_REF: size = B * 4; dsrc = A->d_csc_ref; hsrc = H ? H->csc_ref.data() : nullptr; break;
    case DBS_RAW_PAYLOAD: size = (size_t)A->P * 16; dsrc = A->d_payload; hsrc = H ? H->payload.data() : nullptr; break;
    case DBS_RAW_TILES: size = (size_t)A->T * 16; dsrc = A->d_tiles; hsrc = H ? H->tiles.data() : nullptr; break;
    default: size = nbr * 2; dsrc = A->d_rb_rows; hsrc = H ? H->rb_rows.data() : nullptr; break;
    }
    *bytes = (int64_t)size;
    if (!dst) return DBS_OK;
    if (capacity < (int64_t)size) return DBS_ERR_INVALID_ARG;
    if (size == 0) return DBS_OK;
    if (A->on_device) {
        if (cudaMemcpy(dst, dsrc, size, cudaMemcpyDeviceToHost) != cudaSuccess) { cudaGetLastError(); return DBS_ERR_CUDA; }
    } else {
        if (!hsrc) return DBS_ERR_INVALID_ARG;
        std::memcpy(dst, hsrc, size);
    }
    return DBS_OK;
}

dbs_status dbs_matrix_export_csr(const dbs_matrix *A, int64_t *row_ptr, int32_t *col_idx, float *vals)
{
    if (!A || !row_ptr || (A->nnz > 0 && !col_idx)) return DBS_ERR_INVALID_ARG;
    if (vals && !A->valued) return DBS_ERR_INVALID_ARG;
    HostFormat tmp;
    const HostFormat *H = nullptr;
    try {
        dbs_status st = host_view(A, tmp, &H);
        if (st != DBS_OK) return st;
        const uint8_t *pay = reinterpret_cast<const uint8_t *>(H->payload.data());
        // pass 1: entries per row; pass 2: fill.
        std::vector<int64_t> cnt((size_t)A->m + 1, 0);
        auto for_each_entry = [&](auto &&emit) -> bool {
            for (int64_t rb = 0; rb < A->nbr; ++rb)
                for (uint32_t p = H->rb_ptr[(size_t)rb]; p < H->rb_ptr[(size_t)rb + 1]; ++p) {
                    const uint32_t meta = H->blk_desc[p].y, fmt = meta_fmt(meta), nnz = meta_nnz(meta);
                    const uint32_t cb = H->blk_desc[p].x & DESC_COL_MASK;
                    uint8_t inl[4] = {(uint8_t)(meta & 0xFF), (uint8_t)((meta >> 8) & 0xFF),
                                      (uint8_t)((meta >> 16) & 0xFF), 0};
                    const uint8_t *b = meta_inline(meta) ? inl : pay + (size_t)H->blk_ref[p] * 16;
                    const float *v = reinterpret_cast<const float *>(b + val_offset(fmt, nnz));
                    uint16_t mask[16] = {0};
                    if (fmt != FMT_COO)
                        std::memcpy(mask, b + (fmt == FMT_DENSE ? dense_mask_off(A->valued) : OFF_MASK), 32);
                    uint32_t found = 0;
                    for (int r = 0; r < 16; ++r) {
                        for (int c = 0; c < 16; ++c) {
                            bool present = false;
                            float x = 0.0f;
                            if (fmt == FMT_COO) {
                                for (uint32_t k = 0; k < nnz; ++k)
                                    if (b[k] == ((r << 4) | c)) { present = true; x = A->valued ? v[k] : 0.0f; }
                            } else if (fmt == FMT_DENSE || fmt == FMT_FCSC) {
                                present = (mask[c] >> r) & 1;
                                if (present && A->valued)
                                    x = fmt == FMT_DENSE ? v[c * 16 + r]
                                                         : v[b[OFF_PTR + c] + popc16(mask[c] & ((1u << r) - 1u))];
                            } else {
                                present = (mask[r] >> c) & 1;
                                if (present && A->valued) x = v[b[OFF_PTR + r] + popc16(mask[r] & ((1u << c) - 1u))];
                                if (present && fmt == FMT_PCSR) {
                                    // the column view must reach the same value slot
                                    const uint8_t *cp = b + OFF_PCOLPTR;
                                    uint32_t end = c == 15 ? nnz : cp[c + 1];
                                    bool ok = false;
                                    for (uint32_t k = cp[c]; k < end; ++k) {
                                        uint32_t e = b[OFF_RCSC + k];
                                        if ((int)(e >> 4) == r &&
                                            (int)(e & 15) == popc16(mask[r] & ((1u << c) - 1u))) ok = true;
                                    }
                                    if (!ok) return false;
                                }
                            }
                            if (present) {
                                ++found;
                                int64_t row = rb * 16 + r, col = (int64_t)cb * 16 + c;
                                if (row >= A->m || col >= A->n) return false;
                                emit(row, (int32_t)col, x);
                            }
                        }
                    }
                    if (found != nnz) return false;
                }
            return true;
        };
        if (!for_each_entry([&](int64_t row, int32_t, float) { cnt[(size_t)row + 1]++; })) return DBS_ERR_INTERNAL;
        row_ptr[0] = 0;
        for (int64_t i = 0; i < A->m; ++i) row_ptr[i + 1] = row_ptr[i] + cnt[(size_t)i + 1];
        if (row_ptr[A->m] != A->nnz) return DBS_ERR_INTERNAL;
        std::vector<int64_t> fill(row_ptr, row_ptr + A->m);
        for_each_entry([&](int64_t row, int32_t col, float x) {
            int64_t k = fill[(size_t)row]++;
            col_idx[k] = col;
            if (vals) vals[k] = x;
        });
    } catch (const std::bad_alloc &) {
        return DBS_ERR_OOM;
    }
    return DBS_OK;
}

}  // extern "C"
