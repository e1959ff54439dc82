// Blocked dual-view format shared by the host builder and the CUDA kernels.
//
// DB-SpMSpV (Cong et al., ICPP '26), Section 3.2.1 and Figure 5(b): the matrix
// is cut into 16x16 blocks; a high-level block-CSR view and a block-CSC view
// both reach one low-level payload per nonzero block, stored once in primary
// (block-CSR) order.
//
// Device arrays of a built matrix (B = nonzero blocks, P = payload units):
//   rb_ptr   u32[nbr+1]   block-CSR row-block pointers
//   blk_desc uint2[B]     per primary block: {column block, meta}
//   blk_ref  u32[B]       per primary block: payload offset in 16-byte units
//   cb_ptr   u32[nbc+1]   block-CSC column-block pointers
//   csc_desc uint2[B]     per CSC position: {row block, meta}
//   csc_ref  u32[B]       per CSC position: payload offset of the same block.
//                         This is the paper's csc2csr mapping resolved to the
//                         shared payload, so push reaches a block in one load.
//   payload  uint4[P]     the low-level blocks, 16-byte aligned
//   tiles    uint4[T]     pull work units {p0, p1, rb0, span} (Section 3.3.2)
//
// meta word: bits 0-15 column-occupancy mask of the block (bit c = local
// column c holds an entry), bits 16-18 format, bits 24-31 nnz - 1.
//
// Payload layouts (bytes from the 16-byte aligned start; bit k of a row mask
// is local column k, bit k of a column mask is local row k, as in Figure 5's
// "row_mask 10 = 0b1010 -> columns 1 and 3"):
//   COO         coord u8[nnz] (row << 4 | col, row-major order), values at align4(nnz)
//   Dense       col_mask u16[16] at 0, values f32[256] column-major (v[c*16+r]) at 32;
//               absent entries hold 0 and are excluded through col_mask
//   ForceCSR    row_ptr u8[16] at 0, row_mask u16[16] at 16, values in row order at 48
//   ForceCSC    col_ptr u8[16] at 0, col_mask u16[16] at 16, values in column order at 48
//   PatchedCSR  row_ptr u8[16] at 0, row_mask u16[16] at 16, col_ptr u8[16] at 48,
//               rcsc u8[nnz] at 64 (column order; row << 4 | offset of the entry within
//               its row), values in row order at align4(64 + nnz)
// Pattern-only matrices store the same structure without values.  Every
// payload is padded to a multiple of 16 bytes.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define DBS_HD __host__ __device__ __forceinline__
#else
#define DBS_HD inline
#endif

namespace dbs {

constexpr int BS = 16;
constexpr uint32_t FMT_COO = 0, FMT_DENSE = 1, FMT_FCSR = 2, FMT_FCSC = 3, FMT_PCSR = 4;

// Pull tiles: at most this many blocks (one CTA pass of 256 threads x 8) and
// this many row blocks (shared-memory row accumulators).
constexpr uint32_t TILE_MAX_BLOCKS = 2048;
constexpr uint32_t TILE_MAX_SPAN = 64;
// Push tasks: CSC positions per work item (one warp, one position per lane).
constexpr uint32_t PUSH_CHUNK = 32;

DBS_HD uint32_t meta_pack(uint32_t cmask, uint32_t fmt, uint32_t nnz)
{
    return (cmask & 0xFFFFu) | (fmt << 16) | ((nnz - 1u) << 24);
}
DBS_HD uint32_t meta_cmask(uint32_t m) { return m & 0xFFFFu; }
DBS_HD uint32_t meta_fmt(uint32_t m) { return (m >> 16) & 7u; }
DBS_HD uint32_t meta_nnz(uint32_t m) { return (m >> 24) + 1u; }

// Section 3.3.2: Dense 4, ForceCSR / ForceCSC / (patched) CSR 2, COO 1.
DBS_HD uint32_t fmt_weight(uint32_t fmt)
{
    return fmt == FMT_DENSE ? 4u : (fmt == FMT_COO ? 1u : 2u);
}

DBS_HD uint32_t struct_bytes(uint32_t fmt, uint32_t nnz)
{
    return fmt == FMT_COO ? nnz : fmt == FMT_DENSE ? 32u : fmt == FMT_PCSR ? 64u + nnz : 48u;
}
DBS_HD uint32_t val_offset(uint32_t fmt, uint32_t nnz) { return (struct_bytes(fmt, nnz) + 3u) & ~3u; }
DBS_HD uint32_t val_count(uint32_t fmt, uint32_t nnz) { return fmt == FMT_DENSE ? 256u : nnz; }
DBS_HD uint32_t payload_bytes(uint32_t fmt, uint32_t nnz, bool valued)
{
    return val_offset(fmt, nnz) + (valued ? 4u * val_count(fmt, nnz) : 0u);
}
DBS_HD uint32_t payload_units(uint32_t fmt, uint32_t nnz, bool valued)
{
    return (payload_bytes(fmt, nnz, valued) + 15u) >> 4;
}

// Offsets of the structural arrays.
constexpr uint32_t OFF_PTR = 0;        // row_ptr (ForceCSR, patched) or col_ptr (ForceCSC)
constexpr uint32_t OFF_MASK = 16;      // row_mask / col_mask (Force*, patched)
constexpr uint32_t OFF_PCOLPTR = 48;   // patched CSR col_ptr
constexpr uint32_t OFF_RCSC = 64;      // patched CSR row_idx_csc2csr bytes

}  // namespace dbs
