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
//   tiles    uint4[T]     pull work units {p0, payload offset, rb0, span | flags | count} (Section 3.3.2)
//
// blk_desc.x holds the column block in bits 0-26 and, in bits 27-31, the
// block's row block relative to the first row block of its pull tile, so a
// pull task needs no row-block search.
//
// meta word (the same word in both views):
//   stored block:  bits 0-15 column-occupancy mask (bit c = local column c
//                  holds an entry), bits 16-18 format, bits 19-26 nnz - 1,
//                  bit 31 = 0;
//   inline block:  a pattern-only COO block with at most 3 entries keeps its
//                  coordinates in the word itself and has no payload:
//                  bits 0-23 coordinates (byte k = row << 4 | col of entry k;
//                  unused bytes repeat entry 0), bits 24-25 nnz - 1, bit 31 = 1.
//
// Payload layouts (bytes from the 16-byte aligned start; bit k of a row mask
// is local column k, bit k of a column mask is local row k, as in Figure 5's
// "row_mask 10 = 0b1010 -> columns 1 and 3"):
//   COO         coord u8[nnz] (row << 4 | col, row-major order), values at align4(nnz)
//   Dense       with values: values f32[256] column-major (v[c*16+r]) at 0 and
//               col_mask u16[16] at 1024, the block starting on a 64-byte
//               boundary (padding units before it are zero), so each column's
//               16 values are one aligned 64-byte run; absent entries hold 0
//               and are excluded through col_mask.  Pattern only: col_mask at 0
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

// Pull tiles (one warp task each): at most this many blocks (32 lanes x 8)
// and this many row blocks (the warp's shared-memory row accumulators).
constexpr uint32_t TILE_MAX_BLOCKS = 256;
constexpr uint32_t TILE_MAX_SPAN = 32;
// tiles[] = {p0, payload offset of block p0, first row block rb0, w}.
// w: span in bits 0-15, bit 16: the first row block continues in the
// previous tile, bit 17: the last row block continues in the next tile,
// bits 20-28: block count.  A tile's descriptors, copied in 16-byte units
// from the even index at or below p0, fit 256 slots: (p0 & 1) + count <= 256.
constexpr uint32_t TILE_SPAN_MASK = 0xFFFFu;
constexpr uint32_t TILE_FIRST_SHARED = 1u << 16;
constexpr uint32_t TILE_LAST_SHARED = 1u << 17;
constexpr uint32_t TILE_NBLK_SHIFT = 20;
// Push tasks: CSC positions per work item (one warp, up to eight positions
// per lane); the size is chosen per call from the push work.
constexpr uint32_t PUSH_CHUNK = 256;
constexpr uint32_t PUSH_CHUNK_MIN = 32;

constexpr uint32_t DESC_COL_MASK = 0x07FFFFFFu;   // column block bits of blk_desc.x
constexpr uint32_t DESC_LRB_SHIFT = 27;            // local row block bits of blk_desc.x

constexpr uint32_t META_INLINE = 0x80000000u;
constexpr uint32_t INLINE_MAX_NNZ = 3;

DBS_HD uint32_t meta_pack(uint32_t cmask, uint32_t fmt, uint32_t nnz)
{
    return (cmask & 0xFFFFu) | (fmt << 16) | ((nnz - 1u) << 19);
}
// coords: nnz (1..3) bytes row << 4 | col
DBS_HD uint32_t meta_pack_inline(const uint8_t *coords, uint32_t nnz)
{
    uint32_t w = 0;
    for (uint32_t k = 0; k < 3u; ++k) w |= (uint32_t)coords[k < nnz ? k : 0u] << (8u * k);
    return META_INLINE | ((nnz - 1u) << 24) | w;
}
DBS_HD bool meta_inline(uint32_t m) { return (m & META_INLINE) != 0u; }
DBS_HD uint32_t meta_fmt(uint32_t m) { return meta_inline(m) ? FMT_COO : (m >> 16) & 7u; }
DBS_HD uint32_t meta_nnz(uint32_t m) { return meta_inline(m) ? ((m >> 24) & 3u) + 1u : ((m >> 19) & 0xFFu) + 1u; }
// Section 3.3.2: Dense 4, ForceCSR / ForceCSC / (patched) CSR 2, COO 1.
DBS_HD uint32_t fmt_weight(uint32_t fmt)
{
    return fmt == FMT_DENSE ? 4u : (fmt == FMT_COO ? 1u : 2u);
}

DBS_HD uint32_t struct_bytes(uint32_t fmt, uint32_t nnz)
{
    return fmt == FMT_COO ? nnz : fmt == FMT_DENSE ? 32u : fmt == FMT_PCSR ? 64u + nnz : 48u;
}
// Byte offset of a Dense block's column masks.
DBS_HD uint32_t dense_mask_off(bool valued) { return valued ? 1024u : 0u; }
// Payload units a valued Dense block is aligned to (64 bytes).
constexpr uint32_t DENSE_ALIGN_UNITS = 4;
DBS_HD uint32_t val_offset(uint32_t fmt, uint32_t nnz)
{
    return fmt == FMT_DENSE ? 0u : (struct_bytes(fmt, nnz) + 3u) & ~3u;
}
DBS_HD uint32_t val_count(uint32_t fmt, uint32_t nnz) { return fmt == FMT_DENSE ? 256u : nnz; }
DBS_HD uint32_t payload_bytes(uint32_t fmt, uint32_t nnz, bool valued)
{
    if (fmt == FMT_DENSE) return valued ? 1024u + 32u : 32u;
    return val_offset(fmt, nnz) + (valued ? 4u * val_count(fmt, nnz) : 0u);
}
DBS_HD uint32_t payload_units(uint32_t fmt, uint32_t nnz, bool valued)
{
    return (payload_bytes(fmt, nnz, valued) + 15u) >> 4;
}
// Payload units of a block given its meta word (0 for inline blocks).
DBS_HD uint32_t meta_units(uint32_t m, bool valued)
{
    return meta_inline(m) ? 0u : payload_units(meta_fmt(m), meta_nnz(m), valued);
}

// Offsets of the structural arrays.
constexpr uint32_t OFF_PTR = 0;        // row_ptr (ForceCSR, patched) or col_ptr (ForceCSC)
constexpr uint32_t OFF_MASK = 16;      // row_mask / col_mask (Force*, patched)
constexpr uint32_t OFF_PCOLPTR = 48;   // patched CSR col_ptr
constexpr uint32_t OFF_RCSC = 64;      // patched CSR row_idx_csc2csr bytes

}  // namespace dbs
