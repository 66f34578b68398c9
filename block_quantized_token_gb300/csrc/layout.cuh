// The in-HBM layout of a repacked block-quantized matrix.
//
// A GGUF Q8_0 / Q4_0 matrix [rows x cols] stores each row as cols/32 blocks of
// [fp16 scale d][32 quantised values] (34 / 18 bytes, "EdgeRunner Core
// Architecture" sections 3.1-3.2).  Those sizes are not multiples of 16, so a
// warp cannot read them with aligned 128-bit loads.  The library rearranges
// the same bytes once, at create time, into "units" that match the register
// fragments of the m16n8k16 tensor-core MMA used to form the dot products:
//
//   row group  = 16 consecutive (virtual) rows
//   unit       = one row group x 64 columns (2 blocks per row, 32 blocks)
//   unit bytes = [quant bytes][64 bytes of scales]
//                Q8_0: 1024 + 64 = 1088;   Q4_0: 512 + 64 = 576
//   matrix     = [row group][unit] contiguous; a row with an odd number of
//                blocks gets one zero block (d = 0) to fill its last unit.
//
// Lane l = 4g + t of a warp owns, per block and 16-column half h, the MMA A
// fragment a0..a3 = (row g, col 2t..2t+1), (row g+8, col 2t..2t+1),
// (row g, col 2t+8..2t+9), (row g+8, col 2t+8..2t+9).
//   Q8_0: the unit is 2 x 512 bytes (block 0, block 1); lane l's 16 bytes of
//         block b are at b*512 + 16l; byte j = 8h + 2r + e holds fragment
//         register r, element e of half h, stored as q ^ 0x80.
//   Q4_0: lane l's 16 bytes are at 16l; 32-bit word w = 2b + h of them holds
//         the 8 nibbles of block b, half h; nibble p (bits 4p..4p+3) is
//         register p % 4, element p / 4, stored as the GGUF nibble (q + 8).
//   scales: 8 bytes per g at quant_bytes + 8g: fp16 d(row g, block 0),
//         d(row g+8, block 0), d(row g, block 1), d(row g+8, block 1).
//
// Virtual rows: a row group's 16 fragment rows r = 0..15 come from source
// rows by a row map chosen for the epilogue that consumes them:
//   IDENT : r -> 16*rg + r
//   PAIR  : r < 8 -> 16*rg + 2r, r >= 8 -> 16*rg + 2(r-8) + 1
//           (the two rows a RoPE pair rotates land in one lane)
//   GATEUP: r < 8 -> gate row 8*rg + r, r >= 8 -> up row 8*rg + r - 8
//           (a SwiGLU output's two inputs land in one lane)
#pragma once

#include <stdint.h>

namespace er {

enum QType : int { Q8_0 = 8, Q4_0 = 2 };
enum RowMap : int { MAP_IDENT = 0, MAP_PAIR = 1, MAP_GATEUP = 2 };

template <int QT>
struct QTraits;
template <>
struct QTraits<Q8_0> {
    static constexpr int gguf_block_bytes = 34;
    static constexpr int quant_bytes = 1024;  // per unit
    static constexpr int unit_bytes = 1088;
};
template <>
struct QTraits<Q4_0> {
    static constexpr int gguf_block_bytes = 18;
    static constexpr int quant_bytes = 512;
    static constexpr int unit_bytes = 576;
};

__host__ __device__ inline int unit_bytes_of(int qt) { return qt == Q8_0 ? 1088 : 576; }
__host__ __device__ inline int quant_bytes_of(int qt) { return qt == Q8_0 ? 1024 : 512; }
__host__ __device__ inline int gguf_block_bytes_of(int qt) { return qt == Q8_0 ? 34 : 18; }

// Fragment coordinates of element (row r of the group, column c of the unit):
// c in [0, 64): block b = c / 32, half h = (c % 32) / 16, kl = c % 16.
struct FragPos {
    int lane;      // 4g + t
    int b, h;      // block in unit, half in block
    int reg, e;    // fragment register 0..3, element 0..1
    int g, upper;  // row = g + 8*upper
};

__host__ __device__ inline FragPos frag_pos(int r, int c) {
    FragPos p;
    p.g = r & 7;
    p.upper = r >> 3;
    p.b = c >> 5;
    p.h = (c >> 4) & 1;
    int kl = c & 15;
    int t = (kl & 7) >> 1;
    p.e = kl & 1;
    p.reg = ((kl >> 3) << 1) | p.upper;
    p.lane = 4 * p.g + t;
    return p;
}

// byte offset (within the unit) and, for Q4_0, nibble shift of element (r, c)
__host__ __device__ inline int q8_byte_offset(const FragPos &p) { return p.b * 512 + p.lane * 16 + p.h * 8 + p.reg * 2 + p.e; }
__host__ __device__ inline int q4_byte_offset(const FragPos &p, int &shift) {
    int word = 2 * p.b + p.h;
    int nib = p.reg + 4 * p.e;  // nibble index within the word
    shift = (nib & 1) * 4;
    return p.lane * 16 + word * 4 + (nib >> 1);
}
// byte offset (within the unit) of the fp16 scale of row r, block b
__host__ __device__ inline int scale_offset(int qt, int r, int b) {
    return quant_bytes_of(qt) + (r & 7) * 8 + (b * 2 + (r >> 3)) * 2;
}

}  // namespace er
