// Operand layouts shared by the quantizer, the GEMM epilogue (which writes the
// next GEMM's operand) and the GEMM producer.  All three must agree byte for
// byte.
//
// ROWMAJOR: codes [rows][K/2] (element 2j in the low nibble of byte j),
//           scales [rows][K/16].
//
// TILED / TILED_GROUPED (what the GEMM consumes).  The GEMM streams both
// operands with plain 1-D bulk copies, so operands are stored the way one
// pipeline stage wants them in shared memory.  A matrix [rows, K] is cut into
// 128-row tiles and 256-element K tiles; the (tile, kt) piece consists of
//   codes (16384 bytes): rows 0..127, 128 bytes per row, with the 128-byte
//                   swizzle already applied: code byte b of row r sits at
//                   r * 128 + (((b / 16) ^ (r % 8)) * 16) + b % 16
//   atoms (2048 bytes): four 512-byte scale atoms; atom kk covers K elements
//                   64*kk .. 64*kk+63 of the K tile, and row r's 4 scales
//                   (16 elements each) sit at (r % 32) * 16 + (r / 32) * 4 + b.
//                   Four warps write an atom's 32 rows into TMEM with
//                   tcgen05.st, one 32-lane quarter each (the layout the
//                   block-scaled MMA reads its scale factors in).
// The first 8*j rows of the codes are their first 1024*j bytes, so a partial
// tile can be loaded by a prefix copy.  Bytes of rows past a group's end, and
// of K past K in the last K tile, are never written and never used.
//   TILED_GROUPED (activations): rows grouped by offsets[G+1]; group g's rows
//                   form 128-row tiles numbered from tile_offsets[g] (the
//                   exclusive prefix of ceil(m_g / 128)): tile =
//                   tile_offsets[g] + (row - offsets[g]) / 128.  Piece
//                   (tile, kt) is the 18432-byte chunk [codes][atoms] at
//                   (tile * nkt + kt) * TILE_BYTES, nkt = ceil(K / 256).
//   TILED (weights): rows form equal groups of R rows (one expert's N rows;
//                   the whole matrix when there is one group).  Within a
//                   group, tiles 2p and 2p + 1 form pair p, and K tile kt of
//                   a pair is one 36864-byte unit [codes 2p][codes 2p + 1]
//                   [atoms 2p][atoms 2p + 1]: a 256-column GEMM tile loads it
//                   with one copy into a stage laid out the same way.  When a
//                   group has an odd number of tiles, its last tile's units
//                   are 18432-byte chunks [codes][atoms].  Pair p starts at
//                   group_base + p * 2 * nkt * TILE_BYTES, group_base =
//                   group * ceil(R / 128) * nkt * TILE_BYTES.
#pragma once
#include <cstdint>

namespace nvf {

enum OperandLayout : int { LAYOUT_ROWMAJOR = 0, LAYOUT_TILED = 1, LAYOUT_TILED_GROUPED = 2 };

constexpr int TILE_ROWS = 128;
constexpr int KT_ELEMS = 256;
constexpr int TILE_CODE_BYTES = TILE_ROWS * KT_ELEMS / 2;   // 16384
constexpr int TILE_SF_BYTES = 4 * 512;                      // 2048
constexpr int TILE_BYTES = TILE_CODE_BYTES + TILE_SF_BYTES;  // 18432

__host__ __device__ __forceinline__ uint32_t sf_atom_offset(uint32_t r128, uint32_t b4) {
  return (r128 & 31u) * 16u + (r128 >> 5) * 4u + b4;
}
__host__ __device__ __forceinline__ uint32_t tiled_code_offset(uint32_t r, uint32_t b) {
  return r * 128u + ((((b >> 4) ^ (r & 7u)) << 4) | (b & 15u));
}
__host__ __device__ __forceinline__ int num_k_tiles(int K) { return (K + KT_ELEMS - 1) / KT_ELEMS; }

// TILED (weights): where the codes and the atoms of (row, K tile kt) start, for
// groups of group_rows rows; r is the row within its 128-row tile.
struct TiledPos {
  uint64_t codes, atoms;
  uint32_t r;
};
__host__ __device__ __forceinline__ TiledPos weight_tiled_pos(int64_t row, int kt, int64_t group_rows, int nkt) {
  const int64_t g = row / group_rows, rl = row - g * group_rows;
  const int64_t ntg = (group_rows + TILE_ROWS - 1) / TILE_ROWS;
  const int64_t tile = rl / TILE_ROWS, pair = tile >> 1;
  const uint64_t half = static_cast<uint64_t>(tile & 1);
  const bool paired = 2 * pair + 1 < ntg;
  const uint64_t unit = (static_cast<uint64_t>(g * ntg + 2 * pair) * nkt + static_cast<uint64_t>(kt) * (paired ? 2 : 1)) *
                        TILE_BYTES;
  TiledPos t;
  t.codes = unit + (paired ? half * TILE_CODE_BYTES : 0);
  t.atoms = unit + (paired ? 2 * TILE_CODE_BYTES + half * TILE_SF_BYTES : TILE_CODE_BYTES);
  t.r = static_cast<uint32_t>(rl % TILE_ROWS);
  return t;
}

// Prepared w13 row order: the fused SiLU-and-mul epilogue needs gate row i and
// up row I + i in the same 32-row block.  Prepared row p of a stack of experts
// (2I rows each) is canonical row w13_source_row(p, I) of the same stack:
// within an expert, prepared rows [32c, 32c + 16) are gate rows [16c, 16c + 16)
// and rows [32c + 16, 32c + 32) the up rows [I + 16c, I + 16c + 16).
__host__ __device__ __forceinline__ int64_t w13_source_row(int64_t p, int32_t I) {
  const int64_t e = p / (2 * I);
  const int32_t r = static_cast<int32_t>(p - e * 2 * I);
  const int32_t c = r >> 5, within = r & 31;
  return e * 2 * I + (within < 16 ? 16 * c + within : I + 16 * c + within - 16);
}

// Largest g in [0, G) with offs[g] <= v (offs non-decreasing, offs[0] <= v < offs[G]).
__device__ __forceinline__ int upper_group(const int32_t* offs, int G, int64_t v) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(offs[mid]) <= v) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace nvf
