// Scale-factor layouts shared by the quantizer, the GEMM epilogue and the GEMM
// producer.  All three must agree byte for byte.
//
// The block-scaled FP4 MMA reads its scale factors from TMEM in 128-row x
// 4-scale "atoms" (one atom per 128 rows per 64-element MMA K step).  An atom
// is 512 contiguous bytes: row r, K-block b (0..3) lives at
//     (r % 32) * 16 + (r / 32) * 4 + b
// so that one tcgen05.cp 32x128b.warpx4 moves the whole atom to TMEM.
//
//   ROWMAJOR : scales[row][K/16]
//   MMA      : atom (row / 128, k64) at ((row / 128) * (K / 64) + k64) * 512
//   GROUPED  : rows grouped by offsets[G+1]; group g's rows are cut into
//              128-row tiles numbered from tile_offsets[g] (the exclusive
//              prefix of ceil(m_g / 128)); atom (tile, k64) at
//              (tile * (K / 64) + k64) * 512.  Rows past a group's end in its
//              last tile are never written.
#pragma once
#include <cstdint>

namespace nvf {

enum SfLayout : int { SF_ROWMAJOR = 0, SF_MMA = 1, SF_GROUPED = 2 };

__host__ __device__ __forceinline__ uint32_t sf_atom_offset(uint32_t r128, uint32_t b4) {
  return (r128 & 31u) * 16u + (r128 >> 5) * 4u + b4;
}

// Largest g in [0, G) with offs[g] <= v (offs non-decreasing, offs[0] <= v < offs[G]).
__device__ __forceinline__ int upper_group(const int32_t* __restrict__ offs, int G, int64_t v) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(__ldg(offs + mid)) <= v) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace nvf
