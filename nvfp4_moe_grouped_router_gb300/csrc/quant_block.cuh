// NVFP4 quantization of 16-element blocks, shared by the row quantizer, the
// fused route+quantize kernel and the GEMM1 epilogue (which requantizes
// h = silu(gate) * up): FP32 amax, E4M3 block scale of amax / (6 gs),
// reciprocal of dec(scale) * gs, E2M1 codes of x * r.  Every step is a single
// correctly rounded FP32 operation (the products two per f32x2 multiply) or a
// round-to-nearest-even satfinite conversion instruction.  Also the stores of
// 64-element groups into each operand layout.
#pragma once
#include "layout.cuh"
#include "ptx.cuh"

namespace nvf {

// Returns the E4M3 scale byte; writes the 8 code bytes (element 2j in the low
// nibble of byte j) to w0 (bytes 0-3) and w1 (bytes 4-7).
__device__ __forceinline__ uint32_t quant_block16(const float* v, float gs, float six_gs, uint32_t& w0,
                                                  uint32_t& w1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sb = cvt_e4m3(__fdiv_rn(amax, six_gs));
  const float t3 = __fmul_rn(e4m3_to_f32(sb), gs);
  const float r = (t3 == 0.0f) ? 0.0f : __frcp_rn(t3);
  w0 = e2m1x8_scaled(v, r);
  w1 = e2m1x8_scaled(v + 8, r);
  return sb;
}

// 64 values -> 32 code bytes (w[0..7]) and 4 scale bytes (returned, block b in byte b).
__device__ __forceinline__ uint32_t quant_group64(const float (&v)[64], float gs, uint32_t (&w)[8]) {
  const float six_gs = __fmul_rn(6.0f, gs);
  uint32_t sf = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) sf |= quant_block16(v + 16 * b, gs, six_gs, w[2 * b], w[2 * b + 1]) << (8 * b);
  return sf;
}

// Store one quantized 64-element group (K elements 64*gg .. 64*gg+63) of row p.
//   ROWMAJOR:      codes/scales row-major.
//   TILED_GROUPED: `tile` and `r` locate the row's 128-row tile; codes holds the chunks.
//   TILED:         rows in groups of group_rows (weights); codes holds the units.
__device__ __forceinline__ void store_group64(uint8_t* codes, uint8_t* scales, int layout, int K, int64_t p,
                                              int64_t tile, uint32_t r, int gg, const uint32_t (&w)[8],
                                              uint32_t sf, int64_t group_rows = 0) {
  if (layout == LAYOUT_ROWMAJOR) {
    uint4* dst = reinterpret_cast<uint4*>(codes + p * (K / 2) + gg * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    *reinterpret_cast<uint32_t*>(scales + p * (K / 16) + gg * 4) = sf;
    return;
  }
  uint8_t* cbase;
  uint8_t* abase;
  if (layout == LAYOUT_TILED) {
    const TiledPos t = weight_tiled_pos(p, gg >> 2, group_rows, num_k_tiles(K));
    cbase = codes + t.codes;
    abase = codes + t.atoms;
    r = t.r;
  } else {
    cbase = codes + (static_cast<size_t>(tile) * num_k_tiles(K) + (gg >> 2)) * TILE_BYTES;
    abase = cbase + TILE_CODE_BYTES;
  }
  const uint32_t b = static_cast<uint32_t>(gg & 3) * 32u;
  *reinterpret_cast<uint4*>(cbase + tiled_code_offset(r, b)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(cbase + tiled_code_offset(r, b + 16)) = make_uint4(w[4], w[5], w[6], w[7]);
  *reinterpret_cast<uint32_t*>(abase + (gg & 3) * 512 + sf_atom_offset(r, 0)) = sf;
}

// TILED_GROUPED store of one 64-element group with one 32-byte store for the
// codes: the group's two 16-byte pieces are the two halves of a 32-byte-aligned
// block of the swizzled row (swapped when r is odd).  The chunk base must be
// 32-byte aligned (a 256-byte aligned buffer).
__device__ __forceinline__ void store_group64_tg32(uint8_t* codes, int K, int64_t tile, uint32_t r, int gg,
                                                   const uint32_t (&w)[8], uint32_t sf) {
  uint8_t* cbase = codes + (static_cast<size_t>(tile) * num_k_tiles(K) + (gg >> 2)) * TILE_BYTES;
  const uint32_t b = static_cast<uint32_t>(gg & 3) * 32u;
  uint8_t* dst = cbase + r * 128u + ((((b >> 4) ^ (r & 7u)) & ~1u) << 4);
  if (r & 1u) st_global_v8(dst, w[4], w[5], w[6], w[7], w[0], w[1], w[2], w[3]);
  else st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
  *reinterpret_cast<uint32_t*>(cbase + TILE_CODE_BYTES + (gg & 3) * 512 + sf_atom_offset(r, 0)) = sf;
}

}  // namespace nvf
