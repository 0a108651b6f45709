// One 16-element NVFP4 block, shared by the row quantizer and the GEMM1
// epilogue (which requantizes h = silu(gate) * up): FP32 amax, E4M3 block
// scale of amax / (6 gs), reciprocal of dec(scale) * gs, E2M1 codes of x * r.
// Every step is a single correctly rounded FP32 operation or a documented
// round-to-nearest-even satfinite conversion instruction.
#pragma once
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
  uint32_t b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = cvt_e2m1x2(__fmul_rn(v[2 * j], r), __fmul_rn(v[2 * j + 1], r));
  w0 = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  w1 = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sb;
}

}  // namespace nvf
