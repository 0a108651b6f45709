// NVFP4 quantization kernels: per-tensor global scale (FP32 amax / 2688) and
// the row quantizer, optionally gathering rows (the permute of tokens by
// expert) and writing scales in the layout the block-scaled MMA reads.
//
// Method: FP4 E2M1 values with one unsigned E4M3 scale per 16 elements
// (unsloth "Report: NVFP4 kernel selection on SM120/SM121", SASS paragraph
// under "Why it matters": E2M1.E2M1.UE4M3.4X) and an FP32 block amax
// (FlashInfer issue #2723, "What We Tried", item 2 "FP32 Amax Computation").
// Each 16-element block: amax -> sb = E4M3(amax / (6 gs)) -> r = 1/(dec(sb) gs)
// -> q = E2M1(x r), every step one correctly rounded FP32 operation.
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

__device__ __forceinline__ void load64(const void* x, int xdt, int64_t off, float (&v)[64]) {
  if (xdt == X_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint4 u = __ldg(p + i);
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[i * 8 + 2 * j] = __uint_as_float(w[j] << 16);
        v[i * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float4 f = __ldg(p + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  }
}

__global__ void __launch_bounds__(256) quantize_kernel(QuantArgs a) {
  const int gpr = a.K >> 6;  // 64-element groups per row: one per thread
  const int64_t total = a.rows * gpr;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = idx / gpr;
    const int gg = static_cast<int>(idx - p * gpr);
    const int64_t src = a.gather ? static_cast<int64_t>(__ldg(a.gather + p)) : p;
    const int g = a.offsets ? upper_group(a.offsets, a.G, p) : 0;
    const float gs = __ldg(a.gs + g);
    const float six_gs = __fmul_rn(6.0f, gs);
    float v[64];
    load64(a.x, a.x_dtype, src * a.ldx + gg * 64, v);
    uint32_t w[8];
    uint32_t sf = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) sf |= quant_block16(v + 16 * b, gs, six_gs, w[2 * b], w[2 * b + 1]) << (8 * b);
    uint4* dst = reinterpret_cast<uint4*>(a.codes + p * (a.K / 2) + gg * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    size_t off;
    if (a.layout == SF_ROWMAJOR) {
      off = static_cast<size_t>(p) * (a.K / 16) + gg * 4;
    } else if (a.layout == SF_MMA) {
      off = (static_cast<size_t>(p >> 7) * gpr + gg) * 512 + sf_atom_offset(static_cast<uint32_t>(p & 127), 0);
    } else {
      const int64_t local = p - __ldg(a.offsets + g);
      const int64_t tile = __ldg(a.tile_offs + g) + (local >> 7);
      off = (static_cast<size_t>(tile) * gpr + gg) * 512 + sf_atom_offset(static_cast<uint32_t>(local & 127), 0);
    }
    *reinterpret_cast<uint32_t*>(a.scales + off) = sf;
  }
}

__global__ void amax_kernel(const void* x, int xdt, int64_t n, uint32_t* out) {
  const int64_t g = blockIdx.y;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v = (xdt == X_BF16) ? __bfloat162float(static_cast<const __nv_bfloat16*>(x)[g * n + i])
                              : static_cast<const float*>(x)[g * n + i];
    m = fmaxf(m, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out + g, __float_as_uint(m));
}

__global__ void global_scale_finalize(uint32_t* bits, int64_t groups) {
  const int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (g >= groups) return;
  const float a = __uint_as_float(bits[g]);
  reinterpret_cast<float*>(bits)[g] = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
}

}  // namespace

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const int64_t total = a.rows * (a.K >> 6);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_global_scale(const void* x, int x_dtype, int64_t groups, int64_t n, float* gs_out,
                                cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(gs_out, 0, sizeof(float) * groups, s);
  if (e != cudaSuccess) return e;
  int64_t bx = (n + 255) / 256;
  if (bx > 64) bx = 64;
  if (bx < 1) bx = 1;
  dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(groups));
  amax_kernel<<<grid, 256, 0, s>>>(x, x_dtype, n, reinterpret_cast<uint32_t*>(gs_out));
  global_scale_finalize<<<static_cast<unsigned>((groups + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<uint32_t*>(gs_out), groups);
  return cudaGetLastError();
}

}  // namespace nvf
