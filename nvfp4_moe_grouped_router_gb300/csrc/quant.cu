// NVFP4 quantization kernels: per-tensor global scale (FP32 amax / 2688) and
// the row quantizer, optionally gathering rows (the permute of tokens by
// expert) and writing the operand layouts the GEMM consumes.
//
// Method: FP4 E2M1 values with one unsigned E4M3 scale per 16 elements
// (unsloth "Report: NVFP4 kernel selection on SM120/SM121", SASS paragraph
// under "Why it matters": E2M1.E2M1.UE4M3.4X) and an FP32 block amax
// (FlashInfer issue #2723, "What We Tried", item 2 "FP32 Amax Computation").
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int kMaxSmemGroups = 4096;

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

// One thread per (output row, 64-element group).  Group offsets (when given)
// are staged in shared memory for the row -> group search.
__global__ void __launch_bounds__(256) quantize_kernel(QuantArgs a) {
  extern __shared__ int32_t s_offs[];  // [G+1] offsets, [G+1] tile offsets
  const bool grouped = a.offsets != nullptr;
  const bool smem_offs = grouped && a.G < kMaxSmemGroups;
  const int32_t* offs = a.offsets;
  const int32_t* toffs = a.tile_offs;
  if (smem_offs) {
    for (int i = threadIdx.x; i <= a.G; i += blockDim.x) {
      s_offs[i] = a.offsets[i];
      s_offs[a.G + 1 + i] = a.tile_offs ? a.tile_offs[i] : 0;
    }
    __syncthreads();
    offs = s_offs;
    toffs = s_offs + a.G + 1;
  }
  const int gpr = a.K >> 6;  // 64-element groups per row
  const int64_t total = a.rows * gpr;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = idx / gpr;
    const int gg = static_cast<int>(idx - p * gpr);
    const int64_t src = a.gather ? static_cast<int64_t>(__ldg(a.gather + p))
                                 : (a.w13_I > 0 ? w13_source_row(p, a.w13_I) : p);
    const int g = grouped ? upper_group(offs, a.G, p)
                          : (a.rows_per_group > 0 ? static_cast<int>(p / a.rows_per_group) : 0);
    const float gs = __ldg(a.gs + g);
    float v[64];
    load64(a.x, a.x_dtype, src * a.ldx + gg * 64, v);
    uint32_t w[8];
    const uint32_t sf = quant_group64(v, gs, w);
    int64_t tile = 0;
    uint32_t r = 0;
    if (a.layout == LAYOUT_TILED_GROUPED) {
      const int64_t local = p - offs[g];
      tile = toffs[g] + (local >> 7);
      r = static_cast<uint32_t>(local & 127);
    }
    store_group64(a.codes, a.scales, a.layout, a.K, p, tile, r, gg, w, sf,
                  a.rows_per_group > 0 ? a.rows_per_group : a.rows);
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
  const size_t smem = (a.offsets && a.G < kMaxSmemGroups) ? 2 * (a.G + 1) * sizeof(int32_t) : 0;
  prefer_max_shared(reinterpret_cast<const void*>(quantize_kernel));
  quantize_kernel<<<static_cast<unsigned>(blocks), 256, smem, s>>>(a);
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
