// Weight-only NVFP4 grouped GEMM (W4A16) for sm_103a:
//     D[row, n] = gs_b[g] * sum_k a[row, k] * dB_g[n, k]   for offsets[g] <= row < offsets[g+1]
// with FP16 activations a and NVFP4 weights dB = e2m1 * e4m3 dequantized in the
// kernel and multiplied on the tensor cores as FP16 (tcgen05.mma kind::f16).
// This is the decode alternative the pages keep comparing with the W4A4 path:
// W4A16 unpacks FP4 weights and runs FP16 MMA (unsloth report, SASS paragraph
// under "Why it matters"; Marlin W4A16 in FlashInfer issue #2723, "Speed
// Comparison").  Every e2m1 * e4m3 product is exact in FP16 (at most 6
// significant bits, 2^-10 .. 2688), so the dequantized weights lose nothing.
//
// One CTA per (128-row tile of one group, 256 output columns), 256 threads.
// K advances in steps of 64 elements:
//   - A (FP16 rows, 128 bytes of a row a step) by cp.async, two steps ahead,
//     into 128-byte-swizzled K-major rows;
//   - B: thread i owns weight row i of the block: it loads the row's 32 code
//     bytes and 4 scale bytes of the next step into registers while it
//     converts the current step's (cvt.rn.f16x2.e2m1x2, then one f16x2 multiply
//     by the block scale) straight into the swizzled K-major FP16 tile;
//   - one thread issues four 128 x 256 x 16 MMAs into a 256-column TMEM
//     accumulator and commits the stage.
// A 4-stage ring (4 x 48 KB); the epilogue moves each warp's slice of the
// accumulator to registers, scales by gs_b[g] and stores FP32 or BF16 rows.
// Every wait is bounded; the CTA agrees on a failed wait before leaving.
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvf {
namespace {

constexpr int WM = 128, WN = 256, WKS = 64;   // tile rows, tile columns, K per step
constexpr int W_STAGES = 4;
constexpr int W_THREADS = 256;
constexpr int WA_STAGE = WM * 128;             // 16 KB: 128 rows x 64 fp16
constexpr int WB_STAGE = WN * 128;             // 32 KB: 256 rows x 64 fp16
constexpr int W_SMEM = W_STAGES * (WA_STAGE + WB_STAGE) + 1024 + 128;

// Two E2M1 codes (low nibble = lower element) -> f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  const uint16_t in = static_cast<uint16_t>(byte & 0xFFu);
  asm("{\n .reg .b8 t;\n cvt.u8.u16 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "h"(in));
  return r;
}
// One E4M3 byte -> the same FP16 value in both halves.
__device__ __forceinline__ uint32_t e4m3_to_f16x2_dup(uint32_t b) {
  uint32_t r;
  const uint16_t in = static_cast<uint16_t>((b & 0xFFu) | ((b & 0xFFu) << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__global__ void __launch_bounds__(W_THREADS, 1) w4a16_kernel(const __half* __restrict__ A, int64_t lda,
                                                           const uint8_t* __restrict__ B, const float* __restrict__ gs_b,
                                                           const int32_t* __restrict__ offsets,
                                                           const int32_t* __restrict__ tile_offs, int G, int N, int K,
                                                           int out_bf16, void* D, int64_t ldd, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t a0 = s_base, b0 = s_base + W_STAGES * WA_STAGE;
  const uint32_t bar0 = b0 + W_STAGES * WB_STAGE;                 // mma_done[W_STAGES], then drain
  const uint32_t drain_bar = bar0 + 8 * W_STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + W_STAGES * (WA_STAGE + WB_STAGE) + 8 * (W_STAGES + 1));
  __shared__ int abort_flag;
  __shared__ int s_tile[3];  // group, first row, rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, nb = blockIdx.y;
  if (mt >= __ldg(tile_offs + G)) return;                    // past the groups' tiles (uniform)
  if (tid == 0) {
    int lo = 0, hi = G;                                      // last g with tile_offs[g] <= mt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(tile_offs + mid) <= mt) lo = mid; else hi = mid;
    }
    const int row0 = __ldg(offsets + lo) + (mt - __ldg(tile_offs + lo)) * WM;
    s_tile[0] = lo;
    s_tile[1] = row0;
    s_tile[2] = min(WM, __ldg(offsets + lo + 1) - row0);
    for (int s = 0; s <= W_STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_holder), WN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int g = s_tile[0], row0 = s_tile[1], rows = s_tile[2];
  const int ncols = min(WN, N - nb * WN);                    // 256, or 128 for the last block
  const int nks = K / WKS, nkt = num_k_tiles(K);

  // A step s -> stage s % W_STAGES: 1024 pieces of 16 bytes, 4 a thread; rows past
  // the group's end are zeroed the first time each stage is used and stay zero.
  auto load_a = [&](int s) {
    const uint32_t st = a0 + (s % W_STAGES) * WA_STAGE;
#pragma unroll
    for (int i = 0; i < (WM * 8) / W_THREADS; ++i) {
      const int p = tid + W_THREADS * i, r = p >> 3, c = p & 7;
      const uint32_t dst = st + r * 128 + ((c ^ (r & 7)) << 4);
      if (r < rows) cp_async16(dst, A + static_cast<int64_t>(row0 + r) * lda + s * WKS + c * 8);
      else if (s < W_STAGES) st_shared_zero16(dst);
    }
  };
  // B registers of step s for this thread's weight row (tid < ncols).
  const bool b_row = tid < ncols;
  TiledPos bpos{};
  uint4 bc0 = make_uint4(0, 0, 0, 0), bc1 = make_uint4(0, 0, 0, 0);
  uint32_t bsf = 0;
  auto load_b = [&](int s) {
    if (!b_row) return;
    bpos = weight_tiled_pos(static_cast<int64_t>(g) * N + nb * WN + tid, s >> 2, N, nkt);
    const uint32_t kb = static_cast<uint32_t>(s & 3) * 32;     // code bytes of this step in the K tile
    bc0 = __ldg(reinterpret_cast<const uint4*>(B + bpos.codes + tiled_code_offset(bpos.r, kb)));
    bc1 = __ldg(reinterpret_cast<const uint4*>(B + bpos.codes + tiled_code_offset(bpos.r, kb + 16)));
    bsf = __ldg(reinterpret_cast<const uint32_t*>(B + bpos.atoms + (s & 3) * 512 + sf_atom_offset(bpos.r, 0)));
  };
  // Registers -> FP16 row tid of stage s % W_STAGES (128 bytes, 8 swizzled 16-byte pieces).
  auto store_b = [&](int s) {
    if (!b_row) return;
    const uint32_t row = b0 + (s % W_STAGES) * WB_STAGE + tid * 128;
    const uint32_t cw[8] = {bc0.x, bc0.y, bc0.z, bc0.w, bc1.x, bc1.y, bc1.z, bc1.w};
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {                        // 16 elements: 8 code bytes, one scale
      const uint32_t sc = e4m3_to_f16x2_dup(bsf >> (8 * blk));
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) h[q] = hmul2_u32(e2m1x2_to_f16x2(cw[2 * blk + (q >> 2)] >> (8 * (q & 3))), sc);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c = 2 * blk + half;                          // 16-byte piece (8 fp16) of the 128-byte row
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(row + ((c ^ (tid & 7)) << 4)), "r"(h[4 * half]),
                     "r"(h[4 * half + 1]), "r"(h[4 * half + 2]), "r"(h[4 * half + 3])
                     : "memory");
      }
    }
  };

  const uint32_t idesc = f16kind_idesc(WM, ncols, false);
  bool ok = true;
  load_a(0);
  cp_async_commit();
  if (nks > 1) load_a(1);
  cp_async_commit();
  load_b(0);
  for (int s = 0; s < nks && ok; ++s) {
    const int st = s % W_STAGES;
    if (s >= 2) {
      // stage (s + 2) % 4 was last read by the MMAs of step s - 2
      const int ps = s - 2;
      ok = mbar_wait(bar0 + 8 * (ps % W_STAGES), (ps / W_STAGES) & 1, &abort_flag, err, DEV_TIMEOUT_MMA, mt);
      ok = __syncthreads_and(ok);
      if (!ok) break;
    }
    if (s + 2 < nks) load_a(s + 2);
    cp_async_commit();
    store_b(s);
    if (s + 1 < nks) load_b(s + 1);
    cp_async_wait<2>();                                        // A of step s has landed
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < WKS / 16; ++kk)
        tc_mma_f16kind(tmem, operand_desc_sw128(a0 + st * WA_STAGE + kk * 32),
                       operand_desc_sw128(b0 + st * WB_STAGE + kk * 32), idesc, (s | kk) != 0 ? 1u : 0u);
      tc_commit(bar0 + 8 * st);
    }
  }
  cp_async_wait<0>();
  if (ok && nks > 0)
    ok = mbar_wait(bar0 + 8 * ((nks - 1) % W_STAGES), ((nks - 1) / W_STAGES) & 1, &abort_flag, err,
                   DEV_TIMEOUT_EPILOGUE, mt);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
    // warp w: TMEM lane quarter w % 4 (rows), columns 128 * (w / 4) .. + 127
    const int q = warp & 3, half = warp >> 2;
    const int r = q * 32 + lane;
    if (half * 128 < ncols) {
      const float alpha = __ldg(gs_b + g);
      const uint32_t tb = tmem + half * 128 + (static_cast<uint32_t>(q * 32) << 16);
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tb + c * 32, v[c]);
      tmem_ld_wait();
      if (r < rows) {
        const int64_t row = static_cast<int64_t>(row0) + r;
        const int64_t col0 = static_cast<int64_t>(nb) * WN + half * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(D) + row * ldd + col0 + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int h2 = 0; h2 < 4; ++h2) {
                __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[c][8 * j + 2 * h2]), alpha),
                                                         __fmul_rn(__uint_as_float(v[c][8 * j + 2 * h2 + 1]), alpha));
                w[h2] = *reinterpret_cast<uint32_t*>(&b);
              }
              dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(D) + row * ldd + col0 + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__fmul_rn(__uint_as_float(v[c][4 * j]), alpha),
                                   __fmul_rn(__uint_as_float(v[c][4 * j + 1]), alpha),
                                   __fmul_rn(__uint_as_float(v[c][4 * j + 2]), alpha),
                                   __fmul_rn(__uint_as_float(v[c][4 * j + 3]), alpha));
          }
        }
      }
    }
  } else if (tid == 0) {
    // Every MMA this CTA issued must finish before TMEM is freed (bounded wait).
    tc_commit(drain_bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitTimeoutNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, WN);
}

}  // namespace

cudaError_t launch_w4a16(const void* A, int64_t a_rows, int64_t lda, const uint8_t* B, const float* gs_b,
                         const int32_t* offsets, const int32_t* tile_offs, int32_t G, int32_t N, int32_t K,
                         int out_bf16, void* D, int64_t ldd, int* err, cudaStream_t s) {
  if (a_rows <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, W_SMEM);
  if (e != cudaSuccess) return e;
  const int64_t max_tiles = (a_rows + WM - 1) / WM + G;
  dim3 grid(static_cast<unsigned>(max_tiles), static_cast<unsigned>((N + WN - 1) / WN));
  w4a16_kernel<<<grid, W_THREADS, W_SMEM, s>>>(static_cast<const __half*>(A), lda, B, gs_b, offsets, tile_offs, G, N,
                                               K, out_bf16, D, ldd, err);
  return cudaGetLastError();
}

}  // namespace nvf
