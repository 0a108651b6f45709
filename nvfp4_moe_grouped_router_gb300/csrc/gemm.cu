// Grouped block-scaled FP4 GEMM for sm_103a (tcgen05, kind::mxf4nvf4).
//
// For every group (expert) g with rows [offsets[g], offsets[g+1]) of A:
//     D[row, n] = alpha_g * sum_k dA[row, k] * dB_g[n, k],  alpha_g = gs_a[g] * gs_b[g]
// where dA, dB are E2M1 codes times their UE4M3 block scales (one per 16 K
// elements).  This is the grouped block-scaled FP4 GEMM the MoE expert
// computation runs on (FlashInfer issue #2723, "The Problem"; vLLM PR #29242,
// "Purpose": nvfp4_blockwise_moe_kernel.cu) with a per-expert alpha and beta = 0
// (vLLM PR #29242 review: alpha_ptr_array, beta = 0.0f).
//
// Design (one CTA per SM, persistent, 320 threads):
//   warp 0    producer: per pipeline stage one contiguous 18 KB chunk of B
//             (128 weight rows x 256 K, codes pre-swizzled + scale atoms) and
//             the valid-row prefix of the matching A chunk, moved with 1-D
//             bulk copies (cp.async.bulk) into a STAGES-deep ring guarded by
//             mbarrier full/empty pairs.  Weights therefore stream from HBM as
//             sequential 18 KB runs.
//   warp 1    TMEM owner and MMA issuer: per stage, tcgen05.cp the scale atoms
//             into TMEM, then four 128x128x64 block-scaled MMAs into one of two
//             FP32 TMEM accumulators (128 columns each).
//   warps 2-9 epilogue: two warps per 32-lane TMEM quarter, 64 columns each;
//             tcgen05.ld, scale by alpha, then either store FP32/BF16 rows or
//             compute h = silu(gate) * up and requantize it to NVFP4 straight
//             into the next GEMM's tiled operand.  Warps whose 32 rows are all
//             past the group's end skip the arithmetic.
// Tiles are 128 rows of one group x 128 output columns; the scheduler walks
// (m-tile, n-tile) pairs with the m-tile index taken from the device-side
// tile prefix, so no host synchronisation is needed for group sizes.
// Every mbarrier wait is bounded; on timeout the kernel records an error word,
// drains what it issued, frees TMEM and returns.
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int BM = 128;             // rows of A per tile (MMA M)
constexpr int BN = 128;             // output columns per tile (MMA N)
#ifndef NVF_GEMM_STAGES
#define NVF_GEMM_STAGES 5
#endif
constexpr int STAGES = NVF_GEMM_STAGES;
constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // A chunk + B chunk
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 2 * BN;  // accumulators use columns [0, 256)

constexpr int OFF_BAR = STAGES * STAGE_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, acc_full[2], acc_empty[2], drain
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack

static_assert(SF_COL0 + STAGES * 32 <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(TILE_BYTES % 1024 == 0, "B chunk must stay 1024-byte aligned in shared memory");

struct Tile {
  int g, mt, nt, row0, rows;
};

__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& p, int ntiles) {
  Tile x;
  x.mt = t / ntiles;
  x.nt = t - x.mt * ntiles;
  x.g = upper_group(p.tile_offs, p.G, x.mt);
  const int local = x.mt - __ldg(p.tile_offs + x.g);
  x.row0 = __ldg(p.offsets + x.g) + local * BM;
  x.rows = min(BM, __ldg(p.offsets + x.g + 1) - x.row0);
  return x;
}

// Bounded wait that ignores the abort flag (used when draining).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int* err, int detail) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      report_error(err, DEV_TIMEOUT_DRAIN, detail);
      return false;
    }
  }
  return true;
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_kernel(const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar0 = s_base + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  auto stage_a = [&](int s) { return s_base + static_cast<uint32_t>(s * STAGE_BYTES); };
  auto stage_b = [&](int s) { return s_base + static_cast<uint32_t>(s * STAGE_BYTES + TILE_BYTES); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int ntiles = p.N / BN;
  const int total = __ldg(p.tile_offs + p.G) * ntiles;
  const int k64 = p.K >> 6;
  const int nkt = (k64 + 3) >> 2;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t ph = 0;
      uint32_t pending = 0, pend_par = 0;  // per-stage: load issued, parity of that phase
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile x = decode_tile(t, p, ntiles);
        const uint8_t* a_chunk = p.a + static_cast<size_t>(x.mt) * nkt * TILE_BYTES;
        const uint8_t* b_chunk = p.b + (static_cast<size_t>(x.g) * ntiles + x.nt) * nkt * TILE_BYTES;
        // rows of A to fetch: the valid ones, rounded up to the 8-row swizzle group
        const uint32_t a_code_bytes = static_cast<uint32_t>(min(BM, (x.rows + 7) & ~7)) * 128u;
        for (int kt = 0; kt < nkt; ++kt) {
          if (!mbar_wait(empty_bar(stage), ph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_PRODUCER, t)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), a_code_bytes + TILE_SF_BYTES + TILE_BYTES);
          const uint8_t* ac = a_chunk + static_cast<size_t>(kt) * TILE_BYTES;
          if (a_code_bytes == TILE_CODE_BYTES) {
            bulk_load(stage_a(stage), ac, TILE_BYTES, full_bar(stage));
          } else {
            bulk_load(stage_a(stage), ac, a_code_bytes, full_bar(stage));
            bulk_load(stage_a(stage) + TILE_CODE_BYTES, ac + TILE_CODE_BYTES, TILE_SF_BYTES, full_bar(stage));
          }
          bulk_load(stage_b(stage), b_chunk + static_cast<size_t>(kt) * TILE_BYTES, TILE_BYTES, full_bar(stage));
          pending |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (ph << stage);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok || *abort_flag) {
        // Let every copy this thread issued land before the CTA goes away.
        for (int s = 0; s < STAGES; ++s)
          if ((pending >> s) & 1u) mbar_wait_drain(full_bar(s), (pend_par >> s) & 1u, p.err, s);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = mxf4nvf4_idesc(BM, BN);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      int i = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++i) {
        const int buf = i & 1;
        if (!mbar_wait(acce_bar(buf), ((i >> 1) & 1) ^ 1u, abort_flag, p.err, DEV_TIMEOUT_MMA, t)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int kt = 0; kt < nkt; ++kt) {
          if (!mbar_wait(full_bar(stage), ph, abort_flag, p.err, DEV_TIMEOUT_MMA, t)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int na = min(4, k64 - kt * 4);
          const uint32_t sfa_t = tmem + SF_COL0 + stage * 32;
          const uint32_t sfb_t = sfa_t + 16;
          const uint32_t a_s = stage_a(stage), b_s = stage_b(stage);
          for (int kk = 0; kk < na; ++kk) {
            tc_copy_sf_atom(sfa_t + kk * 4, sf_atom_desc(a_s + TILE_CODE_BYTES + kk * 512));
            tc_copy_sf_atom(sfb_t + kk * 4, sf_atom_desc(b_s + TILE_CODE_BYTES + kk * 512));
          }
          for (int kk = 0; kk < na; ++kk) {
            tc_mma_nvfp4(d_tmem, operand_desc_sw128(a_s + kk * 32), operand_desc_sw128(b_s + kk * 32), idesc,
                         sfa_t + kk * 4, sfb_t + kk * 4, (kt | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (ok) tc_commit(accf_bar(buf));
      }
      // Every MMA / copy this thread issued must finish before TMEM is freed.
      tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.err, -1);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;       // which 64 of the tile's 128 columns
    const int r = q * 32 + lane;            // tile row handled by this thread
    int i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const Tile x = decode_tile(t, p, ntiles);
      const int buf = i & 1;
      if (!mbar_wait(accf_bar(buf), (i >> 1) & 1, abort_flag, p.err, DEV_TIMEOUT_EPILOGUE, t)) break;
      tc_fence_after();
      if (q * 32 < x.rows) {
        const uint32_t tb = tmem + buf * BN + half * 64 + (static_cast<uint32_t>(q * 32) << 16);
        const float alpha = __fmul_rn(__ldg(p.gs_a + x.g), __ldg(p.gs_b + x.g));
        const bool valid = r < x.rows;
        const int64_t row = static_cast<int64_t>(x.row0) + r;
        if constexpr (EPI == EPI_SWIGLU_QUANT) {
          const int I = p.N >> 1;
          const float gsq = __ldg(p.gs_q + x.g);
          const float six_gsq = __fmul_rn(6.0f, gsq);
          uint32_t cw[4];
          uint32_t sfw = 0;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
            tmem_ld32(tb + cc * 32, v);
            tmem_ld_wait();
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              // rows past the group's end carry whatever their scale bytes held: use zeros
              const float g = valid ? __fmul_rn(__uint_as_float(v[j]), alpha) : 0.0f;
              const float u = valid ? __fmul_rn(__uint_as_float(v[16 + j]), alpha) : 0.0f;
              h[j] = __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u);
            }
            const int c = half * 2 + cc;   // 16-wide block of this n-tile's 64 h values
            if (p.h_dump != nullptr && valid) {
              float4* hd = reinterpret_cast<float4*>(p.h_dump + row * I + x.nt * 64 + c * 16);
#pragma unroll
              for (int j = 0; j < 4; ++j) hd[j] = make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
            }
            sfw |= quant_block16(h, gsq, six_gsq, cw[2 * cc], cw[2 * cc + 1]) << (8 * cc);
          }
          // A2 is the down GEMM's A operand (TILED_GROUPED, K = I): this n-tile's 64
          // h values are MMA step nt % 4 of K tile nt / 4; this warp's 32 of them
          // are one 16-byte code chunk and two scale bytes of row r.
          uint8_t* chunk = p.q_codes + (static_cast<size_t>(x.mt) * num_k_tiles(I) + (x.nt >> 2)) * TILE_BYTES;
          if (valid)
            *reinterpret_cast<uint4*>(chunk + tiled_code_offset(r, (x.nt & 3) * 32 + half * 16)) =
                make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t*>(chunk + TILE_CODE_BYTES + (x.nt & 3) * 512 +
                                       sf_atom_offset(static_cast<uint32_t>(r), half * 2)) =
              static_cast<uint16_t>(sfw);
        } else {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
            tmem_ld32(tb + cc * 32, v);
            tmem_ld_wait();
            if (valid) {
              const int64_t col = static_cast<int64_t>(x.nt) * BN + half * 64 + cc * 32;
              if constexpr (EPI == EPI_STORE_F32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.d) + row * p.ldd + col);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  dst[j] = make_float4(__fmul_rn(__uint_as_float(v[4 * j]), alpha),
                                       __fmul_rn(__uint_as_float(v[4 * j + 1]), alpha),
                                       __fmul_rn(__uint_as_float(v[4 * j + 2]), alpha),
                                       __fmul_rn(__uint_as_float(v[4 * j + 3]), alpha));
              } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.d) + row * p.ldd + col);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t w[4];
#pragma unroll
                  for (int h2 = 0; h2 < 4; ++h2) {
                    __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[8 * j + 2 * h2]), alpha),
                                                             __fmul_rn(__uint_as_float(v[8 * j + 2 * h2 + 1]), alpha));
                    w[h2] = *reinterpret_cast<uint32_t*>(&b);
                  }
                  dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int EPI>
cudaError_t launch_epi(const GemmArgs& a, int grid, cudaStream_t s) {
  auto k = grouped_gemm_kernel<EPI>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  k<<<grid, THREADS, SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s, const char** why) {
  *why = nullptr;
  if (a.a_rows <= 0) return cudaSuccess;
  const int64_t max_tiles = ((a.a_rows + BM - 1) / BM + a.G) * (a.N / BN);
  int grid = a.max_ctas > 0 ? a.max_ctas : sm_count();
  if (grid > max_tiles) grid = static_cast<int>(max_tiles);
  if (grid < 1) grid = 1;
  switch (a.epilogue) {
    case EPI_STORE_F32: return launch_epi<EPI_STORE_F32>(a, grid, s);
    case EPI_STORE_BF16: return launch_epi<EPI_STORE_BF16>(a, grid, s);
    case EPI_SWIGLU_QUANT: return launch_epi<EPI_SWIGLU_QUANT>(a, grid, s);
    default: *why = "unknown epilogue"; return cudaErrorInvalidValue;
  }
}

}  // namespace nvf
