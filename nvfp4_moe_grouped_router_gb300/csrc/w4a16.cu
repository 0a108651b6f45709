// Weight-only NVFP4 grouped GEMM (W4A16) for sm_103a:
//     D[row, n] = gs_b[g] * sum_k a[row, k] * dB_g[n, k]   for offsets[g] <= row < offsets[g+1]
// with FP16 activations a (BF16 ones are rounded to FP16 in the kernel) and NVFP4 weights dB = e2m1 * e4m3 dequantized in the
// kernel and multiplied on the tensor cores as FP16 (tcgen05.mma kind::f16).
// This is the decode alternative the pages keep comparing with the W4A4 path:
// W4A16 unpacks FP4 weights and runs FP16 MMA (unsloth report, SASS paragraph
// under "Why it matters"; Marlin W4A16 in FlashInfer issue #2723, "Speed
// Comparison").  Every e2m1 * e4m3 product is exact in FP16 (at most 6
// significant bits, 2^-10 .. 2688), so the dequantized weights lose nothing.
//
// The product is computed transposed, D^T = dB * a^T: the weights are the MMA's
// A operand, and A may sit in tensor memory.  The dequantized FP16 weights go
// from registers straight into TMEM (tcgen05.st) and never touch shared memory,
// whose bandwidth would otherwise bound the kernel (two FP16 bytes written and
// read per weight against 0.56 bytes streamed from HBM).  The tokens of a
// 128-row token tile are the MMA's N (16 .. 128, rounded up to 16), so a decode
// group of one or two tokens costs an N = 16 MMA.
//
// Persistent CTAs, one per SM, take work items (128-row token tile, 256-row
// weight pair) in turn.  Roles (NW warps):
//   RAW_WARP     streams the pair's raw weight units (one 36864-byte bulk copy
//                per 256-element K tile, the TILED layout) into a 4-stage ring;
//   ACT_WARP     copies the token tile's activations (cp.async, 16 bytes a lane)
//                into 128-byte-swizzled K-major rows, one 64-element K step a
//                16 KB stage (4 stages), completing each stage's mbarrier;
//   CVT_WARP     BF16 activations only: waits for each landed stage, rounds it
//                to FP16 in place and completes the stage for the MMA (so the
//                copies stay as deep in flight as for FP16 rows);
//   warps 0-15   convert: warpgroup (par, j) owns weight tile j of the pair for
//                the K steps of parity par, thread (quarter q, lane l) its row
//                32 q + l: per K step it reads the row's 32 code bytes and 4
//                scale bytes, converts them (cvt e2m1x2 -> f16x2, times the e4m3
//                scale) and writes the 64 FP16 values into its TMEM lane, 32
//                columns of one of 4 slots;
//   MMA warps    one thread per (weight tile j, accumulator) issues the step's
//                four 128 x N x 16 MMAs (A from TMEM, B the activation stage)
//                and commits the step.  A single thread needs ~57 cycles to
//                issue one tcgen05.mma, and at N = 16 a step's 8 MMAs would
//                otherwise take longer than its HBM time;
//   EPI warps    the epilogue: accumulator -> registers, times gs_b[g], stored
//                as D rows (each warp writes 32 consecutive columns a token).
// TMEM (512 columns): tile j's accumulator at columns 128 j, the weight slots
// at 256 + 64 s + 32 j.  The MMAs of step s commit to mma_done[s % 4], which
// frees both the activation stage and the TMEM slot.  Rows of an activation
// stage past the tile's tokens hold stale values: they only feed accumulator
// columns that are never stored.  Every wait is bounded; a failed wait raises
// the CTA's abort flag and every role leaves (no role waits at a barrier that
// another role could leave).
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvf {
namespace {

constexpr int DQ_WARPS = 16;
constexpr int MMA_WARP0 = 16, N_MMA = 2, EPI_WARP0 = MMA_WARP0 + N_MMA, RAW_WARP = EPI_WARP0 + 4, ACT_WARP = RAW_WARP + 1;
constexpr int CVT_WARP = ACT_WARP + 1;            // BF16 activations: rounds each landed stage to FP16
constexpr int W_THREADS = 32 * (CVT_WARP + 1);
constexpr int RAW_STAGES = 4;
constexpr int RAW_STAGE = 2 * TILE_BYTES;        // 36864: one K tile of a weight pair
constexpr int SLOTS = 4;                         // activation stages = TMEM weight slots
constexpr int ACT_STAGE = TILE_ROWS * 128;       // 16 KB: 128 token rows x 64 fp16
constexpr int TMEM_COLS = 512;
constexpr int A_COL = 256;
constexpr int OFF_ACT = RAW_STAGES * RAW_STAGE;  // 147456
constexpr int OFF_BAR = OFF_ACT + SLOTS * ACT_STAGE;
// raw_full[4] raw_empty[4] act_full[4] a_full[4] mma_done[4] d_full d_empty drain[N_MMA] act_landed[4]
constexpr int NUM_BARS = 2 * RAW_STAGES + 4 * SLOTS + 2 + N_MMA;
constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
constexpr int W_SMEM = OFF_MISC + 16 + 1024;     // + alignment slack

// Four bytes of E2M1 code pairs (low nibble = lower element) -> four f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}
// Four E4M3 scale bytes -> each as an FP16 pair (both halves the same value).
__device__ __forceinline__ void e4m3x4_to_f16x2_dup(uint32_t s, uint32_t (&h)[4]) {
  const uint32_t lo = __byte_perm(s, 0, 0x1100), hi = __byte_perm(s, 0, 0x3322);
  asm("{\n .reg .b16 a, b, c, d;\n mov.b32 {a, b}, %4;\n mov.b32 {c, d}, %5;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n"
      " cvt.rn.f16x2.e4m3x2 %2, c;\n cvt.rn.f16x2.e4m3x2 %3, d;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(lo), "r"(hi));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

struct W16Args {
  const __half* a;          // FP16 rows, or BF16 rows when a_bf16 (16-bit elements either way)
  int a_bf16;
  int64_t a_rows, lda;
  const uint8_t* b;
  const float* gs_b;
  const int32_t* offsets;
  const int32_t* tile_offs;
  int G, N, K;
  int out_bf16;
  void* d;
  int64_t ldd;
  int* err;
};

// Work item = (128-row token tile mt, weight pair p).
struct Item {
  int g, row0, rows, p, tiles;
};
__device__ __forceinline__ Item decode_item(int item, int n_pairs, int ntg, const W16Args& a) {
  Item x;
  const int mt = item / n_pairs;
  x.p = item - mt * n_pairs;
  x.g = upper_group(a.tile_offs, a.G, mt);
  x.row0 = __ldg(a.offsets + x.g) + (mt - __ldg(a.tile_offs + x.g)) * TILE_ROWS;
  x.rows = min(TILE_ROWS, __ldg(a.offsets + x.g + 1) - x.row0);
  if (x.rows <= 0 || x.row0 < 0 || x.row0 + x.rows > a.a_rows) x.rows = 0;   // inconsistent tables: no rows
  x.tiles = 2 * x.p + 1 < ntg ? 2 : 1;
  return x;
}

__global__ void __launch_bounds__(W_THREADS, 1) w4a16_kernel(const W16Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar0 = s_base + OFF_BAR;
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto raw_empty = [&](int s) { return bar0 + 8u * (RAW_STAGES + s); };
  auto act_full = [&](int s) { return bar0 + 8u * (2 * RAW_STAGES + s); };
  auto a_full = [&](int s) { return bar0 + 8u * (2 * RAW_STAGES + SLOTS + s); };
  auto mma_done = [&](int s) { return bar0 + 8u * (2 * RAW_STAGES + 2 * SLOTS + s); };
  const uint32_t d_full = bar0 + 8u * (2 * RAW_STAGES + 3 * SLOTS), d_empty = d_full + 8, drain_bar0 = d_full + 16;
  auto act_landed = [&](int s) { return drain_bar0 + 8u * (N_MMA + s); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_empty(s), DQ_WARPS);
    }
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(act_full(s), 32);
      mbar_init(a_full(s), DQ_WARPS / 2);                 // the 8 warps of the step's parity
      mbar_init(mma_done(s), N_MMA);
      mbar_init(act_landed(s), 32);
    }
    mbar_init(d_full, N_MMA);
    mbar_init(d_empty, 4);
    for (int i = 0; i < N_MMA; ++i) mbar_init(drain_bar0 + 8 * i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP0) tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int ntg = a.N / TILE_ROWS, n_pairs = (ntg + 1) >> 1;
  const int nks = a.K >> 6, nkt = num_k_tiles(a.K);
  const int total = __ldg(a.tile_offs + a.G) * n_pairs;

  if (warp == RAW_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------------- raw weights
      uint32_t kc = 0, pending = 0, pend_par = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const Item x = decode_item(it, n_pairs, ntg, a);
        const uint8_t* unit0 = a.b + (static_cast<size_t>(x.g) * ntg + 2 * x.p) * nkt * TILE_BYTES;
        const uint32_t bytes = static_cast<uint32_t>(x.tiles) * TILE_BYTES;
        for (int kt = 0; kt < nkt; ++kt, ++kc) {
          const int s = kc % RAW_STAGES;
          const uint32_t ph = (kc / RAW_STAGES) & 1u;
          if (!mbar_wait(raw_empty(s), ph ^ 1u, abort_flag, a.err, DEV_TIMEOUT_PRODUCER, it)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(raw_full(s), bytes);
          bulk_load(s_base + s * RAW_STAGE, unit0 + static_cast<size_t>(kt) * bytes, bytes, raw_full(s));
          pending |= 1u << s;
          pend_par = (pend_par & ~(1u << s)) | (ph << s);
        }
      }
      if (!ok || *abort_flag) {
        // Let every copy this thread issued land before the CTA goes away.
        for (int s = 0; s < RAW_STAGES; ++s)
          if ((pending >> s) & 1u) mbar_wait_drain(raw_full(s), (pend_par >> s) & 1u, a.err, s);
      }
    }
  } else if (warp == ACT_WARP) {
    // ------------------------------------------------------------------ activations
    uint32_t sc = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
      const Item x = decode_item(it, n_pairs, ntg, a);
      const __half* arow = a.a + static_cast<int64_t>(x.row0) * a.lda;
      for (int ks = 0; ks < nks; ++ks, ++sc) {
        const int s = sc % SLOTS;
        // the stage was last read by the MMAs of step sc - SLOTS
        const bool got = mbar_wait(mma_done(s), ((sc / SLOTS) & 1u) ^ 1u, abort_flag, a.err, DEV_TIMEOUT_PRODUCER, it);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t st = s_base + OFF_ACT + s * ACT_STAGE;
        for (int q = lane; q < x.rows * 8; q += 32) {
          const int r = q >> 3, c = q & 7;
          cp_async16(st + r * 128 + ((c ^ (r & 7)) << 4), arow + static_cast<int64_t>(r) * a.lda + ks * 64 + c * 8);
        }
        // FP16 rows are the MMA's operand as they land; BF16 rows go to the
        // rounding warp first
        cp_async_mbar_arrive(a.a_bf16 ? act_landed(s) : act_full(s));
      }
    }
    cp_async_wait_all();
  } else if (warp == CVT_WARP) {
    // ------------------------------------------------------------------ BF16 -> FP16
    // Each lane rounds the 16-byte chunks of a landed stage (BF16 pairs -> FP16
    // pairs, to nearest) in place; then the stage is the MMA's operand.
    if (a.a_bf16) {
      uint32_t sc = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const Item x = decode_item(it, n_pairs, ntg, a);
        for (int ks = 0; ks < nks; ++ks, ++sc) {
          const int s = sc % SLOTS;
          const bool got = mbar_wait(act_landed(s), (sc / SLOTS) & 1u, abort_flag, a.err, DEV_TIMEOUT_PRODUCER, it);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint32_t st = s_base + OFF_ACT + s * ACT_STAGE;
          for (int q = lane; q < x.rows * 8; q += 32) {
            const int r = q >> 3, c = q & 7;
            const uint32_t addr = st + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(addr)
                         : "memory");
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 v = __floats2half2_rn(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
              w[e] = *reinterpret_cast<const uint32_t*>(&v);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
          }
          fence_proxy_async();                  // the MMA reads the stage through the async proxy
          mbar_arrive(act_full(s));
        }
      }
    }
  } else if (warp >= MMA_WARP0 && warp < EPI_WARP0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuers
      // Thread j issues weight tile j's MMAs; on an item with one weight tile,
      // thread 1 waits and commits all the same, so that every barrier phase
      // gets one arrival from each.
      const int j = warp - MMA_WARP0;
      uint32_t sc = 0, n_items = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x, ++n_items) {
        const Item x = decode_item(it, n_pairs, ntg, a);
        const uint32_t idesc = f16kind_idesc(TILE_ROWS, max(16, (x.rows + 15) & ~15), false);
        // the epilogue has moved the previous item's accumulators out of TMEM
        if (!mbar_wait(d_empty, (n_items & 1u) ^ 1u, abort_flag, a.err, DEV_TIMEOUT_MMA, it)) break;
        for (int ks = 0; ks < nks; ++ks, ++sc) {
          const int s = sc % SLOTS;
          const uint32_t ph = (sc / SLOTS) & 1u;
          if (!mbar_wait(act_full(s), ph, abort_flag, a.err, DEV_TIMEOUT_MMA, it) ||
              !mbar_wait(a_full(s), ph, abort_flag, a.err, DEV_TIMEOUT_MMA, it)) {
            ok = false;
            break;
          }
          if (j < x.tiles) {
            // the stage was written by cp.async (generic proxy); the MMA reads it
            // through the async proxy
            fence_proxy_async();
            tc_fence_after();
            // K step kk: 32 bytes further into the swizzled rows (start address field + 2)
            const uint64_t bdesc = operand_desc_sw128(s_base + OFF_ACT + s * ACT_STAGE);
            const uint32_t d_tm = tmem + 128 * j, a_tm = tmem + A_COL + 64 * s + 32 * j;
            tc_mma_f16kind_ts(d_tm, a_tm, bdesc, idesc, ks != 0 ? 1u : 0u);
            tc_mma_f16kind_ts(d_tm, a_tm + 8, bdesc + 2, idesc, 1u);
            tc_mma_f16kind_ts(d_tm, a_tm + 16, bdesc + 4, idesc, 1u);
            tc_mma_f16kind_ts(d_tm, a_tm + 24, bdesc + 6, idesc, 1u);
          }
          tc_commit(mma_done(s));
        }
        if (ok) tc_commit(d_full);
      }
      // Every MMA this thread issued must finish before TMEM is freed.
      tc_commit(drain_bar0 + 8 * j);
      mbar_wait_drain(drain_bar0 + 8 * j, 0, a.err, -1);
    }
  } else if (warp < DQ_WARPS) {
    // ------------------------------------------------------------------ converters
    const int j = (warp >> 2) & 1, par = warp >> 3, q = warp & 3, r = q * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    uint32_t sc = 0, kc = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
      const Item x = decode_item(it, n_pairs, ntg, a);
      const bool mine = j < x.tiles;
      const uint32_t codes_off = static_cast<uint32_t>(j) * TILE_CODE_BYTES;
      const uint32_t atoms_off = static_cast<uint32_t>(x.tiles) * TILE_CODE_BYTES + j * TILE_SF_BYTES;
      for (int kt = 0; kt < nkt && ok; ++kt, ++kc) {
        const int rs = kc % RAW_STAGES;
        const bool got = mbar_wait(raw_full(rs), (kc / RAW_STAGES) & 1u, abort_flag, a.err, DEV_TIMEOUT_PRODUCER, it);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t raw = s_base + rs * RAW_STAGE;
        const int steps = min(4, nks - 4 * kt);
        for (int ks = par; ks < steps; ks += 2) {
          const uint32_t step = sc + ks;
          const int s = step % SLOTS;
          // TMEM slot s was last read by the MMAs of step - SLOTS
          const bool free_ = mbar_wait(mma_done(s), ((step / SLOTS) & 1u) ^ 1u, abort_flag, a.err, DEV_TIMEOUT_MMA, it);
          if (!__all_sync(0xffffffffu, free_)) {
            ok = false;
            break;
          }
          if (mine) {
            tc_fence_after();
            const uint4 c0 = lds128(raw + codes_off + tiled_code_offset(r, ks * 32));
            const uint4 c1 = lds128(raw + codes_off + tiled_code_offset(r, ks * 32 + 16));
            const uint32_t sfw = lds32(raw + atoms_off + ks * 512 + sf_atom_offset(r, 0));
            uint32_t sc2[4];
            e4m3x4_to_f16x2_dup(sfw, sc2);
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t v[32];
#pragma unroll
            for (int w = 0; w < 8; ++w) {                     // word w: elements 8 w .. 8 w + 7
              uint32_t h[4];
              e2m1x8_to_f16x2(cw[w], h);
#pragma unroll
              for (int e = 0; e < 4; ++e) v[4 * w + e] = hmul2_u32(h[e], sc2[w >> 1]);
            }
            tmem_st32(tmem + lanes + A_COL + 64 * s + 32 * j, v);
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(a_full(s));
        }
        sc += steps;
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty(rs));
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint32_t n_items = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x, ++n_items) {
      const Item x = decode_item(it, n_pairs, ntg, a);
      const float alpha = __ldg(a.gs_b + x.g);
      if (!mbar_wait(d_full, n_items & 1u, abort_flag, a.err, DEV_TIMEOUT_EPILOGUE, it)) break;
      tc_fence_after();
      const int nchunks = (max(x.rows, 1) + 31) >> 5;
      for (int j = 0; j < x.tiles; ++j) {
        const int64_t col = static_cast<int64_t>(2 * x.p + j) * TILE_ROWS + q * 32 + lane;
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + 128 * j + 32 * c, v);
          tmem_ld_wait();
          if (j == x.tiles - 1 && c == nchunks - 1) {
            // both accumulators are in registers or stored: release them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty);
          }
          const int n_here = min(32, x.rows - 32 * c);
          const int64_t row = static_cast<int64_t>(x.row0) + 32 * c;
          if (a.out_bf16) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.d) + row * a.ldd + col;
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (t < n_here) dst[t * a.ldd] = __float2bfloat16_rn(__fmul_rn(__uint_as_float(v[t]), alpha));
          } else {
            float* dst = static_cast<float*>(a.d) + row * a.ldd + col;
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (t < n_here) dst[t * a.ldd] = __fmul_rn(__uint_as_float(v[t]), alpha);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_w4a16(const void* A, int a_bf16, int64_t a_rows, int64_t lda, const uint8_t* B, const float* gs_b,
                         const int32_t* offsets, const int32_t* tile_offs, int32_t G, int32_t N, int32_t K,
                         int out_bf16, void* D, int64_t ldd, int* err, cudaStream_t s) {
  if (a_rows <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, W_SMEM);
  if (e != cudaSuccess) return e;
  prefer_max_shared(reinterpret_cast<const void*>(w4a16_kernel));
  const int64_t n_pairs = (N / TILE_ROWS + 1) / 2;
  const int64_t max_items = ((a_rows + TILE_ROWS - 1) / TILE_ROWS + G) * n_pairs;
  const int grid = static_cast<int>(max_items < sm_count() ? max_items : sm_count());
  W16Args args{static_cast<const __half*>(A), a_bf16, a_rows, lda, B, gs_b, offsets, tile_offs, G, N, K, out_bf16, D,
               ldd, err};
  w4a16_kernel<<<grid, W_THREADS, W_SMEM, s>>>(args);
  return cudaGetLastError();
}

}  // namespace nvf
