// Router gate GEMM (the step before routing): logits[t, j] = sum_h x[t, h] *
// w_gate[j, h] for BF16 activations and gate rows, FP32 accumulate, on the 5th
// generation tensor cores (tcgen05.mma kind::f16, both operands BF16).
//
// The pages name the routed experts the gate scores (FlashInfer issue #2723,
// "Model" table: 512 routed + 1 shared expert, 10 routed per token) but give
// no gate formula; the reading is a plain linear gate, one row per routed
// expert, plus optionally one row whose logit gates the shared expert.
//
// Above 64 tokens: one CTA per 128 tokens x 32 gate rows, 128 threads (the
// most CTAs, which measured fastest: the per-CTA ring is load-latency-bound).
// K advances in blocks of 64 elements, one 64-element swizzle atom of 128-byte
// rows: every thread copies 16-byte pieces with cp.async into a 4-stage ring
// (80 KB: two CTAs a SM) laid out the way the MMA reads K-major operands with
// the 128-byte swizzle; after the async-proxy fence, one thread issues four
// 128x32x16 MMAs per block into a 32-column TMEM accumulator and commits the
// stage.  Rows past T and gate rows past n are zero-filled once, while the ring
// first fills.  The epilogue moves each warp's 32 TMEM lanes to registers and
// stores the FP32 logits.  Every wait is bounded.
//
// Up to 64 tokens the same logits come from CUDA cores, one warp per (token,
// gate row): the tensor-core tile would be mostly padding and its per-block
// round trips, not arithmetic, would set the time.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int RM = 128;                   // tokens per CTA
constexpr int RN = 32;                    // gate rows per CTA (MMA N)
constexpr int RK = 64;                    // K elements per block: one 64-element swizzle atom
constexpr int RATOMS = RK / 64;
constexpr int RSTAGES = 4;
constexpr int R_THREADS = 128;
constexpr int A_ATOM = RM * 128;          // 16 KB: 128 rows x 128 bytes
constexpr int B_ATOM = RN * 128;          // 4 KB
constexpr int A_STAGE = RATOMS * A_ATOM;  // 16 KB
constexpr int B_STAGE = RATOMS * B_ATOM;  // 4 KB
constexpr int R_SMEM = RSTAGES * (A_STAGE + B_STAGE) + 1024 + 64;

__global__ void __launch_bounds__(R_THREADS) router_gemm_kernel(const __nv_bfloat16* __restrict__ x,
                                                                const __nv_bfloat16* __restrict__ wg, int T, int H,
                                                                int n, float* __restrict__ logits, int64_t ldl,
                                                                int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t a0 = s_base, b0 = s_base + RSTAGES * A_STAGE;
  const uint32_t bar0 = b0 + RSTAGES * B_STAGE;                 // mma_done[RSTAGES], then drain
  const uint32_t drain_bar = bar0 + 8 * RSTAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + RSTAGES * (A_STAGE + B_STAGE) + 8 * (RSTAGES + 1));
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s <= RSTAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_holder), RN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int m0 = blockIdx.x * RM, n0 = blockIdx.y * RN;
  const int nkb = H / RK;

  // Stage s <- K block kb: per row RK / 8 pieces of 16 bytes; piece c of row r
  // goes to atom c / 8 at row r's 128 bytes, 16-byte unit (c % 8) ^ (r % 8).
  // Rows past T / n are zeroed while the ring first fills and stay zero.
  auto load_stage = [&](int kb) {
    const int s = kb % RSTAGES;
    const bool first = kb < RSTAGES;
#pragma unroll
    for (int i = 0; i < (RM * RK / 8) / R_THREADS; ++i) {
      const int p = tid + R_THREADS * i, r = p / (RK / 8), c = p % (RK / 8);
      const uint32_t dst = a0 + s * A_STAGE + (c >> 3) * A_ATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4);
      if (m0 + r < T) cp_async16(dst, x + static_cast<int64_t>(m0 + r) * H + kb * RK + c * 8);
      else if (first) st_shared_zero16(dst);
    }
#pragma unroll
    for (int i = 0; i < (RN * RK / 8) / R_THREADS; ++i) {
      const int p = tid + R_THREADS * i, r = p / (RK / 8), c = p % (RK / 8);
      const uint32_t dst = b0 + s * B_STAGE + (c >> 3) * B_ATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4);
      if (n0 + r < n) cp_async16(dst, wg + static_cast<int64_t>(n0 + r) * H + kb * RK + c * 8);
      else if (first) st_shared_zero16(dst);
    }
  };

  const uint32_t idesc = f16kind_idesc(RM, RN, true);
  bool ok = true;
  for (int kb = 0; kb < RSTAGES - 1; ++kb) {
    if (kb < nkb) load_stage(kb);
    cp_async_commit();
  }
  for (int kb = 0; kb < nkb && ok; ++kb) {
    const int s = kb % RSTAGES;
    cp_async_wait<RSTAGES - 2>();      // this thread's copies of block kb have landed
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < RK / 16; ++kk) {
        const int at = kk >> 2, ks = kk & 3;     // swizzle atom, 16-element step inside it
        tc_mma_f16kind(tmem, operand_desc_sw128(a0 + s * A_STAGE + at * A_ATOM + ks * 32),
                    operand_desc_sw128(b0 + s * B_STAGE + at * B_ATOM + ks * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      tc_commit(bar0 + 8 * s);
    }
    // Block kb + RSTAGES - 1 goes to the stage block kb - 1 used, once its MMAs are done.
    const int nk = kb + RSTAGES - 1;
    if (nk < nkb) {
      if (kb >= 1) {
        const int pk = kb - 1;
        ok = mbar_wait(bar0 + 8 * (pk % RSTAGES), (pk / RSTAGES) & 1, &abort_flag, err, DEV_TIMEOUT_MMA, blockIdx.x);
      }
      ok = __syncthreads_and(ok);       // every thread leaves together if a wait gave up
      if (ok) load_stage(nk);
    }
    cp_async_commit();
  }
  cp_async_wait<0>();
  // The last block's MMAs (and with them every earlier one) have completed.
  if (ok && nkb > 0)
    ok = mbar_wait(bar0 + 8 * ((nkb - 1) % RSTAGES), ((nkb - 1) / RSTAGES) & 1, &abort_flag, err,
                   DEV_TIMEOUT_EPILOGUE, blockIdx.x);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
    const int row = m0 + warp * 32 + lane;
#pragma unroll
    for (int c = 0; c < RN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, v);
      tmem_ld_wait();
      if (row < T) {
        float* dst = logits + static_cast<int64_t>(row) * ldl + n0 + c * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (n0 + c * 32 + j < n) dst[j] = __uint_as_float(v[j]);
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
  if (warp == 0) tmem_dealloc(tmem, RN);
}

// One warp per (token t, gate row j): lane l sums the products of elements
// 8 l .. 8 l + 7 of every 256-element slice in order (FP32 FMA), then the warp
// adds the 32 partial sums in a fixed tree.  Grid: (n / 8 rounded up, T),
// 8 warps per CTA, one gate row each.
__global__ void __launch_bounds__(256) router_dot_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ wg, int T, int H, int n,
                                                         float* __restrict__ logits, int64_t ldl) {
  const int t = blockIdx.y, j = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (j >= n) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H);
  const uint4* wr = reinterpret_cast<const uint4*>(wg + static_cast<int64_t>(j) * H);
  float acc = 0.0f;
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 a = __ldg(xr + c), b = __ldg(wr + c);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc = fmaf(__uint_as_float(aw[q] << 16), __uint_as_float(bw[q] << 16), acc);
      acc = fmaf(__uint_as_float(aw[q] & 0xFFFF0000u), __uint_as_float(bw[q] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) logits[static_cast<int64_t>(t) * ldl + j] = acc;
}

}  // namespace

cudaError_t launch_router_gemm(const void* x, const void* w_gate, int32_t T, int32_t H, int32_t n, float* logits,
                               int64_t ldl, int* err, cudaStream_t s) {
  if (T == 0 || n == 0) return cudaSuccess;
  if (T <= 64) {
    router_dot_kernel<<<dim3((n + 7) / 8, T), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                           static_cast<const __nv_bfloat16*>(w_gate), T, H, n, logits,
                                                           ldl);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((T + RM - 1) / RM, (n + RN - 1) / RN);
  router_gemm_kernel<<<grid, R_THREADS, R_SMEM, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                      static_cast<const __nv_bfloat16*>(w_gate), T, H, n, logits,
                                                      ldl, err);
  return cudaGetLastError();
}

}  // namespace nvf
