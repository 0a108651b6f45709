// Router gate GEMM (the step before routing): logits[t, j] = sum_h x[t, h] *
// w_gate[j, h] for BF16 activations and gate rows, FP32 accumulate, on the 5th
// generation tensor cores (tcgen05.mma kind::f16, both operands BF16).
//
// The pages name the routed experts the gate scores (FlashInfer issue #2723,
// "Model" table: 512 routed + 1 shared expert, 10 routed per token) but give
// no gate formula; the reading is a plain linear gate, one row per routed
// expert, plus optionally one row whose logit gates the shared expert.
//
// One CTA per 128 tokens x 32 gate rows, 128 threads.  K advances in blocks of
// 64 elements (one 128-byte row per token / gate row): every thread copies
// 16-byte pieces with cp.async into a 4-stage ring laid out the way the MMA
// reads K-major operands with the 128-byte swizzle; after the async-proxy
// fence, one thread issues four 128x32x16 MMAs per block into a 32-column TMEM
// accumulator and commits the stage.  Rows past T and gate rows past n are
// zero-filled.  The epilogue moves each warp's 32 TMEM lanes to registers and
// stores the FP32 logits.  Every wait is bounded.
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int RM = 128;                   // tokens per CTA
constexpr int RN = 32;                    // gate rows per CTA (MMA N)
constexpr int RK = 64;                    // K elements per block (128 bytes)
constexpr int RSTAGES = 4;
constexpr int R_THREADS = 128;
constexpr int A_STAGE = RM * 128;         // 16 KB
constexpr int B_STAGE = RN * 128;         // 4 KB
constexpr int R_SMEM = RSTAGES * (A_STAGE + B_STAGE) + 1024 + 64;

// Instruction descriptor of a kind::f16 MMA: D FP32 (bits 4-5 = 1), A and B
// BF16 (bits 7-9 and 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t bf16_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Shared-memory writes made by these threads become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
}

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

  // Stage s <- K block kb: 1024 pieces of A (token rows), 256 of B (gate rows).
  auto load_stage = [&](int kb) {
    const int s = kb % RSTAGES;
#pragma unroll
    for (int i = 0; i < (RM * 8) / R_THREADS; ++i) {
      const int p = tid + R_THREADS * i, r = p >> 3, c = p & 7;
      const uint32_t dst = a0 + s * A_STAGE + r * 128 + ((c ^ (r & 7)) << 4);
      if (m0 + r < T) cp_async16(dst, x + static_cast<int64_t>(m0 + r) * H + kb * RK + c * 8);
      else st_shared_zero16(dst);
    }
#pragma unroll
    for (int i = 0; i < (RN * 8) / R_THREADS; ++i) {
      const int p = tid + R_THREADS * i, r = p >> 3, c = p & 7;
      const uint32_t dst = b0 + s * B_STAGE + r * 128 + ((c ^ (r & 7)) << 4);
      if (n0 + r < n) cp_async16(dst, wg + static_cast<int64_t>(n0 + r) * H + kb * RK + c * 8);
      else st_shared_zero16(dst);
    }
  };

  const uint32_t idesc = bf16_idesc(RM, RN);
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
      for (int kk = 0; kk < RK / 16; ++kk)
        tc_mma_bf16(tmem, operand_desc_sw128(a0 + s * A_STAGE + kk * 32), operand_desc_sw128(b0 + s * B_STAGE + kk * 32),
                    idesc, (kb | kk) != 0 ? 1u : 0u);
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
    uint32_t v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
    tmem_ld_wait();
    const int row = m0 + warp * 32 + lane;
    if (row < T) {
      float* dst = logits + static_cast<int64_t>(row) * ldl + n0;
#pragma unroll
      for (int j = 0; j < RN; ++j)
        if (n0 + j < n) dst[j] = __uint_as_float(v[j]);
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

}  // namespace

cudaError_t launch_router_gemm(const void* x, const void* w_gate, int32_t T, int32_t H, int32_t n, float* logits,
                               int64_t ldl, int* err, cudaStream_t s) {
  if (T == 0 || n == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((T + RM - 1) / RM, (n + RN - 1) / RN);
  router_gemm_kernel<<<grid, R_THREADS, R_SMEM, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                      static_cast<const __nv_bfloat16*>(w_gate), T, H, n, logits,
                                                      ldl, err);
  return cudaGetLastError();
}

}  // namespace nvf
