// Router gate GEMM (the step before routing): logits[t, j] = sum_h x[t, h] *
// w_gate[j, h] for BF16 activations and gate rows, FP32 accumulate, on the 5th
// generation tensor cores (tcgen05.mma kind::f16, both operands BF16).
//
// The pages name the routed experts the gate scores (FlashInfer issue #2723,
// "Model" table: 512 routed + 1 shared expert, 10 routed per token) but give
// no gate formula; the reading is a plain linear gate, one row per routed
// expert, plus optionally one row whose logit gates the shared expert.
//
// Above 64 tokens: one CTA (8 warps) per 128 tokens x up to 256 gate rows
// (every gate row of a 128 + 1 row gate, so x is read once), K split over a
// cluster of S CTAs (S <= 8, chosen so that the grid fills the SMs).  Per
// 64-element K block one thread issues two TMA tensor copies
// (cp.async.bulk.tensor, 128-byte swizzle, rows past T and past n zero-filled
// by the copy) into a ring of up to 8 stages; another thread issues four
// 128 x NB x 16 MMAs (NB = the block's gate rows rounded up to 16) into a TMEM
// accumulator and commits the stage.  The cluster then sums its S partial
// tiles in a fixed order: the partial rows go into the shared memory of the
// CTA that owns them (128 / S rows a CTA; 16-byte remote stores, each warp
// instruction covering four rows' 128 contiguous bytes after a transpose
// through the warp's own shared memory), and after a cluster barrier each CTA
// adds the S partials of its rows, rank by rank, and stores the logits.  Every
// mbarrier wait is bounded; every thread reaches both cluster barriers.
// (Measured on the 4096-token batch: 4 us of copies and MMAs, 2 us of remote
// stores, 1 us of sums; ~10 us a call against 28 us for a cp.async ring of
// 32-row tiles without the K split.)
//
// Up to 64 tokens the same logits come from CUDA cores, one warp per (token,
// gate row): the tensor-core tile would be mostly padding and its per-block
// round trips, not arithmetic, would set the time.
#include "internal.h"
#include "ptx.cuh"

#include <cuda.h>   // CUtensorMap and its enums (types only: the encoder is fetched at run time)
#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int RM = 128;                   // tokens per CTA (MMA M)
constexpr int RN_MAX = 256;               // gate rows per CTA at most (MMA N)
constexpr int RK = 64;                    // K elements per block: one 128-byte swizzle atom a row
constexpr int R_THREADS = 256;           // 8 warps: two a TMEM lane quarter in the epilogue
constexpr int R_MAX_STAGES = 8;
constexpr int R_MAX_SPLIT = 8;            // cluster size (portable limit)
constexpr int A_STAGE = RM * 128;         // 16 KB: 128 token rows x 128 bytes
constexpr int R_RING = 200 * 1024;        // ring; after the MMAs, the partial tiles of the cluster's sum
constexpr int R_SMEM = R_RING + 1024 + 256;
// After the MMAs the ring holds the cluster's partial tiles (at 0: 128 rows of
// NB + 4 floats) and, behind them, each warp's 32 x 32 transpose buffer.
constexpr int R_STG_PITCH = 36;           // floats: 9 16-byte units, odd, so 16-byte accesses spread over the banks
constexpr int R_STG_OFF = RM * (RN_MAX + 4) * 4;
static_assert(R_STG_OFF + (R_THREADS / 32) * 32 * R_STG_PITCH * 4 <= R_RING,
              "partial-sum and transpose buffers must fit in the ring");

struct RouterArgs {
  int T, n;
  int box_rows;      // gate rows a w_gate copy brings (the tensor map's box): min(256, n rounded up to 16)
  int kblocks;       // 64-element K blocks of one CTA's slice
  float* logits;
  int64_t ldl;
  int* err;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of this CTA's shared-memory location `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

__global__ void __launch_bounds__(R_THREADS, 1) router_gemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                                   const __grid_constant__ CUtensorMap tm_w,
                                                                   const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_addr(smem);
  const int b_stage = a.box_rows * 128;
  const int stage_bytes = A_STAGE + b_stage;               // a multiple of 2048 (box_rows % 16 == 0)
  const int stages = min(R_MAX_STAGES, R_RING / stage_bytes);
  const uint32_t bar0 = s_base + R_RING;                   // full[8], empty[8], acc_full, drain
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (R_MAX_STAGES + s); };
  const uint32_t accf_bar = bar0 + 8u * (2 * R_MAX_STAGES), drain_bar = accf_bar + 8u;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + R_RING + 8 * (2 * R_MAX_STAGES + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + R_RING + 8 * (2 * R_MAX_STAGES + 2) + 4);
  auto a_addr = [&](int s) { return s_base + static_cast<uint32_t>(s * stage_bytes); };
  auto b_addr = [&](int s) { return s_base + static_cast<uint32_t>(s * stage_bytes + A_STAGE); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < R_MAX_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_holder), RN_MAX);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int S = static_cast<int>(gridDim.z);
  const int z = static_cast<int>(cluster_rank());          // == blockIdx.z: clusters are 1 x 1 x S
  const int m0 = blockIdx.x * RM, n0 = blockIdx.y * RN_MAX;
  const int NB = min(RN_MAX, (a.n - n0 + 15) & ~15);       // this CTA's MMA N
  const int k0 = z * a.kblocks * RK;

  uint32_t pending = 0, pend_par = 0;                      // producer: per stage, a copy issued and its parity
  if (warp == 0 && lane == 0) {
    // -------------------------------------------------------------- producer
    for (int kb = 0; kb < a.kblocks; ++kb) {
      const int s = kb % stages;
      const uint32_t ph = (kb / stages) & 1u;
      if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, a.err, DEV_TIMEOUT_PRODUCER, blockIdx.x)) break;
      mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(stage_bytes));
      tma_load_2d(a_addr(s), &tm_x, k0 + kb * RK, m0, full_bar(s));
      tma_load_2d(b_addr(s), &tm_w, k0 + kb * RK, n0, full_bar(s));
      pending |= 1u << s;
      pend_par = (pend_par & ~(1u << s)) | (ph << s);
    }
  } else if (warp == 1 && lane == 0) {
    // -------------------------------------------------------------- MMA issuer
    const uint32_t idesc = f16kind_idesc(RM, NB, true);
    bool ok = true;
    for (int kb = 0; kb < a.kblocks; ++kb) {
      const int s = kb % stages;
      if (!mbar_wait(full_bar(s), (kb / stages) & 1u, abort_flag, a.err, DEV_TIMEOUT_MMA, blockIdx.x)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t da = operand_desc_sw128(a_addr(s)), db = operand_desc_sw128(b_addr(s));
      // K step kk: 32 bytes further into the swizzled rows (start address field + 2)
      tc_mma_f16kind(tmem, da, db, idesc, kb != 0 ? 1u : 0u);
      tc_mma_f16kind(tmem, da + 2, db + 2, idesc, 1u);
      tc_mma_f16kind(tmem, da + 4, db + 4, idesc, 1u);
      tc_mma_f16kind(tmem, da + 6, db + 6, idesc, 1u);
      tc_commit(empty_bar(s));
    }
    if (ok) tc_commit(accf_bar);
    // every MMA this thread issued completes before TMEM is freed
    tc_commit(drain_bar);
    mbar_wait_drain(drain_bar, 0, a.err, -1);
  }

  // ---------------------------------------------------------------- epilogue
  const bool got = mbar_wait(accf_bar, 0, abort_flag, a.err, DEV_TIMEOUT_EPILOGUE, blockIdx.x);
  const bool ok = __syncthreads_and(got) != 0;
  tc_fence_after();
  if (!ok && tid == 0) {
    // a wait gave up: every copy issued lands before the shared memory is reused or the CTA leaves
    for (int s = 0; s < stages; ++s)
      if ((pending >> s) & 1u) mbar_wait_drain(full_bar(s), (pend_par >> s) & 1u, a.err, s);
  }
  // Every CTA of the cluster is done with its ring (its copies landed, its MMAs
  // completed): the rings now hold the partial tiles.
  cluster_sync_all();
  const int rpo = RM / S;                                  // rows a CTA owns
  // floats a partial row: NB + 4, an odd number of 16-byte units, so that the
  // 16-byte stores of eight consecutive rows fall on distinct bank groups
  const int pitch = NB + 4;
  if (ok) {
    // Warps w and w + 4 share TMEM lane quarter w % 4 (rows 32 (w % 4) ..) and
    // take alternate 32-column chunks.  A chunk goes through 4.5 KB of the
    // warp's own shared memory so that each remote store instruction writes
    // four rows' 128 contiguous bytes.
    const int qd = warp & 3;
    const uint32_t stg = s_base + R_STG_OFF + static_cast<uint32_t>(warp * 32 * R_STG_PITCH * 4);
    const int rr0 = lane >> 3, piece = lane & 7;
    for (int c = 32 * (warp >> 2); c < NB; c += 64) {
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(qd * 32) << 16) + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(stg + static_cast<uint32_t>((lane * R_STG_PITCH + 4 * q) * 4), v[4 * q], v[4 * q + 1],
                     v[4 * q + 2], v[4 * q + 3]);
      __syncwarp();
      if (c + 4 * piece < NB) {
        // all eight loads first, then the eight stores
        uint4 d[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) d[i] = ld_shared_u4(stg + static_cast<uint32_t>(((4 * i + rr0) * R_STG_PITCH + 4 * piece) * 4));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = qd * 32 + 4 * i + rr0;
          const int owner = row / rpo, local = row - owner * rpo;
          const uint32_t at = s_base + static_cast<uint32_t>(((z * rpo + local) * pitch + c + 4 * piece) * 4);
          if (owner == z) st_shared_v4(at, d[i].x, d[i].y, d[i].z, d[i].w);   // own rows stay local
          else st_cluster_v4(map_shared(at, static_cast<uint32_t>(owner)), d[i].x, d[i].y, d[i].z, d[i].w);
        }
      }
      __syncwarp();
    }
  }
  cluster_sync_all();
  if (ok) {
    // rows z * rpo .. z * rpo + rpo - 1 of the tile: the S partials added rank
    // by rank, four consecutive logits a thread
    const int t0 = m0 + z * rpo;
    const int rows = min(rpo, a.T - t0), nq = NB / 4;
    for (int idx = tid; idx < rows * nq; idx += R_THREADS) {
      const int r = idx / nq, c = 4 * (idx - r * nq);
      uint4 v[R_MAX_SPLIT];
#pragma unroll
      for (int q = 0; q < R_MAX_SPLIT; ++q)
        if (q < S) v[q] = ld_shared_u4(s_base + static_cast<uint32_t>(((q * rpo + r) * pitch + c) * 4));
      float acc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[e] = __uint_as_float((&v[0].x)[e]);
#pragma unroll
        for (int q = 1; q < R_MAX_SPLIT; ++q)
          if (q < S) acc[e] = __fadd_rn(acc[e], __uint_as_float((&v[q].x)[e]));
      }
      float* dst = a.logits + static_cast<int64_t>(t0 + r) * a.ldl + n0 + c;
      const int left = a.n - n0 - c;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (e < left) dst[e] = acc[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, RN_MAX);
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

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no link against the driver library).
EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A [rows, H] bf16 matrix (row pitch H) read in boxes of 64 elements x box_rows rows, 128-byte swizzle.
cudaError_t encode_rows(CUtensorMap* map, const void* base, int64_t rows, int H, int box_rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(RK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
  const int mt = (T + RM - 1) / RM, nbk = (n + RN_MAX - 1) / RN_MAX;
  const int box_rows = min(RN_MAX, (n + 15) & ~15);
  // K split: the largest power of two (<= 8) that keeps the grid within the SMs
  // and divides the K blocks
  const int kb_total = H / RK;
  int S = 1;
  while (2 * S <= R_MAX_SPLIT && static_cast<int64_t>(mt) * nbk * 2 * S <= sm_count() && kb_total % (2 * S) == 0)
    S *= 2;
  CUtensorMap tm_x, tm_w;
  cudaError_t e = encode_rows(&tm_x, x, T, H, RM);
  if (e != cudaSuccess) return e;
  e = encode_rows(&tm_w, w_gate, n, H, box_rows);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
  if (e != cudaSuccess) return e;
  RouterArgs args{T, n, box_rows, kb_total / S, logits, ldl, err};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(mt, nbk, S);
  cfg.blockDim = dim3(R_THREADS);
  cfg.dynamicSmemBytes = R_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = S;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_gemm_kernel, tm_x, tm_w, args);
}

}  // namespace nvf
