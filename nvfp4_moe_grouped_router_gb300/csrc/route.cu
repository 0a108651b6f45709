// Routing, permutation and combine kernels.
//
//   route_topk    : one warp per token: top-k of (logit + bias) by repeated warp
//                   argmax (ties to the lower expert id), softmax over the k
//                   selected (renormalised) or over all E, and a per-chunk
//                   expert histogram.
//   route_scan    : one CTA: per-expert totals, exclusive prefix -> expert
//                   offsets, prefix of ceil(m_e / 128) -> tile offsets, and the
//                   first output slot of every (chunk, expert).
//   route_scatter : one warp per chunk walks its assignments a = t*k + j in
//                   order and places each at offsets[e] + rank, which makes the
//                   permutation a stable sort by expert (deterministic, no
//                   global atomics).
//   combine       : out[t] = sum_j w[t,j] * y[src_to_perm[t*k+j]] (+ shared row).
//
// Sources: top-k routing over many routed experts plus one shared expert
// (FlashInfer issue #2723, "Model" table: 512 routed + 1 shared, 10 routed per
// token); per-expert problem sizes / offsets feeding the grouped GEMM (vLLM PR
// #29242, commit "Fix get_cutlass_moe_mm_data not compiling" and the review
// of nvfp4_blockwise_moe_kernel.cu naming num_experts, M, N, K).
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int kMaxE = 1024;            // routed experts
constexpr int kPerLane = kMaxE / 32;   // logits held per lane
constexpr int kTopkWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Top-k of one token by one warp.  NV = logits held per lane (E <= 32 * NV).
// Writes ids / weights of token t and returns, in lanes j < k, the j-th
// selected expert (-1 in the other lanes).
template <int NV>
__device__ __forceinline__ int topk_token(const RouteArgs& a, int t, int lane) {
  const int E = a.E, k = a.k;
  const float* row = a.logits + static_cast<int64_t>(t) * E;
  float v[NV];
  uint32_t taken = 0;  // bit i: value i of this lane is used or absent
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = i * 32 + lane;
    if (e < E) {
      v[i] = a.bias ? __fadd_rn(__ldg(row + e), __ldg(a.bias + e)) : __ldg(row + e);
    } else {
      v[i] = 0.0f;
      taken |= 1u << i;
    }
  }
  float sel_v = 0.0f;
  int sel_e = -1;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      // indices grow with i, so a strict '>' keeps the lower id on ties
      if (!((taken >> i) & 1u) && (bi == 0x7fffffff || v[i] > bv)) {
        bv = v[i];
        bi = i * 32 + lane;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool better = (oi != 0x7fffffff) && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
      if (better) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) { sel_v = bv; sel_e = bi; }
  }
  const float m = __shfl_sync(0xffffffffu, sel_v, 0);
  const float p = (lane < k) ? expf(sel_v - m) : 0.0f;
  float denom;
  if (a.renormalize) {
    denom = warp_sum(p);
  } else {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (i * 32 + lane < E) s += expf(v[i] - m);
    denom = warp_sum(s);
  }
  if (lane < k) {
    a.ids[static_cast<int64_t>(t) * k + lane] = sel_e;
    a.weights[static_cast<int64_t>(t) * k + lane] = p / denom;
  }
  return sel_e;
}

template <int NV>
__global__ void __launch_bounds__(kTopkWarps * 32) route_topk_kernel(RouteArgs a, int tpc) {
  extern __shared__ int hist[];  // [E]
  const int E = a.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * tpc;
  const int t1 = min(a.T, t0 + tpc);
  for (int t = t0 + warp; t < t1; t += kTopkWarps) {
    const int e = topk_token<NV>(a, t, lane);
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) a.chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// Exclusive scan over n <= 2048 values held in smem by one warp; returns the total.
__device__ int warp_exclusive_scan(int* vals, int n, int lane) {
  const int per = (n + 31) / 32;
  const int lo = min(n, lane * per), hi = min(n, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += vals[i];
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  int run = incl - s;
  for (int i = lo; i < hi; ++i) {
    const int c = vals[i];
    vals[i] = run;
    run += c;
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

__global__ void __launch_bounds__(1024) route_scan_kernel(RouteArgs a, int nchunks) {
  __shared__ int cnt[kMaxE + 1];
  __shared__ int til[kMaxE + 1];
  const int E = a.E, Et = a.E + a.shared;
  for (int e = threadIdx.x; e < Et; e += blockDim.x) {
    int total = 0;
    if (e < E) {
      for (int c = 0; c < nchunks; ++c) {
        const int64_t i = static_cast<int64_t>(c) * E + e;
        const int v = a.chunk_counts[i];
        a.chunk_base[i] = total;
        total += v;
      }
    } else {
      total = a.T;  // the shared expert sees every token
    }
    cnt[e] = total;
    til[e] = (total + 127) >> 7;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int tot = warp_exclusive_scan(cnt, Et, threadIdx.x);
    const int ttot = warp_exclusive_scan(til, Et, threadIdx.x);
    if (threadIdx.x == 0) {
      a.offsets[Et] = tot;
      a.tile_offs[Et] = ttot;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < Et; e += blockDim.x) {
    a.offsets[e] = cnt[e];
    a.tile_offs[e] = til[e];
  }
  for (int64_t i = threadIdx.x; i < static_cast<int64_t>(nchunks) * E; i += blockDim.x)
    a.chunk_base[i] += cnt[i % E];
}

__global__ void __launch_bounds__(32) route_scatter_kernel(RouteArgs a, int tpc) {
  extern __shared__ int next[];  // [E]: next free slot of each expert for this chunk
  const int E = a.E, k = a.k, lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) next[e] = a.chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
  __syncwarp();
  const int t0 = blockIdx.x * tpc;
  const int t1 = min(a.T, t0 + tpc);
  const int64_t a0 = static_cast<int64_t>(t0) * k, a1 = static_cast<int64_t>(t1) * k;
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t base = a0; base < a1; base += 32) {
    const int64_t as = base + lane;
    const bool active = as < a1;
    const uint32_t mask = __ballot_sync(0xffffffffu, active);
    int e = 0;
    uint32_t peers = 0;
    if (active) {
      e = a.ids[as];
      peers = __match_any_sync(mask, e);
      const int pos = next[e] + __popc(peers & lt);
      a.perm_to_src[pos] = static_cast<int32_t>(as);
      a.src_to_perm[as] = pos;
      a.perm_token[pos] = static_cast<int32_t>(as / k);
    }
    __syncwarp();
    if (active && lane == 31 - __clz(peers)) next[e] += __popc(peers);
    __syncwarp();
  }
  if (a.shared) {
    const int64_t R = static_cast<int64_t>(a.T) * k;
    for (int t = t0 + lane; t < t1; t += 32) {
      a.perm_to_src[R + t] = static_cast<int32_t>(R + t);
      a.src_to_perm[R + t] = static_cast<int32_t>(R + t);
      a.perm_token[R + t] = t;
    }
  }
}

template <int OUT_BF16>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, int H, const float* __restrict__ w,
                                                     const int32_t* __restrict__ s2p, int T, int k, int shared,
                                                     void* out) {
  const int h4 = H >> 2;
  const int64_t total = static_cast<int64_t>(T) * h4;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / h4);
    const int c = static_cast<int>(idx - static_cast<int64_t>(t) * h4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int64_t a = static_cast<int64_t>(t) * k + j;
      const float wj = __ldg(w + a);
      const float4 v = __ldg(reinterpret_cast<const float4*>(y + static_cast<int64_t>(__ldg(s2p + a)) * H) + c);
      acc.x = fmaf(wj, v.x, acc.x);
      acc.y = fmaf(wj, v.y, acc.y);
      acc.z = fmaf(wj, v.z, acc.z);
      acc.w = fmaf(wj, v.w, acc.w);
    }
    if (shared) {
      const int64_t a = static_cast<int64_t>(T) * k + t;
      const float4 v = __ldg(reinterpret_cast<const float4*>(y + static_cast<int64_t>(__ldg(s2p + a)) * H) + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (OUT_BF16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + static_cast<int64_t>(t) * H)[c] = u;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<int64_t>(t) * H)[c] = acc;
    }
  }
}

}  // namespace

int route_tokens_per_chunk(int32_t T) {
  int tpc = 64;
  while ((T + tpc - 1) / tpc > 2048) tpc *= 2;
  return tpc;
}
int route_num_chunks(int32_t T) {
  const int tpc = route_tokens_per_chunk(T);
  return T == 0 ? 0 : (T + tpc - 1) / tpc;
}

namespace {

constexpr int kSmallAssign = 4096;   // T*k handled by the single-CTA path

// Small batches: top-k, histogram, prefix sums and the stable scatter in one
// CTA of 32 warps: one launch, no scratch memory.
template <int NV>
__global__ void __launch_bounds__(1024) route_small_kernel(RouteArgs a) {
  __shared__ int cnt[kMaxE + 1];
  __shared__ int til[kMaxE + 1];
  __shared__ int s_ids[kSmallAssign];
  const int E = a.E, Et = a.E + a.shared, k = a.k, T = a.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < Et; e += blockDim.x) cnt[e] = (e < E) ? 0 : T;  // shared expert: every token
  __syncthreads();
  for (int t = warp; t < T; t += 32) {
    const int e = topk_token<NV>(a, t, lane);
    if (e >= 0) {
      s_ids[t * k + lane] = e;
      atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  if (warp == 0) {
    for (int e = lane; e < Et; e += 32) til[e] = (cnt[e] + 127) >> 7;
    __syncwarp();
    const int tot = warp_exclusive_scan(cnt, Et, lane);
    const int ttot = warp_exclusive_scan(til, Et, lane);
    __syncwarp();
    for (int e = lane; e < Et; e += 32) {
      a.offsets[e] = cnt[e];
      a.tile_offs[e] = til[e];
    }
    if (lane == 0) {
      a.offsets[Et] = tot;
      a.tile_offs[Et] = ttot;
    }
    // Stable scatter in assignment order; cnt[e] is now expert e's next free slot.
    const int R = T * k;
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = 0; base < R; base += 32) {
      const int as = base + lane;
      const bool active = as < R;
      const uint32_t mask = __ballot_sync(0xffffffffu, active);
      int e = 0;
      uint32_t peers = 0;
      if (active) {
        e = s_ids[as];
        peers = __match_any_sync(mask, e);
        const int pos = cnt[e] + __popc(peers & lt);
        a.perm_to_src[pos] = as;
        a.src_to_perm[as] = pos;
        a.perm_token[pos] = as / k;
      }
      __syncwarp();
      if (active && lane == 31 - __clz(peers)) cnt[e] += __popc(peers);
      __syncwarp();
    }
  }
  if (a.shared) {
    const int R = T * k;
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
      a.perm_to_src[R + t] = R + t;
      a.src_to_perm[R + t] = R + t;
      a.perm_token[R + t] = t;
    }
  }
}

template <int NV>
cudaError_t launch_route_nv(const RouteArgs& a, cudaStream_t s) {
  if (static_cast<int64_t>(a.T) * a.k <= kSmallAssign) {
    route_small_kernel<NV><<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
  }
  const int tpc = route_tokens_per_chunk(a.T);
  const int nch = route_num_chunks(a.T);
  route_topk_kernel<NV><<<nch, kTopkWarps * 32, a.E * sizeof(int), s>>>(a, tpc);
  route_scan_kernel<<<1, 1024, 0, s>>>(a, nch);
  route_scatter_kernel<<<nch, 32, a.E * sizeof(int), s>>>(a, tpc);
  return cudaGetLastError();
}

}  // namespace

int route_kernel_launches(int32_t T, int32_t k) {
  return static_cast<int64_t>(T) * k <= kSmallAssign ? 1 : 3;
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  if (a.E <= 128) return launch_route_nv<4>(a, s);
  if (a.E <= 256) return launch_route_nv<8>(a, s);
  if (a.E <= 512) return launch_route_nv<16>(a, s);
  return launch_route_nv<32>(a, s);
}

cudaError_t launch_combine(const float* y, int32_t H, const float* weights, const int32_t* s2p, int32_t T, int32_t k,
                           int32_t shared, int out_dtype, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t total = static_cast<int64_t>(T) * (H / 4);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  if (out_dtype == X_BF16)
    combine_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, s>>>(y, H, weights, s2p, T, k, shared, out);
  else
    combine_kernel<0><<<static_cast<unsigned>(blocks), 256, 0, s>>>(y, H, weights, s2p, T, k, shared, out);
  return cudaGetLastError();
}

}  // namespace nvf
