// Per-token top-k routing by one warp and a one-warp exclusive scan, used by
// the routing kernels.  Top-k of (logit + bias) by repeated warp argmax, ties to the lower
// expert id, then a softmax over the k selected (renormalised) or over all E
// (FlashInfer issue #2723, "Model" table: top-k over routed experts).
#pragma once
#include "internal.h"

namespace nvf {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order-preserving 32-bit key of an FP32 logit: a > b (as floats) exactly
// when key(a) > key(b), and +0 and -0 share a key (they compare equal).  Keys
// 0 (absent or already taken) and 1 (NaN) sit below every number.
__device__ __forceinline__ uint32_t logit_key(float f) {
  if (f != f) return 1u;
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// What the top-k reads and writes, small enough to stay in registers (a copy
// of the whole argument block would live in local memory).
struct TopkIO {
  const float* logits;   // [T, ldl]
  int64_t ldl;
  const float* bias;     // nullable [E]
  int32_t E, k, renormalize;
  int32_t* ids;          // nullable [T, k]: ids and weights are written when set
  float* weights;        // [T, k]
};
__device__ __forceinline__ TopkIO topk_io(const RouteArgs& a, bool write) {
  return TopkIO{a.logits, a.ldl, a.bias, a.E, a.k, a.renormalize, write ? a.ids : nullptr, a.weights};
}

// Top-k of NT tokens by one warp (the routing kernels use NT = 1).  Each round takes the warp maximum of the remaining keys with one
// redux.sync and the lowest expert id holding it with one ballot per value a
// lane holds (id = 32 i + lane, so the first i with a hit, then the lowest
// lane): the largest logit, ties to the lower id.  NV = logits held per lane
// (E <= 32 * NV).  Token tt[q] < 0 is absent.  Then a softmax over the k
// selected (renormalised) or over all E.  Writes ids / weights of each token
// (unless a.ids is null) and returns in sel[q], lanes j < k, the j-th selected
// expert (-1 elsewhere).
template <int NV, int NT>
__device__ __forceinline__ void topk_tokens(const TopkIO a, const int (&tt)[NT], int lane, int (&sel)[NT]) {
  const int E = a.E, k = a.k;
  float v[NT][NV];
  uint32_t key[NT][NV];
  uint32_t taken[NT];  // bit i: value i of this lane is selected (a mask, not a store into key[])
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    taken[q] = 0u;
    const float* row = a.logits + static_cast<int64_t>(tt[q] < 0 ? 0 : tt[q]) * a.ldl;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = i * 32 + lane;
      if (tt[q] >= 0 && e < E) {
        v[q][i] = a.bias ? __fadd_rn(__ldg(row + e), __ldg(a.bias + e)) : __ldg(row + e);
        key[q][i] = logit_key(v[q][i]);
      } else {
        v[q][i] = 0.0f;
        key[q][i] = 0u;
      }
    }
    sel[q] = -1;
  }
  for (int j = 0; j < k; ++j) {
    uint32_t m[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      m[q] = 0u;
#pragma unroll
      for (int i = 0; i < NV; ++i) m[q] = max(m[q], ((taken[q] >> i) & 1u) ? 0u : key[q][i]);
    }
#pragma unroll
    for (int q = 0; q < NT; ++q) m[q] = __reduce_max_sync(0xffffffffu, m[q]);
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      int id = -1;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const uint32_t b = __ballot_sync(0xffffffffu, key[q][i] == m[q] && !((taken[q] >> i) & 1u));
        if (id < 0 && b != 0u) id = i * 32 + __ffs(b) - 1;
      }
      if ((id & 31) == lane) taken[q] |= 1u << (id >> 5);
      if (lane == j) sel[q] = id;
    }
  }
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    // the selected logits: lane j < k fetches its expert's value from the lane holding it
    float sv = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float o = __shfl_sync(0xffffffffu, v[q][i], sel[q] & 31);
      if (sel[q] >= 0 && (sel[q] >> 5) == i) sv = o;
    }
    const float m = __shfl_sync(0xffffffffu, sv, 0);
    const float pr = (lane < k) ? expf(sv - m) : 0.0f;
    float denom;
    if (a.renormalize) {
      denom = warp_sum(pr);
    } else {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (i * 32 + lane < E) s += expf(v[q][i] - m);
      denom = warp_sum(s);
    }
    if (tt[q] >= 0 && lane < k && a.ids != nullptr) {
      a.ids[static_cast<int64_t>(tt[q]) * k + lane] = sel[q];
      a.weights[static_cast<int64_t>(tt[q]) * k + lane] = pr / denom;
    }
  }
}

// One token per warp.
template <int NV>
__device__ __forceinline__ int topk_token(const RouteArgs& a, int t, int lane) {
  const int tt[1] = {t};
  int sel[1];
  topk_tokens<NV, 1>(topk_io(a, true), tt, lane, sel);
  return sel[0];
}

// Exclusive scan over n <= 2048 values held in smem by one warp; returns the total.
__device__ __forceinline__ int warp_exclusive_scan(int* vals, int n, int lane) {
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

}  // namespace nvf
