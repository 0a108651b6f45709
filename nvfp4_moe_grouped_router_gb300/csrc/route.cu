// Routing, permutation and combine kernels.
//
//   route_topk      : (up to 256 tokens) one warp per token, four per CTA:
//                     top-k and routing weights only.
//   route_topk_bits : one warp per token: top-k of (logit + bias) by repeated
//                     warp argmax (ties to the lower expert id) and a softmax
//                     over the k selected (renormalised) or over all E.  Each
//                     CTA owns 32 consecutive tokens and writes, for every
//                     expert e, one 32-bit word whose bit i says that token
//                     32*blockIdx + i chose e.
//   route_prefix    : (many tokens only) per expert, exclusive prefix of the
//                     popcounts of its words: how many earlier tokens chose it.
//   route_small_permute / route_permute : every CTA scans the per-expert
//                     counts (expert offsets and the 128-row tile prefix);
//                     each assignment goes to offsets[e] + (number of earlier
//                     tokens that chose e).  A token picks k distinct experts,
//                     so this is exactly the stable order of assignments
//                     a = t*k + j by expert -- computed in parallel,
//                     deterministically.  Up to 256 tokens the bitmaps are
//                     rebuilt from the ids in shared memory.  With activations
//                     given, the token's row is quantized with each slot's
//                     expert global scale into that slot of the gate_up GEMM's
//                     TILED_GROUPED operand: one 16-element block per lane up
//                     to 256 tokens, one warp per token (once per distinct
//                     scale) above.
//   combine         : out[t] = sum_j w[t,j] * y[src_to_perm[t*k+j]] (+ shared row).
//
// Sources: top-k routing over many routed experts plus one shared expert
// (FlashInfer issue #2723, "Model" table: 512 routed + 1 shared, 10 routed per
// token); per-expert problem sizes / offsets feeding the grouped GEMM (vLLM PR
// #29242, commit "Fix get_cutlass_moe_mm_data not compiling" and the review
// of nvfp4_blockwise_moe_kernel.cu naming num_experts, M, N, K); BF16 -> FP4
// per-token activation quantization (FlashInfer issue #2723, "Why 39 vs 49
// tok/s?").
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"
#include "route_topk.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int kMaxE = 1024;          // routed experts
constexpr int kInlineWords = 8;      // up to 256 tokens the permute kernel counts bits itself
constexpr int kPermWarps = 16;       // tokens per permute CTA (up to 256 tokens)
constexpr int kPermTokWarps = 4;     // tokens per permute CTA (more than 256 tokens: up to 8 CTAs a SM)
constexpr int kCombineSlots = 8;     // the combine keeps up to this many slots in flight per thread

template <int NV>
constexpr int topk_threads() { return NV <= 8 ? 1024 : 512; }

template <int NV>
__global__ void __launch_bounds__(topk_threads<NV>()) route_topk_bits_kernel(RouteArgs a) {
  extern __shared__ uint32_t s_words[];  // [E]
  griddep_wait();
  griddep_launch_dependents();
  const int E = a.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_words[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int t0 = blockIdx.x * 32;
  for (int i = warp; i < 32; i += nwarps) {
    const int t = t0 + i;
    if (t >= a.T) break;
    const int e = topk_token<NV>(a, t, lane);
    if (e >= 0) atomicOr(&s_words[e], 1u << i);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) a.words[static_cast<int64_t>(blockIdx.x) * E + e] = s_words[e];
}

// Up to 256 tokens: one token per warp, four warps per CTA, so the top-k of a
// decode batch spreads over several SMs; writes ids and weights only (the
// permutation kernel builds the per-expert bitmaps itself).
template <int NV>
__global__ void __launch_bounds__(128) route_topk_kernel(RouteArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t < a.T) topk_token<NV>(a, t, threadIdx.x & 31);
}

// One warp per expert: exclusive prefix over word columns of the popcounts.
__global__ void __launch_bounds__(256) route_prefix_kernel(RouteArgs a, int W) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= a.E) return;
  int carry = 0;
  for (int w0 = 0; w0 < W; w0 += 32) {
    const int w = w0 + lane;
    const int c = w < W ? __popc(a.words[static_cast<int64_t>(w) * a.E + e]) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (w < W) a.prefix[static_cast<int64_t>(w) * a.E + e] = carry + incl - c;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) a.counts[e] = carry;
}

// Stable position of assignment (t, j) in the expert-sorted order, and the
// expert it goes to (the shared expert's slot j == k sits after all routed rows).
__device__ __forceinline__ int assignment_pos(const RouteArgs& a, const int* offs, int W, int t, int j, int& e) {
  if (j == a.k) {
    e = a.E;
    return a.T * a.k + t;
  }
  e = a.ids[static_cast<int64_t>(t) * a.k + j];
  const int wc = t >> 5;
  const uint32_t below = (1u << (t & 31)) - 1u;
  int rank = __popc(a.words[static_cast<int64_t>(wc) * a.E + e] & below);
  if (W <= kInlineWords) {
    for (int w = 0; w < wc; ++w) rank += __popc(a.words[static_cast<int64_t>(w) * a.E + e]);
  } else {
    rank += a.prefix[static_cast<int64_t>(wc) * a.E + e];
  }
  return offs[e] + rank;
}

// Expert offsets, tile offsets and the tile -> expert map, from shared memory.
__device__ __forceinline__ void write_offsets(const RouteArgs& a, const int* offs, const int* til, int Et) {
  for (int e = threadIdx.x; e <= Et; e += blockDim.x) {
    a.offsets[e] = offs[e];
    a.tile_offs[e] = til[e];
  }
  if (a.tile_group != nullptr) {
    // expert of every 128-row tile: the last e with til[e] <= tile
    for (int j = threadIdx.x; j < til[Et]; j += blockDim.x) {
      int lo = 0, hi = Et;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (til[mid] <= j) lo = mid; else hi = mid;
      }
      a.tile_group[j] = lo;
    }
  }
}

// Up to 256 tokens (W <= kInlineWords bitmap words per expert).  Every CTA
// rebuilds the per-expert token bitmaps in shared memory from the ids (at most
// 8 x E words), scans the counts and ranks each assignment by a popcount.
//   QUANT: grid (ceil(T * wpt / kPermWarps), slots), wpt = ceil(H / 512) warps
//          per (token, slot); lane l of warp q quantizes 16-element block
//          32 q + l of the token's row into the slot.  The row is loaded before
//          the wait on the top-k kernel (x does not depend on it), and every
//          lane does one block, so a decode batch's quantization has little
//          latency to hide.
//   !QUANT: grid (ceil(T / kPermWarps), 1), lane j of a warp places slot j.
template <bool QUANT>
__global__ void __launch_bounds__(kPermWarps * 32) route_small_permute_kernel(RouteArgs a, int W) {
  extern __shared__ uint32_t s_words[];  // [W][E]
  __shared__ int offs[kMaxE + 2];
  __shared__ int til[kMaxE + 2];
  const int E = a.E, Et = a.E + a.shared, k = a.k, T = a.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wpt = QUANT ? (a.H + 511) / 512 : 1;
  const int gw = blockIdx.x * kPermWarps + warp;
  const int t = gw / wpt, q = gw - t * wpt;
  const int blk = q * 32 + lane;  // 16-element block of the row
  const bool has_blk = QUANT && t < T && blk < (a.H >> 4);
  float v[16];
  if (has_blk) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) +
                                                      static_cast<int64_t>(t) * a.H + blk * 16);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 u = __ldg(src + i);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        v[i * 8 + 2 * c] = __uint_as_float(w4[c] << 16);
        v[i * 8 + 2 * c + 1] = __uint_as_float(w4[c] & 0xFFFF0000u);
      }
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  for (int i = threadIdx.x; i < W * E; i += blockDim.x) s_words[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int tt = i / k;
    atomicOr(&s_words[(tt >> 5) * E + __ldg(a.ids + i)], 1u << (tt & 31));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < Et; e += blockDim.x) {
    int c = T;  // the shared expert sees every token
    if (e < E) {
      c = 0;
      for (int w = 0; w < W; ++w) c += __popc(s_words[w * E + e]);
    }
    offs[e] = c;
    til[e] = (c + 127) >> 7;
  }
  __syncthreads();
  if (warp == 0) {
    const int tot = warp_exclusive_scan(offs, Et, lane);
    const int ttot = warp_exclusive_scan(til, Et, lane);
    if (lane == 0) {
      offs[Et] = tot;
      til[Et] = ttot;
    }
  }
  __syncthreads();
  if (blockIdx.x == 0 && blockIdx.y == 0) write_offsets(a, offs, til, Et);
  if (t >= T) return;
  // position of slot j of token t
  auto place = [&](int j, int& e) -> int {
    if (j == k) {
      e = E;
      return T * k + t;
    }
    e = __ldg(a.ids + static_cast<int64_t>(t) * k + j);
    const int wc = t >> 5;
    int rank = __popc(s_words[wc * E + e] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < wc; ++w) rank += __popc(s_words[w * E + e]);
    return offs[e] + rank;
  };
  if constexpr (!QUANT) {
    if (lane < k + a.shared) {
      int e;
      const int pos = place(lane, e);
      const int as = lane < k ? t * k + lane : pos;
      a.perm_to_src[pos] = as;
      a.src_to_perm[as] = pos;
      a.perm_token[pos] = t;
    }
  } else {
    const int j = blockIdx.y;
    int e;
    const int pos = place(j, e);
    if (q == 0 && lane == 0) {
      const int as = j < k ? t * k + j : pos;
      a.perm_to_src[pos] = as;
      a.src_to_perm[as] = pos;
      a.perm_token[pos] = t;
    }
    if (has_blk) {
      const float gs = __ldg(a.gs_a1 + e);
      uint32_t w0, w1;
      const uint32_t sb = quant_block16(v, gs, __fmul_rn(6.0f, gs), w0, w1);
      const int local = pos - offs[e];
      const uint32_t r = static_cast<uint32_t>(local & 127);
      const int bk = blk & 15;
      uint8_t* chunk = a.a1 + (static_cast<size_t>(til[e] + (local >> 7)) * num_k_tiles(a.H) + (blk >> 4)) *
                                  TILE_BYTES;
      *reinterpret_cast<uint2*>(chunk + tiled_code_offset(r, bk * 8)) = make_uint2(w0, w1);
      chunk[TILE_CODE_BYTES + (bk >> 2) * 512 + sf_atom_offset(r, bk & 3)] = static_cast<uint8_t>(sb);
    }
  }
}

// More than 256 tokens (bitmaps from route_topk_bits_kernel, ranks from
// route_prefix_kernel; also the empty batch).  Grid (ceil(T / kPermTokWarps), 1),
// one warp per token t = bx * kPermTokWarps + w; lane j places slot j.  With
// PERM_TOKEN the warp then quantizes the row once per distinct global scale
// among the token's slots and stores it to every slot (the arithmetic is done
// once per token, not once per slot).
enum PermMode : int { PERM_ONLY = 0, PERM_TOKEN = 2 };

// 64 BF16 values (K elements 64 gg ..) of row t, kept packed (32 registers).
__device__ __forceinline__ void load_group64_packed(const RouteArgs& a, int t, int gg, uint4 (&xr)[8]) {
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) +
                                                    static_cast<int64_t>(t) * a.H + gg * 64);
#pragma unroll
  for (int i = 0; i < 8; ++i) xr[i] = __ldg(src + i);
}

// Quantize a packed 64-value group one 16-element block at a time (so that only
// 16 floats are live): 32 code bytes in w, the four scale bytes returned.
__device__ __forceinline__ uint32_t quant_packed64(const uint4 (&xr)[8], float gs, uint32_t (&w)[8]) {
  const float six_gs = __fmul_rn(6.0f, gs);
  uint32_t sf = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float v[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = xr[2 * b + h];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[h * 8 + 2 * q] = __uint_as_float(w4[q] << 16);
        v[h * 8 + 2 * q + 1] = __uint_as_float(w4[q] & 0xFFFF0000u);
      }
    }
    sf |= quant_block16(v, gs, six_gs, w[2 * b], w[2 * b + 1]) << (8 * b);
  }
  return sf;
}

template <int MODE>
__global__ void __launch_bounds__(kPermTokWarps * 32, 8) route_permute_kernel(RouteArgs a, int W) {
  __shared__ int offs[kMaxE + 2];
  __shared__ int til[kMaxE + 2];
  __shared__ int s_pos[MODE == PERM_TOKEN ? kPermTokWarps : 1][33];
  __shared__ int s_exp[MODE == PERM_TOKEN ? kPermTokWarps : 1][33];
  const int E = a.E, Et = a.E + a.shared, k = a.k, T = a.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kPermTokWarps + warp;
  // The token's first 64-value group per lane, fetched before the wait on the
  // routing kernels (x does not depend on them).
  uint4 xr[8];
  if (MODE == PERM_TOKEN && t < T && lane < (a.H >> 6)) load_group64_packed(a, t, lane, xr);
  griddep_wait();
  griddep_launch_dependents();
  // per-expert counts -> expert offsets and tile offsets (every CTA, redundantly)
  for (int e = threadIdx.x; e < Et; e += blockDim.x) {
    int c;
    if (e == E) {
      c = T;  // the shared expert sees every token
    } else if (W <= kInlineWords) {
      c = 0;
      for (int w = 0; w < W; ++w) c += __popc(a.words[static_cast<int64_t>(w) * E + e]);
    } else {
      c = a.counts[e];
    }
    offs[e] = c;
    til[e] = (c + 127) >> 7;
  }
  __syncthreads();
  if (warp == 0) {
    const int tot = warp_exclusive_scan(offs, Et, lane);
    const int ttot = warp_exclusive_scan(til, Et, lane);
    if (lane == 0) {
      offs[Et] = tot;
      til[Et] = ttot;
    }
  }
  __syncthreads();
  if (blockIdx.x == 0 && blockIdx.y == 0) write_offsets(a, offs, til, Et);
  if (t >= T) return;
  {
    const int slots = k + a.shared;
    if (lane < slots) {
      int e;
      const int pos = assignment_pos(a, offs, W, t, lane, e);
      const int as = lane < k ? t * k + lane : pos;
      a.perm_to_src[pos] = as;
      a.src_to_perm[as] = pos;
      a.perm_token[pos] = t;
      if constexpr (MODE == PERM_TOKEN) {
        s_pos[warp][lane] = pos;
        s_exp[warp][lane] = e;
      }
    }
    if constexpr (MODE == PERM_TOKEN) {
      __syncwarp();
      const int gpr = a.H >> 6;
      for (int gg = lane; gg < gpr; gg += 32) {
        if (gg != lane) load_group64_packed(a, t, gg, xr);
        uint32_t w[8];
        uint32_t sf = 0;
        float gs_done = -1.0f;  // global scales are positive
        for (int j = 0; j < slots; ++j) {
          const int ej = s_exp[warp][j], pj = s_pos[warp][j];
          const float gs = __ldg(a.gs_a1 + ej);
          if (gs != gs_done) {
            sf = quant_packed64(xr, gs, w);
            gs_done = gs;
          }
          const int local = pj - offs[ej];
          // one 32-byte store for the codes (the workspace is 256-byte aligned)
          store_group64_tg32(a.a1, a.H, til[ej] + (local >> 7), static_cast<uint32_t>(local & 127), gg, w, sf);
        }
      }
    }
  }
}

// Eight consecutive outputs of one token per thread: one 256-bit (FP32 y) or
// 128-bit (BF16 y) load per slot row (y rows are 32-byte aligned: 256-byte
// workspace, H % 128 == 0).  The sum runs over the slots in order with one FMA
// per slot in FP32, then the shared row.  y and out have the same type: FP32
// for parity runs, BF16 for production (half the bytes of the y round trip).
__device__ __forceinline__ void ld_nc_v8(const float* p, float (&v)[8]) {
  asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}
// Raw y of 8 consecutive outputs: 16 bytes (BF16) or 32 bytes (FP32).
template <bool BF16>
struct Y8 {
  uint32_t w[BF16 ? 4 : 8];
};
template <bool BF16>
__device__ __forceinline__ Y8<BF16> load_y8_raw(const void* y, int64_t off) {
  Y8<BF16> r;
  if constexpr (BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(y) + off));
    r.w[0] = u.x; r.w[1] = u.y; r.w[2] = u.z; r.w[3] = u.w;
  } else {
    float v[8];
    ld_nc_v8(static_cast<const float*>(y) + off, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) r.w[e] = __float_as_uint(v[e]);
  }
  return r;
}
template <bool BF16>
__device__ __forceinline__ float y8_at(const Y8<BF16>& r, int e) {
  if constexpr (BF16) return __uint_as_float((e & 1) ? (r.w[e >> 1] & 0xFFFF0000u) : (r.w[e >> 1] << 16));
  else return __uint_as_float(r.w[e]);
}

// One thread per 8 consecutive outputs of one token (grid covers every output
// once).  The token's slot rows and routing weights come from the routing
// kernel, three launches back, which is complete before this kernel may begin
// (the down GEMM it follows waited on the gate_up GEMM, which waited on the
// routing): they are loaded before the dependency wait, and only the y rows
// after it, all slots at once.
template <bool BF16>
__global__ void __launch_bounds__(256, BF16 ? 4 : 2) combine_kernel(const void* __restrict__ y, int H, const float* __restrict__ w,
                                                     const int32_t* __restrict__ s2p, int T, int k, int shared,
                                                     void* out, const float* __restrict__ sgate, int64_t ldg) {
  const int h8 = H >> 3;
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const bool live = idx < static_cast<int64_t>(T) * h8;
  const int t = live ? static_cast<int>(idx / h8) : 0;
  const int c = live ? static_cast<int>(idx - static_cast<int64_t>(t) * h8) : 0;
  const int kb = min(k, kCombineSlots);
  int64_t row[kCombineSlots];
  float wv[kCombineSlots];
  int64_t srow = 0;
  float sw = 1.0f;
  if (live) {
#pragma unroll
    for (int j = 0; j < kCombineSlots; ++j)
      if (j < kb) {
        const int64_t a = static_cast<int64_t>(t) * k + j;
        wv[j] = __ldg(w + a);
        row[j] = static_cast<int64_t>(__ldg(s2p + a)) * H + c * 8;
      }
    if (shared) {
      srow = static_cast<int64_t>(__ldg(s2p + static_cast<int64_t>(T) * k + t)) * H + c * 8;
      // gated shared expert: sigmoid of the token's gate logit (written by the router, before this launch)
      if (sgate != nullptr) sw = 1.0f / (1.0f + expf(-__ldg(sgate + static_cast<int64_t>(t) * ldg)));
    }
  }
  griddep_wait();
  // A decode batch: the next kernel may launch now (it waits for this grid to
  // finish before it reads anything).  A large batch keeps the SMs to itself:
  // an early launch there parks the next kernel's CTAs on them (prefill +3 us).
  if (T <= 256) griddep_launch_dependents();
  if (!live) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  {
    Y8<BF16> v[kCombineSlots];
#pragma unroll
    for (int j = 0; j < kCombineSlots; ++j)
      if (j < kb) v[j] = load_y8_raw<BF16>(y, row[j]);
#pragma unroll
    for (int j = 0; j < kCombineSlots; ++j)
      if (j < kb) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wv[j], y8_at<BF16>(v[j], e), acc[e]);
      }
  }
  for (int j = kCombineSlots; j < k; ++j) {   // more than kCombineSlots slots: the rest one at a time
    const int64_t a = static_cast<int64_t>(t) * k + j;
    const float wj = __ldg(w + a);
    const Y8<BF16> v = load_y8_raw<BF16>(y, static_cast<int64_t>(__ldg(s2p + a)) * H + c * 8);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(wj, y8_at<BF16>(v, e), acc[e]);
  }
  if (shared) {
    const Y8<BF16> v = load_y8_raw<BF16>(y, srow);
    if (sgate == nullptr) {
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += y8_at<BF16>(v, e);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(sw, y8_at<BF16>(v, e), acc[e]);
    }
  }
  if constexpr (BF16) {
    uint32_t u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      u[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + static_cast<int64_t>(t) * H)[c] =
        make_uint4(u[0], u[1], u[2], u[3]);
  } else {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<int64_t>(t) * H) + 2 * c;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

template <int NV>
cudaError_t launch_route_nv(const RouteArgs& a, cudaStream_t s) {
  const int W = (a.T + 31) / 32;
  // the first kernel follows the caller's choice; the others always depend
  // programmatically on the kernel before them
  bool pdl = a.pdl;
  cudaError_t e = cudaSuccess;
  if (W > 0 && W <= kInlineWords) {
    // up to 256 tokens: spread top-k, bitmaps rebuilt in shared memory
    auto kt = route_topk_kernel<NV>;
    prefer_max_shared(reinterpret_cast<const void*>(kt));
    e = launch_kernel(kt, dim3((a.T + 3) / 4), dim3(128), 0, s, pdl, a);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(W) * a.E * sizeof(uint32_t);
    if (a.x != nullptr) {
      const int wpt = (a.H + 511) / 512;
      auto kp = route_small_permute_kernel<true>;
      prefer_max_shared(reinterpret_cast<const void*>(kp));
      return launch_kernel(kp, dim3((a.T * wpt + kPermWarps - 1) / kPermWarps, a.k + a.shared),
                           dim3(kPermWarps * 32), smem, s, true, a, W);
    }
    auto kp = route_small_permute_kernel<false>;
    prefer_max_shared(reinterpret_cast<const void*>(kp));
    return launch_kernel(kp, dim3((a.T + kPermWarps - 1) / kPermWarps), dim3(kPermWarps * 32), smem, s, true, a, W);
  }
  if (W > 0) {
    auto kt = route_topk_bits_kernel<NV>;
    prefer_max_shared(reinterpret_cast<const void*>(kt));
    e = launch_kernel(kt, dim3(W), dim3(topk_threads<NV>()), a.E * sizeof(uint32_t), s, pdl, a);
    if (e != cudaSuccess) return e;
    pdl = true;
    if (W > kInlineWords) {
      e = launch_kernel(route_prefix_kernel, dim3((a.E + 7) / 8), dim3(256), 0, s, pdl, a, W);
      if (e != cudaSuccess) return e;
    }
  }
  const int blocks = a.T > 0 ? (a.T + kPermTokWarps - 1) / kPermTokWarps : 1;
  if (a.x != nullptr) {
    prefer_max_shared(reinterpret_cast<const void*>(route_permute_kernel<PERM_TOKEN>));
    e = launch_kernel(route_permute_kernel<PERM_TOKEN>, dim3(blocks), dim3(kPermTokWarps * 32), 0, s, pdl, a, W);
  } else {
    prefer_max_shared(reinterpret_cast<const void*>(route_permute_kernel<PERM_ONLY>));
    e = launch_kernel(route_permute_kernel<PERM_ONLY>, dim3(blocks), dim3(kPermTokWarps * 32), 0, s, pdl, a, W);
  }
  return e;
}

}  // namespace

size_t route_scratch_bytes(int32_t T, int32_t E) {
  const size_t W = (static_cast<size_t>(T) + 31) / 32;
  return (2 * W * E + E) * sizeof(int32_t);
}

int route_kernel_launches(int32_t T, int32_t k) {
  (void)k;
  const int W = (T + 31) / 32;
  return W == 0 ? 1 : (W > kInlineWords ? 3 : 2);  // top-k (+ prefix) + permute
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  if (a.E <= 128) return launch_route_nv<4>(a, s);
  if (a.E <= 256) return launch_route_nv<8>(a, s);
  if (a.E <= 512) return launch_route_nv<16>(a, s);
  return launch_route_nv<32>(a, s);
}

cudaError_t launch_combine(const void* y, int32_t H, const float* weights, const int32_t* s2p, int32_t T, int32_t k,
                           int32_t shared, int dtype, void* out, cudaStream_t s, bool pdl, const float* shared_gate,
                           int64_t ldg) {
  if (T == 0) return cudaSuccess;
  const int64_t total = static_cast<int64_t>(T) * (H / 8);
  const int64_t blocks = (total + 255) / 256;   // one output group per thread (T <= 2^24, H <= 2^20: fits the grid)
  auto kern = dtype == X_BF16 ? combine_kernel<true> : combine_kernel<false>;
  prefer_max_shared(reinterpret_cast<const void*>(kern));
  return launch_kernel(kern, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, pdl, y, H, weights, s2p, T, k,
                       shared, out, shared_gate, ldg);
}

}  // namespace nvf
