// Expert-parallel dispatch and return on one rank (the data movement around
// the all-to-all of the pages' DeepEP prepare/finalize: vLLM PR #35737, CI
// failure logs, `all2all_manager.get_handle` and the `deepep_high_throughput`
// MoE prepare/finalize).  Rank `rank` of G owns routed experts
// [rank El, (rank+1) El), El = E / G; a shared expert is replicated and stays
// on its rank.  The exchange itself is the caller's collective; these kernels
// produce and consume its buffers:
//
//   dispatch   permuted row p (routing's stable order: by expert, then
//              assignment) of expert e goes to rank e / El, so the rows for
//              each rank are one slice of the permutation; a rank's own
//              segment ends with its shared rows.  Each row is quantized
//              (NVFP4 with the expert's activation global scale, the block
//              quantizer of the fused routing kernel) into a send row of
//              H/2 code bytes then H/16 scale bytes (padded to 16 bytes), at
//              its send position; src_to_send[a] records where assignment a
//              went, and send_counts[r][j] the rows for local expert j of
//              rank r (column El: the shared expert, own rank only).
//   receive    the arriving rows (sources back to back, each source's rows by
//              local expert) are grouped by local expert, source by source,
//              into the grouped GEMM's TILED_GROUPED A operand;
//              recv_to_grp[i] is received row i's grouped row, grp_to_recv
//              its inverse (the down GEMM can store y rows straight in
//              received order with it).
//   return     y rows, grouped order -> received order, so that the return
//              exchange delivers each sender its rows at their send
//              positions, and the combine reads them through src_to_send.
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

#include <algorithm>
#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int kEpMaxRanks = 1024;

// One warp per permuted row, 4 rows a CTA.
__global__ void __launch_bounds__(128) ep_dispatch_kernel(EpDispatchArgs a) {
  __shared__ int64_t send_off[kEpMaxRanks + 1];
  const int El = a.E / a.G, Et = a.E + a.shared;
  if (threadIdx.x == 0) {
    int64_t acc = 0;
    for (int r = 0; r < a.G; ++r) {
      send_off[r] = acc;
      acc += __ldg(a.offsets + (r + 1) * El) - __ldg(a.offsets + r * El);
      if (r == a.rank && a.shared) acc += __ldg(a.offsets + a.E + 1) - __ldg(a.offsets + a.E);
    }
    send_off[a.G] = acc;
  }
  if (blockIdx.x == 0) {
    for (int c = threadIdx.x; c < a.G * (El + 1); c += blockDim.x) {
      const int r = c / (El + 1), j = c - r * (El + 1);
      int n = 0;
      if (j < El) n = __ldg(a.offsets + r * El + j + 1) - __ldg(a.offsets + r * El + j);
      else if (r == a.rank && a.shared) n = __ldg(a.offsets + a.E + 1) - __ldg(a.offsets + a.E);
      a.send_counts[c] = n;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int64_t R = __ldg(a.offsets + Et);
  if (p >= R) return;
  const int e = upper_group(a.offsets, Et, p);
  int64_t pos;
  if (e < a.E) {
    const int dest = e / El;
    pos = send_off[dest] + (p - __ldg(a.offsets + dest * El));
  } else {
    const int64_t own_routed = __ldg(a.offsets + (a.rank + 1) * El) - __ldg(a.offsets + a.rank * El);
    pos = send_off[a.rank] + own_routed + (p - __ldg(a.offsets + a.E));
  }
  const int t = __ldg(a.perm_token + p);
  if (lane == 0) a.src_to_send[__ldg(a.perm_to_src + p)] = static_cast<int32_t>(pos);
  const float gs = __ldg(a.gs_a1 + e);
  const float six_gs = __fmul_rn(6.0f, gs);
  const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + static_cast<int64_t>(t) * a.H);
  uint8_t* row = a.send + pos * static_cast<int64_t>(a.row_bytes);
  for (int b = lane; b < a.H / 16; b += 32) {
    const uint4 u0 = __ldg(xr + 2 * b), u1 = __ldg(xr + 2 * b + 1);
    const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(wv[i] << 16);               // bf16 -> fp32 is exact
      v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
    }
    uint32_t w0, w1;
    const uint32_t sb = quant_block16(v, gs, six_gs, w0, w1);
    *reinterpret_cast<uint2*>(row + b * 8) = make_uint2(w0, w1);
    row[a.H / 2 + b] = static_cast<uint8_t>(sb);
  }
}

// Above 256 tokens the dispatch runs token by token, so that a token is
// quantized once per distinct global scale among its slots (once, when every
// expert shares one) instead of once per slot.  Pass 1, one thread per
// permuted row: the row's send position into src_to_send, and its expert id
// into the first 4 bytes of its send row, where pass 2 reads it before it
// writes the row.
__global__ void __launch_bounds__(256) ep_dispatch_place_kernel(EpDispatchArgs a) {
  __shared__ int64_t send_off[kEpMaxRanks + 1];
  extern __shared__ int32_t s_offsets[];                 // [Et + 1]: the binary search runs here
  const int El = a.E / a.G, Et = a.E + a.shared;
  for (int e = threadIdx.x; e <= Et; e += blockDim.x) s_offsets[e] = __ldg(a.offsets + e);
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t acc = 0;
    for (int r = 0; r < a.G; ++r) {
      send_off[r] = acc;
      acc += s_offsets[(r + 1) * El] - s_offsets[r * El];
      if (r == a.rank && a.shared) acc += s_offsets[a.E + 1] - s_offsets[a.E];
    }
    send_off[a.G] = acc;
  }
  if (blockIdx.x == 0) {
    for (int c = threadIdx.x; c < a.G * (El + 1); c += blockDim.x) {
      const int r = c / (El + 1), j = c - r * (El + 1);
      int n = 0;
      if (j < El) n = s_offsets[r * El + j + 1] - s_offsets[r * El + j];
      else if (r == a.rank && a.shared) n = s_offsets[a.E + 1] - s_offsets[a.E];
      a.send_counts[c] = n;
    }
  }
  __syncthreads();
  const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t R = s_offsets[Et];
  if (p >= R) return;
  const int e = upper_group(s_offsets, Et, p);
  int64_t pos;
  if (e < a.E) {
    const int dest = e / El;
    pos = send_off[dest] + (p - s_offsets[dest * El]);
  } else {
    const int64_t own_routed = s_offsets[(a.rank + 1) * El] - s_offsets[a.rank * El];
    pos = send_off[a.rank] + own_routed + (p - s_offsets[a.E]);
  }
  a.src_to_send[__ldg(a.perm_to_src + p)] = static_cast<int32_t>(pos);
  *reinterpret_cast<int32_t*>(a.send + pos * static_cast<int64_t>(a.row_bytes)) = e;
}

// Pass 2, one warp per token: lane j first reads slot j's send position and
// expert (every slot's before any lane writes a row), then each lane quantizes
// its 16-element blocks of the token once per distinct global scale and writes
// them to every slot's row.
constexpr int kDispatchTokWarps = 4;
__global__ void __launch_bounds__(kDispatchTokWarps * 32) ep_dispatch_token_kernel(EpDispatchArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kDispatchTokWarps + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int slots = a.k + a.shared;
  int pos_j = 0, e_j = 0;
  if (lane < slots) {
    const int64_t as = lane < a.k ? static_cast<int64_t>(t) * a.k + lane : static_cast<int64_t>(a.T) * a.k + t;
    pos_j = __ldg(a.src_to_send + as);
    e_j = *reinterpret_cast<const int32_t*>(a.send + static_cast<int64_t>(pos_j) * a.row_bytes);
  }
  __syncwarp();
  const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + static_cast<int64_t>(t) * a.H);
  for (int b = lane; b < a.H / 16; b += 32) {
    const uint4 u0 = __ldg(xr + 2 * b), u1 = __ldg(xr + 2 * b + 1);
    const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(wv[i] << 16);               // bf16 -> fp32 is exact
      v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
    }
    float gs_done = -1.0f;                                   // global scales are positive
    uint32_t w0 = 0, w1 = 0, sb = 0;
    for (int j = 0; j < slots; ++j) {
      const int e = __shfl_sync(0xffffffffu, e_j, j), pos = __shfl_sync(0xffffffffu, pos_j, j);
      const float gs = __ldg(a.gs_a1 + e);
      if (gs != gs_done) {
        sb = quant_block16(v, gs, __fmul_rn(6.0f, gs), w0, w1);
        gs_done = gs;
      }
      uint8_t* row = a.send + static_cast<int64_t>(pos) * a.row_bytes;
      *reinterpret_cast<uint2*>(row + b * 8) = make_uint2(w0, w1);
      row[a.H / 2 + b] = static_cast<uint8_t>(sb);
    }
  }
}

// Exclusive prefix sum over the 256 threads of the block (warp shuffles, then
// the warps' totals); *total gets the sum.  Every thread must call it.
__device__ __forceinline__ int32_t block_scan_excl(int32_t v, int32_t* warp_sums, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) warp_sums[lane] = w;
  }
  __syncthreads();
  const int32_t base = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[nw - 1];
  __syncthreads();                                       // warp_sums is reused by the next scan
  return base + x - v;
}

// The receive plan, computed by one whole CTA: local offsets, tile offsets
// and, per (source s, local expert j) cell c = s * J + j, the cell's first
// received row (recv_base) and first grouped row (grp_base).  J = El + 1 count
// columns; Et_l = El + shared local experts.  Thread t handles a contiguous
// chunk of experts, then of cells.  The outputs may be in global or shared
// memory; warp_sums is 32 ints of shared memory.
__device__ void receive_plan(const int32_t* __restrict__ counts, int G, int El, int shared, int32_t* local_offsets,
                             int32_t* local_tile_offsets, int32_t* recv_base, int32_t* grp_base,
                             int32_t* warp_sums) {
  const int J = El + 1, Et_l = El + shared, cells = G * J;
  // experts [j0, j1) of this thread: totals over the sources, then the prefix
  const int per_e = (J + blockDim.x - 1) / blockDim.x;
  const int j0 = min(J, static_cast<int>(threadIdx.x) * per_e), j1 = min(J, j0 + per_e);
  int32_t rows = 0, tiles = 0;
  for (int j = j0; j < min(j1, Et_l); ++j) {
    int32_t n = 0;
    for (int s = 0; s < G; ++s) n += __ldg(counts + s * J + j);
    rows += n;
    tiles += (n + 127) / 128;
  }
  int32_t total_rows, total_tiles;
  int32_t off = block_scan_excl(rows, warp_sums, &total_rows);
  int32_t toff = block_scan_excl(tiles, warp_sums, &total_tiles);
  for (int j = j0; j < j1; ++j) {
    int32_t n = 0;
    if (j < Et_l) {
      local_offsets[j] = off;
      local_tile_offsets[j] = toff;
    }
    int32_t acc = j < Et_l ? off : total_rows;           // the shared column of a layer without one is empty
    for (int s = 0; s < G; ++s) {
      grp_base[s * J + j] = acc;
      const int32_t c = __ldg(counts + s * J + j);
      acc += c;
      n += c;
    }
    if (j < Et_l) {
      off += n;
      toff += (n + 127) / 128;
    }
  }
  if (threadIdx.x == 0) {
    local_offsets[Et_l] = total_rows;
    local_tile_offsets[Et_l] = total_tiles;
  }
  // recv_base: exclusive prefix over the cells in (s, j) order
  const int per = (cells + blockDim.x - 1) / blockDim.x;
  const int c0 = min(cells, static_cast<int>(threadIdx.x) * per), c1 = min(cells, c0 + per);
  int32_t sum = 0;
  for (int c = c0; c < c1; ++c) sum += __ldg(counts + c);
  int32_t total_cells;
  int32_t acc = block_scan_excl(sum, warp_sums, &total_cells);
  for (int c = c0; c < c1; ++c) {
    recv_base[c] = acc;
    acc += __ldg(counts + c);
  }
}

// The plan alone (one CTA of 256 threads), for plans too large for the scatter
// kernel's shared memory.
__global__ void __launch_bounds__(256) ep_receive_plan_kernel(const int32_t* __restrict__ counts, int G, int El,
                                                              int shared, int32_t* local_offsets,
                                                              int32_t* local_tile_offsets, int32_t* recv_base,
                                                              int32_t* grp_base) {
  __shared__ int32_t warp_sums[32];
  receive_plan(counts, G, El, shared, local_offsets, local_tile_offsets, recv_base, grp_base, warp_sums);
}

// One warp per received row, `rows` rows a CTA of 8 warps (8 up to 4096
// received rows, 64 above, so that large receives do not run thousands of
// CTAs).  With PLAN (G * (El + 1) <= kScatterPlanCells) every CTA first
// computes the receive plan itself into shared memory -- a separate
// single-CTA plan kernel ahead of the scatter cost ~5 us of latency -- and
// CTA 0 writes the local offsets out; otherwise the plan comes from
// ep_receive_plan_kernel.  Either way the binary search for a row's (source,
// expert) cell runs over cell starts in shared memory, not along a chain of
// dependent global loads.
constexpr int kScatterWarps = 8, kScatterPlanCells = 4096;
constexpr int kScatterRowsSmall = 8, kScatterRowsLarge = 64, kScatterFusedMaxRows = 4096;
template <bool PLAN>
__global__ void __launch_bounds__(kScatterWarps * 32) ep_receive_scatter_kernel(
    const uint8_t* __restrict__ recv, int64_t n_recv, int row_bytes, int H, int G, int El, int shared,
    int32_t* local_offsets, int32_t* local_tile_offsets, const int32_t* __restrict__ recv_base_g,
    const int32_t* __restrict__ grp_base_g, const int32_t* __restrict__ counts, uint8_t* a1, int32_t* recv_to_grp,
    int32_t* grp_to_recv, int* err, int rows) {
  extern __shared__ int32_t s_plan[];
  __shared__ int32_t warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int J = El + 1, cells = G * J, Et_l = El + shared;
  int32_t* s_rb = s_plan;                                // [cells]
  int32_t* s_gb = s_plan + cells;                        // [cells] (PLAN)
  int32_t* s_lo = s_plan + 2 * cells;                    // [Et_l + 1] (PLAN)
  int32_t* s_lt = s_lo + Et_l + 1;                       // [Et_l + 1] (PLAN)
  const int32_t* gb = grp_base_g;
  const int32_t* lo = local_offsets;
  const int32_t* lt = local_tile_offsets;
  if constexpr (PLAN) {
    receive_plan(counts, G, El, shared, s_lo, s_lt, s_rb, s_gb, warp_sums);
    __syncthreads();
    if (blockIdx.x == 0)
      for (int j = threadIdx.x; j <= Et_l; j += blockDim.x) {
        local_offsets[j] = s_lo[j];
        local_tile_offsets[j] = s_lt[j];
      }
    gb = s_gb;
    lo = s_lo;
    lt = s_lt;
  } else {
    for (int c = threadIdx.x; c < cells; c += blockDim.x) s_rb[c] = __ldg(recv_base_g + c);
    __syncthreads();
  }
  const bool a1_32 = (reinterpret_cast<uintptr_t>(a1) & 31u) == 0;
  for (int m = warp; m < rows; m += kScatterWarps) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * rows + m;
    if (i >= n_recv) break;
    const int c = upper_group(s_rb, cells, i);         // the (source, expert) cell holding row i
    if (i - s_rb[c] >= __ldg(counts + c)) {            // more rows than the counts hold: stay in bounds
      if (lane == 0) report_error(err, DEV_BAD_OFFSETS, static_cast<int>(i));
      continue;
    }
    const int j = c % J;
    const int32_t g = gb[c] + static_cast<int32_t>(i - s_rb[c]);
    const int32_t local = g - lo[j];
    const int64_t tile = lt[j] + (local >> 7);
    const uint32_t r = static_cast<uint32_t>(local & 127);
    if (lane == 0) {
      recv_to_grp[i] = g;
      if (grp_to_recv != nullptr) grp_to_recv[g] = static_cast<int32_t>(i);
    }
    const uint8_t* row = recv + i * static_cast<int64_t>(row_bytes);
    for (int gg = lane; gg < H / 64; gg += 32) {
      const uint4 u0 = *reinterpret_cast<const uint4*>(row + gg * 32);
      const uint4 u1 = *reinterpret_cast<const uint4*>(row + gg * 32 + 16);
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      const uint32_t sf = *reinterpret_cast<const uint32_t*>(row + H / 2 + gg * 4);
      // one 32-byte store for the codes when a1 is 32-byte aligned (chunks are 18432 bytes)
      if (a1_32) store_group64_tg32(a1, H, tile, r, gg, w, sf);
      else store_group64(a1, nullptr, LAYOUT_TILED_GROUPED, H, g, tile, r, gg, w, sf);
    }
  }
}

// out row i = in row idx[i]; 16 bytes a thread.
__global__ void ep_gather_rows_kernel(const uint4* __restrict__ in, int64_t n, int row_units,
                                      const int32_t* __restrict__ idx, uint4* out) {
  const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q >= n * row_units) return;
  const int64_t i = q / row_units;
  const int u = static_cast<int>(q - i * row_units);
  out[q] = in[static_cast<int64_t>(__ldg(idx + i)) * row_units + u];
}

}  // namespace

size_t ep_row_bytes(int H) { return (static_cast<size_t>(H) / 2 + static_cast<size_t>(H) / 16 + 15) & ~size_t(15); }

cudaError_t launch_ep_dispatch(const EpDispatchArgs& a, cudaStream_t s) {
  if (a.G > kEpMaxRanks) return cudaErrorInvalidValue;
  const int64_t R = static_cast<int64_t>(a.T) * a.k + (a.shared ? a.T : 0);
  if (a.T > 256) {
    ep_dispatch_place_kernel<<<static_cast<unsigned>((R + 255) / 256), 256,
                               static_cast<size_t>(a.E + a.shared + 1) * sizeof(int32_t), s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ep_dispatch_token_kernel<<<static_cast<unsigned>((a.T + kDispatchTokWarps - 1) / kDispatchTokWarps),
                               kDispatchTokWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
  }
  const int64_t blocks = R > 0 ? (R + 3) / 4 : 1;     // one CTA at least: it writes send_counts
  ep_dispatch_kernel<<<static_cast<unsigned>(blocks), 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ep_receive(const uint8_t* recv, int64_t n_recv, int row_bytes, const int32_t* counts, int G,
                              int El, int shared, int H, uint8_t* a1, int32_t* local_offsets,
                              int32_t* local_tile_offsets, int32_t* recv_to_grp, int32_t* grp_to_recv,
                              int32_t* scratch, int* err, cudaStream_t s) {
  int32_t* recv_base = scratch;
  int32_t* grp_base = scratch + static_cast<int64_t>(G) * (El + 1);
  const int cells = G * (El + 1), Et_l = El + shared;
  if (cells <= kScatterPlanCells) {
    const int rows = n_recv <= kScatterFusedMaxRows ? kScatterRowsSmall : kScatterRowsLarge;
    const unsigned blocks = static_cast<unsigned>(std::max<int64_t>((n_recv + rows - 1) / rows, 1));
    // plan and scatter in one kernel (at least one CTA: it writes the local offsets)
    const size_t smem = static_cast<size_t>(2 * cells + 2 * (Et_l + 1)) * 4;
    ep_receive_scatter_kernel<true><<<blocks, kScatterWarps * 32, smem, s>>>(
        recv, n_recv, row_bytes, H, G, El, shared, local_offsets, local_tile_offsets, recv_base, grp_base, counts, a1,
        recv_to_grp, grp_to_recv, err, rows);
    return cudaGetLastError();
  }
  ep_receive_plan_kernel<<<1, 256, 0, s>>>(counts, G, El, shared, local_offsets, local_tile_offsets, recv_base,
                                            grp_base);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_recv == 0) return e;
  const size_t smem = static_cast<size_t>(cells) * 4;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(ep_receive_scatter_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int rows = n_recv <= kScatterFusedMaxRows ? kScatterRowsSmall : kScatterRowsLarge;
  const unsigned blocks = static_cast<unsigned>((n_recv + rows - 1) / rows);
  ep_receive_scatter_kernel<false><<<blocks, kScatterWarps * 32, smem, s>>>(
      recv, n_recv, row_bytes, H, G, El, shared, local_offsets, local_tile_offsets, recv_base, grp_base, counts, a1,
      recv_to_grp, grp_to_recv, err, rows);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* in, int64_t n, int64_t row_bytes, const int32_t* idx, void* out,
                               cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int units = static_cast<int>(row_bytes / 16);
  const int64_t total = n * units;
  ep_gather_rows_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, s>>>(
      static_cast<const uint4*>(in), n, units, idx, static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace nvf
