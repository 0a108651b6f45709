// Host-side launchers shared between the kernel translation units and the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace nvf {

enum XDtype : int { X_F32 = 0, X_BF16 = 1 };

// Launch `kernel` on stream `s`.  With `pdl` the launch is a programmatic
// dependent launch: it may begin while the previous kernel of the stream is
// still running, and the kernel executes griddep_wait() before it touches
// anything that kernel (or an earlier one) wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct QuantArgs {
  const void* x;            // [src_rows, ldx] f32 or bf16
  int x_dtype;
  int64_t rows;             // output rows
  int32_t K;                // multiple of 64
  int64_t ldx;              // elements
  const int32_t* gather;    // nullable [rows]: output row p reads x row gather[p]
  const int32_t* offsets;   // nullable [G+1]: row groups (per-group global scale, grouped layout)
  const int32_t* tile_offs; // [G+1], TILED_GROUPED only
  int32_t G;
  const float* gs;          // [G] when offsets given, else [1]
  uint8_t* codes;           // ROWMAJOR: [rows, K/2]; tiled layouts: the chunk buffer
  uint8_t* scales;          // ROWMAJOR: [rows, K/16]; unused otherwise
  int layout;               // OperandLayout
  // Weight preparation (no device tables): without offsets, row p uses
  // gs[p / rows_per_group] when rows_per_group > 0; with w13_I > 0 (and no
  // gather) output row p reads input row w13_source_row(p, w13_I).
  int32_t rows_per_group = 0;
  int32_t w13_I = 0;
};
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t s);
cudaError_t launch_global_scale(const void* x, int x_dtype, int64_t groups, int64_t n_per_group, float* gs_out,
                                cudaStream_t s);

struct RouteArgs {
  const float* logits;      // [T, ldl]: row t's E logits first
  int64_t ldl;              // logits row stride (elements), >= E
  const float* bias;        // nullable [E]
  int32_t T, E, k, renormalize, shared;
  int32_t* ids;             // [T, k]
  float* weights;           // [T, k]
  int32_t* offsets;         // [E'+1]
  int32_t* tile_offs;       // [E'+1]
  int32_t* perm_to_src;     // [R']
  int32_t* src_to_perm;     // [R']
  int32_t* perm_token;      // [R']
  uint32_t* words;          // scratch [ceil(T/32), E]: bit i of words[w][e]: token 32w+i chose e
  int32_t* prefix;          // scratch [ceil(T/32), E]: earlier tokens that chose e (many tokens only)
  int32_t* counts;          // scratch [E]
  // Optional activation quantization done by the permute kernel (A1 of the forward pass):
  const void* x;            // nullable bf16 [T, H]
  int32_t H;
  const float* gs_a1;       // [E']
  uint8_t* a1;              // TILED_GROUPED operand, K = H
  int32_t* tile_group;      // nullable [tiles]: expert of each 128-row tile (written with the offsets)
  bool pdl;                 // first kernel as a programmatic dependent launch
};
size_t route_scratch_bytes(int32_t T, int32_t E);
int route_kernel_launches(int32_t T, int32_t k);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);

// y [R, H] and out [T, H] of the same dtype (X_F32 or X_BF16).  shared_gate:
// nullable; with a shared expert, its row is scaled by sigmoid(shared_gate[t * ldg])
// instead of 1.
cudaError_t launch_combine(const void* y, int32_t H, const float* weights, const int32_t* src_to_perm, int32_t T,
                           int32_t k, int32_t shared, int dtype, void* out, cudaStream_t s, bool pdl,
                           const float* shared_gate = nullptr, int64_t ldg = 0);

// Weight-only NVFP4 grouped GEMM: FP16 (or BF16, a_bf16) A [a_rows, lda] rows grouped by offsets, B the
// TILED weights of G groups of N rows, D [rows, ldd] FP32 (out_bf16 = 0) or BF16.
cudaError_t launch_w4a16(const void* A, int a_bf16, int64_t a_rows, int64_t lda, const uint8_t* B, const float* gs_b,
                         const int32_t* offsets, const int32_t* tile_offs, int32_t G, int32_t N, int32_t K,
                         int out_bf16, void* D, int64_t ldd, int* err, cudaStream_t s);

// Router gate: logits[t * ldl + j] = sum_h x[t, h] * w_gate[j, h] (BF16 in, FP32 out),
// j < n; H a multiple of 128.
cudaError_t launch_router_gemm(const void* x, const void* w_gate, int32_t T, int32_t H, int32_t n, float* logits,
                               int64_t ldl, int* err, cudaStream_t s);

enum GemmEpilogue : int { EPI_STORE_F32 = 0, EPI_STORE_BF16 = 1, EPI_SWIGLU_QUANT = 2 };

struct GemmArgs {
  const uint8_t* a;         // TILED_GROUPED operand (K columns)
  int64_t a_rows;           // rows the groups may hold (grid sizing)
  const uint8_t* b;         // TILED operand of the [G*N, K] weights
  const float* gs_a;        // [G]
  const float* gs_b;        // [G]
  const int32_t* offsets;   // [G+1]
  const int32_t* tile_offs; // [G+1]
  const int32_t* tile_group; // nullable [tile_offs[G]]: group of each 128-row tile of A
  int32_t G, N, K;
  int epilogue;
  void* d;                  // STORE: [rows, ldd]
  int64_t ldd;
  const int32_t* d_rows;    // STORE: nullable [a_rows]: output row of each grouped row (identity if null)
  uint8_t* q_codes;         // SWIGLU: TILED_GROUPED operand with K2 = N/2 (the next GEMM's A)
  const float* gs_q;        // SWIGLU: [G]
  float* h_dump;            // SWIGLU: nullable [a_rows, N/2]
  int* err;                 // device error word
  bool d_align32;           // STORE: d and ldd * element size are multiples of 32 bytes (256-bit stores)
  bool small_a;             // every group has at most 32 rows (a deeper pipeline fits)
  int max_ctas;             // 0: one CTA per SM
  bool pdl;                 // programmatic dependent launch
  // offsets / tile_offs were complete before the preceding kernel began, so the
  // producer may start pulling weights into L2 before its dependency wait
  bool early_weights;
};
cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s, const char** why);

int* device_error_word();   // per current device, nullptr on failure
// Expert-parallel dispatch / receive / return (ep.cu).
struct EpDispatchArgs {
  const void* x;                  // bf16 [T, H]
  int32_t T, H, E, k, shared, G, rank;
  const int32_t* offsets;         // routing's expert offsets [E + shared + 1]
  const int32_t* perm_token;      // [R]
  const int32_t* perm_to_src;     // [R]
  const float* gs_a1;             // [E + shared], global expert ids
  uint8_t* send;                  // [R, row_bytes]
  int32_t row_bytes;
  int32_t* send_counts;           // [G, E/G + 1]
  int32_t* src_to_send;           // [R]
};
size_t ep_row_bytes(int H);
cudaError_t launch_ep_dispatch(const EpDispatchArgs& a, cudaStream_t s);
cudaError_t launch_ep_receive(const uint8_t* recv, int64_t n_recv, int row_bytes, const int32_t* counts, int G,
                              int El, int shared, int H, uint8_t* a1, int32_t* local_offsets,
                              int32_t* local_tile_offsets, int32_t* recv_to_grp, int32_t* grp_to_recv,
                              int32_t* scratch, int* err, cudaStream_t s);
cudaError_t launch_gather_rows(const void* in, int64_t n, int64_t row_bytes, const int32_t* idx, void* out,
                               cudaStream_t s);

int sm_count();
// Ask for the largest shared-memory carveout once per (device, kernel), so that
// consecutive kernels of the layer do not reconfigure L1 / shared memory.
void prefer_max_shared(const void* func);

}  // namespace nvf
