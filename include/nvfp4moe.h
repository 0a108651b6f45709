/*
 * nvfp4moe.h - C ABI of the GB300 (sm_103a) NVFP4 mixture-of-experts layer.
 *
 * The layer computes, for tokens x[T,H] (bf16) and router logits[T,E] (fp32):
 *   1. top-k routing            ids, w = topk/softmax(logits + bias)
 *   2. permute by expert        stable sort of assignments a = t*k + j by expert
 *   3. NVFP4 activation quant   A1 = Q(x[token(p)]) with gs_a1[e]
 *   4. grouped FP4 GEMM gate_up C1 = alpha1_e * A1 . W13_e^T
 *   5. SiLU-and-mul + requant   A2 = Q(silu(C1[:, gate]) * C1[:, up]) with gs_a2[e]
 *   6. grouped FP4 GEMM down    y  = alpha2_e * A2 . W2_e^T
 *   7. weighted combine         out[t] = sum_j w[t,j] * y[perm(t,j)] (+ shared expert row)
 * Sources (web pages on NVFP4 MoE kernels):
 *   - vLLM PR #29242 "[Kernel] Add NVFP4 MoE CUTLASS support for SM120": the
 *     NVFP4 experts quant and grouped block-scaled GEMM kernels ("Purpose"),
 *     per-expert alpha pointers with beta = 0 and per-group M, N, K in the error
 *     text (review of nvfp4_blockwise_moe_kernel.cu), per-expert MoE offsets
 *     (commit "Fix get_cutlass_moe_mm_data not compiling").
 *   - FlashInfer issue #2723 "SM120 (RTX Blackwell) NVFP4 MoE: CUTLASS Grouped
 *     Block-Scaled GEMM Produces Invalid Output ...": "Model" table (512 routed
 *     + 1 shared expert, 10 per token, FP4 weights with FP8 block scales), "The
 *     Problem" (grouped GEMM is the MoE expert path), "What We Tried" item 2
 *     (FP32 block amax), "Why 39 vs 49 tok/s?" (BF16 -> FP4 per-token
 *     activation quantization).
 *   - unsloth "Report: NVFP4 kernel selection on SM120/SM121", SASS paragraph
 *     under "Why it matters": E2M1 x E2M1 operands with UE4M3 scales, 4 per
 *     64-element MMA step (one scale per 16 elements).
 *
 * NVFP4 data (everywhere in this ABI):
 *   codes  : two E2M1 codes per byte, K-index 2j in bits 0-3 of byte j.
 *   scales : one unsigned E4M3 byte per 16 consecutive K elements.
 *   gs     : float32 per-tensor (or per-expert) decode scale; value = e2m1 *
 *            e4m3 * gs.  A block scale is E4M3(amax_block / (6 * gs)).
 * Operand layouts (enum nvf_layout):
 *   NVF_LAYOUT_ROWMAJOR      : codes uint8[rows][K/2], scales uint8[rows][K/16].
 *   The tiled layouts cut a matrix into 128-row tiles and 256-element K tiles
 *   (nkt = ceil(K / 256)); piece (tile, kt) holds K elements [256 kt, 256 kt + 256)
 *   of 128 rows as
 *     codes (16384 bytes): 128 per row, code byte b of row r at
 *                          r*128 + (((b/16) ^ (r%8))*16) + b%16;
 *     atoms (2048 bytes):  four 512-byte scale atoms, atom kk for K elements
 *                          [64 kk, 64 kk + 64) of the piece, scale s (0..3) of
 *                          row r at (r%32)*16 + (r/32)*4 + s.
 *   NVF_LAYOUT_TILED_GROUPED : (activations) rows grouped by offsets[G+1]: group
 *                              g's rows form 128-row tiles numbered from
 *                              tile_offsets[g] (exclusive prefix of
 *                              ceil(m_g / 128)); piece (tile, kt) is the
 *                              18432-byte chunk [codes][atoms] at
 *                              (tile * nkt + kt) * 18432.
 *                              Size: nvfp4_tiled_bytes(rows, G, K).
 *   NVF_LAYOUT_TILED         : (weights) rows form G equal groups of R rows (one
 *                              expert's N rows; G = 1 for a single matrix).
 *                              Within a group, tiles 2p and 2p+1 form pair p,
 *                              and K tile kt of pair p is one 36864-byte unit
 *                              [codes 2p][codes 2p+1][atoms 2p][atoms 2p+1] at
 *                              group_base + (2p*nkt + 2kt) * 18432; a group's
 *                              last tile, when ceil(R/128) is odd, has
 *                              18432-byte units [codes][atoms] at group_base +
 *                              (2p*nkt + kt) * 18432.  group_base = g *
 *                              ceil(R/128) * nkt * 18432.  A 256-column GEMM
 *                              tile reads one unit per K tile with one copy.
 *                              Size: nvfp4_tiled_bytes(rows, 0, K) (R a multiple
 *                              of 128 when G > 1).
 *   Bytes of rows past a group's end, and of K past K in the last K tile, are
 *   neither written nor read as data.
 *
 * Conventions.  All pointers marked "device" are device memory owned by the
 * caller; the library never allocates, frees or synchronises on these paths.
 * `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 * asynchronous and reads no device data on the host.  Host-detectable errors
 * return a status before anything is launched; launch failures return
 * NVF_ERR_CUDA; errors detected on the device (a bounded wait that expired)
 * are recorded in a per-device error word read by nvf_device_status().  The
 * library never aborts, traps or prints.  Requires a compute-capability 10.3
 * GPU (GB300); other devices get NVF_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvf_status {
  NVF_OK = 0,
  NVF_ERR_INVALID_ARG = 1,
  NVF_ERR_UNSUPPORTED_DEVICE = 2,
  NVF_ERR_WORKSPACE = 3,
  NVF_ERR_CUDA = 4,
  NVF_ERR_TIMEOUT = 5,
  NVF_ERR_DEVICE_CHECK = 6
} nvf_status;

typedef enum nvf_dtype { NVF_F32 = 0, NVF_BF16 = 1, NVF_F16 = 2 } nvf_dtype;
typedef enum nvf_layout {
  NVF_LAYOUT_ROWMAJOR = 0,
  NVF_LAYOUT_TILED = 1,
  NVF_LAYOUT_TILED_GROUPED = 2
} nvf_layout;

/* Name of a status code (static string). */
const char* nvf_status_string(nvf_status s);
/* Detail of the last error returned on this host thread (names the bad argument
 * and the problem sizes); empty after a successful call. */
const char* nvf_last_error_message(void);
/* Version of the ABI (major * 100 + minor). */
int32_t nvf_abi_version(void);

/* Synchronises `stream`, then reads and clears the current device's error word.
 * *code = 0 if no kernel reported an error, else the first kernel error code
 * (1..4: a pipeline wait expired in the producer / MMA / epilogue / drain;
 * 5: a group larger than the GEMM's layout was promised (it then computes
 * wrong rows but stays in bounds); 6: the wait of nvf_selftest_bounded_wait);
 * *detail = the tile or stage it happened at.  Returns NVF_ERR_TIMEOUT for
 * codes 1-4 and 6, NVF_ERR_DEVICE_CHECK for 5, NVF_ERR_CUDA on a CUDA error,
 * else NVF_OK. */
nvf_status nvf_device_status(void* stream, int32_t* code, int32_t* detail);

/* Failure-detection self-test (no counterpart on the pages): launches one CTA
 * that waits on an mbarrier nothing will ever arrive on, through the same
 * bounded wait the GEMM pipeline uses, with a limit of `limit_ns` (1 us .. 10 s)
 * instead of the kernels' 2 s.  The wait gives up, records code 6 in the
 * device error word and the kernel returns: the context stays usable, and
 * nvf_device_status then reports NVF_ERR_TIMEOUT with code 6.  Asynchronous on
 * `stream`. */
nvf_status nvf_selftest_bounded_wait(uint64_t limit_ns, void* stream);

/* Row order of prepared w13 (host helper).  The fused SiLU-and-mul epilogue
 * needs gate and up rows of the same intermediate index side by side: row r of
 * the prepared [2I, H] matrix is canonical row map[r], where canonical rows
 * [0, I) are gate and [I, 2I) are up.  Blocks of 16 rows alternate: prepared
 * rows [32c, 32c+16) = gate rows [16c, 16c+16), [32c+16, 32c+32) = up rows
 * [16c, 16c+16).  map: host int32[2I].  I must be a positive multiple of 64. */
nvf_status nvf_w13_row_map(int32_t I, int32_t* map);

/* Bytes of a tiled operand buffer for up to `rows` rows, K columns and G
 * groups (G = 0: NVF_LAYOUT_TILED, with groups of a multiple of 128 rows or one
 * group; G >= 1: NVF_LAYOUT_TILED_GROUPED). */
size_t nvfp4_tiled_bytes(int64_t rows, int32_t G, int32_t K);

/* Per-group global scales gs[g] = amax(x[g]) / 2688 (1 when the group is all
 * zero): x device [groups, n] of dtype x_dtype (NVF_F32 | NVF_BF16), gs_out
 * device float[groups].  The FP32 decode-scale reading of the pages' "FP32
 * global scale". */
nvf_status nvfp4_global_scale(const void* x, int32_t x_dtype, int64_t groups, int64_t n, float* gs_out,
                              void* stream);

/* NVFP4 quantization of rows along K (step 3, and weight preparation).
 *   x            device [*, ldx] NVF_F32 or NVF_BF16; output row p reads input
 *                row gather_rows[p] (device int32[rows], nullable = identity).
 *   rows, K      K a positive multiple of 64; ldx >= K, x 16-byte aligned,
 *                ldx * element size a multiple of 16.
 *   group_offsets device int32[G+1] (nullable): rows [offsets[g], offsets[g+1])
 *                use gscale[g]; required for NVF_LAYOUT_TILED_GROUPED together
 *                with tile_offsets (device int32[G+1]).  NVF_LAYOUT_TILED takes
 *                no offsets: rows form G equal groups (rows % G == 0), group g
 *                using gscale[g].  Otherwise gscale[0] is used for every row.
 *   gscale       device float (see above), finite and > 0.
 *   codes        device, 16-byte aligned: uint8[rows, K/2] for ROWMAJOR, the
 *                whole tiled buffer for the tiled layouts.
 *   scales       device uint8[rows, K/16] (4-byte aligned) for ROWMAJOR; unused
 *                (may be NULL) for the tiled layouts.
 * Each 16-element block: amax (FP32) -> sb = E4M3_rn_sat(amax / (6 gs)) ->
 * r = 1 / (dec(sb) * gs) (0 if that product is 0) -> q = E2M1_rn_sat(x * r). */
nvf_status nvfp4_quantize(const void* x, int32_t x_dtype, int64_t rows, int32_t K, int64_t ldx,
                          const int32_t* gather_rows, const int32_t* group_offsets, const int32_t* tile_offsets,
                          int32_t G, const float* gscale, uint8_t* codes, uint8_t* scales, int32_t layout,
                          void* stream);

/* Weight preparation (the offline step before the layer runs; not timed).
 * Turns FP32 or BF16 expert weights into the prepared form nvf_moe_weights
 * points to, for experts e0 .. e0 + n_experts - 1 (so a caller can stream a
 * large expert set through a small source buffer):
 *   w13_src   device [n_experts, 2I, H] of src_dtype: rows [0, I) gate (w1),
 *             rows [I, 2I) up (w3) of each expert.
 *   w2_src    device [n_experts, H, I].
 *   gs_w13, gs_w2  device float[E'] (entries e0 .. e0 + n_experts - 1 written):
 *             amax(expert) / 2688, or 1 for an all-zero expert.
 *   w13       device NVF_LAYOUT_TILED buffer of the [E' * 2I, H] stack
 *             (nvfp4_tiled_bytes(E' * 2I, 0, H) bytes), rows of each expert in
 *             nvf_w13_row_map order; w2 the NVF_LAYOUT_TILED [E' * H, I] stack.
 *   H a positive multiple of 128, I of 64; all buffers 16-byte aligned.
 * Every 16 consecutive input elements of a row become one NVFP4 block as in
 * nvfp4_quantize.  Source: "FP4 weights with FP8 block scales" per expert
 * (FlashInfer issue #2723, "Model" table); one FP32 scale per expert that the
 * grouped GEMM's epilogue folds into a per-expert alpha with beta = 0 (vLLM PR
 * #29242, review of nvfp4_blockwise_moe_kernel.cu: alpha_ptr_array).
 * Asynchronous on `stream`; four kernel launches, no allocation. */
nvf_status nvfp4_prepare_weights(const void* w13_src, const void* w2_src, int32_t src_dtype, int32_t e0,
                                 int32_t n_experts, int32_t H, int32_t I, uint8_t* w13, float* gs_w13, uint8_t* w2,
                                 float* gs_w2, void* stream);

/* Top-k routing and permutation (steps 1-2).
 *   logits       device float[T, E]; bias device float[E] or NULL, added in FP32.
 *   T >= 0, 1 <= E <= 1024, 1 <= k <= min(E, 32); renormalize: softmax over
 *   the k selected logits (1) or over all E (0); shared_expert 0|1 adds expert
 *   id E seen by every token with weight 1 (its rows follow all routed rows).
 * Outputs (device): topk_ids int32[T,k] (descending logit, ties -> lower id),
 *   topk_w float[T,k], expert_offsets int32[E'+1] (E' = E + shared),
 *   tile_offsets int32[E'+1] (prefix of ceil(m_e/128)), perm_to_src int32[R],
 *   src_to_perm int32[R], perm_token int32[R] (R = T*k + shared*T; assignment
 *   a = t*k + j, shared rows a = T*k + t).
 *   ws / ws_bytes: device scratch of at least moe_route_permute_workspace_size(). */
nvf_status moe_route_permute_workspace_size(int32_t T, int32_t E, size_t* bytes);
nvf_status moe_route_permute(const float* logits, const float* bias, int32_t T, int32_t E, int32_t k,
                             int32_t renormalize, int32_t shared_expert, int32_t* topk_ids, float* topk_w,
                             int32_t* expert_offsets, int32_t* tile_offsets, int32_t* perm_to_src,
                             int32_t* src_to_perm, int32_t* perm_token, void* ws, size_t ws_bytes, void* stream);

/* moe_route_permute for callers that cannot allocate device memory.  (The
 * source pages have no counterpart to this entry point: it is a library
 * convenience, not a step of the method.)
 * Some callers have no way to hand this library scratch memory: code that runs
 * inside a framework whose caching allocator owns every device allocation,
 * plug-ins that are given only their input and output buffers, or
 * latency-critical loops where a cudaMalloc (and the device-wide
 * synchronisation it can imply) is not acceptable.  This entry point takes the
 * same inputs and outputs as moe_route_permute but no workspace: its scratch
 * is a fixed 2 MiB array in device memory that the library reserves on every
 * GPU that loads it, for the life of the process.
 *   - Sizes: the scratch a call needs, moe_route_permute_workspace_size(T, E)
 *     = (2 * ceil(T / 32) * E + E) * 4 bytes rounded up to a multiple of 256,
 *     must not exceed NVF_ROUTE_STATIC_SCRATCH_BYTES (2 MiB); larger calls
 *     return NVF_ERR_WORKSPACE before any launch.  That allows T <= 65504
 *     tokens with 128 experts, T <= 32736 with 256, T <= 8160 with 1024.
 *     Device and argument checks come first and return what moe_route_permute
 *     returns (NVF_ERR_UNSUPPORTED_DEVICE, NVF_ERR_INVALID_ARG).
 *   - Allocation: none.  No cudaMalloc/cudaFree or allocating library call is
 *     made.  The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     outside any stream capture.
 *   - Sharing: every call on a device uses the same array, and the array keeps
 *     the last call's contents.  Nothing in it has to start at zero (each call
 *     overwrites every byte it reads).  Calls that can overlap on the GPU (on
 *     different streams without ordering between them) race on the array and
 *     must be serialised by the caller. */
#define NVF_ROUTE_STATIC_SCRATCH_BYTES (2u << 20)
nvf_status moe_route_permute_noalloc(const float* logits, const float* bias, int32_t T, int32_t E, int32_t k,
                                     int32_t renormalize, int32_t shared_expert, int32_t* topk_ids, float* topk_w,
                                     int32_t* expert_offsets, int32_t* tile_offsets, int32_t* perm_to_src,
                                     int32_t* src_to_perm, int32_t* perm_token, void* stream);

/* Grouped block-scaled FP4 GEMM (steps 4 / 6 with a plain epilogue):
 *   D[row, n] = gs_a[g] * gs_b[g] * sum_k A[row, k] B[g*N + n, k]   for offsets[g] <= row < offsets[g+1].
 *   A       device NVF_LAYOUT_TILED_GROUPED buffer of K columns; a_rows bounds
 *           the rows (offsets[G] <= a_rows, buffer of nvfp4_tiled_bytes(a_rows, G, K)).
 *   B       device NVF_LAYOUT_TILED buffer of the [G*N, K] weight matrix (G groups of N rows).
 *   gs_a, gs_b device float[G]; group_offsets, tile_offsets device int32[G+1].
 *   N a positive multiple of 128, K a positive multiple of 64.
 *   D       device [a_rows, ldd] of out_dtype (NVF_F32 | NVF_BF16); only rows of
 *           groups are written.  ldd * element size a multiple of 16. */
nvf_status nvfp4_grouped_gemm(const uint8_t* A, int64_t a_rows, const uint8_t* B, const float* gs_a,
                              const float* gs_b, const int32_t* group_offsets, const int32_t* tile_offsets, int32_t G,
                              int32_t N, int32_t K, int32_t out_dtype, void* D, int64_t ldd, void* stream);

/* Weight-only NVFP4 grouped GEMM (W4A16), the decode alternative the pages
 * compare with the W4A4 path: 16-bit activations times NVFP4 weights
 * dequantized in the kernel to FP16 (every e2m1 * e4m3 product is exact in
 * FP16) on the tensor cores (unsloth report, SASS paragraph under "Why it
 * matters": W4A16 unpacks FP4 and runs FP16 MMA; Marlin W4A16 in FlashInfer
 * issue #2723, "Speed Comparison"):
 *   D[row, n] = gs_b[g] * sum_k A[row, k] * dB_g[n, k]   for offsets[g] <= row < offsets[g+1].
 *   A       device [a_rows, lda] of a_dtype, 16-byte aligned, lda >= K and a
 *           multiple of 8: NVF_F16, or NVF_BF16 (rounded to FP16 by the kernel,
 *           to nearest: exact for magnitudes in [2^-14, 65504]; larger
 *           magnitudes become infinities, smaller ones FP16 subnormals).
 *           Any other a_dtype: NVF_ERR_INVALID_ARG.
 *   B, gs_b, group_offsets, tile_offsets, G, N, K, out_dtype, D, ldd as
 *           nvfp4_grouped_gemm (B the TILED weights of G groups of N rows). */
nvf_status nvfp4_w4a16_grouped_gemm(const void* A, int32_t a_dtype, int64_t a_rows, int64_t lda, const uint8_t* B,
                                    const float* gs_b, const int32_t* group_offsets, const int32_t* tile_offsets,
                                    int32_t G, int32_t N, int32_t K, int32_t out_dtype, void* D, int64_t ldd,
                                    void* stream);

/* Prepared expert weights (all device pointers). */
typedef struct nvf_moe_weights {
  int32_t E;               /* routed experts */
  int32_t H, I;            /* hidden, intermediate: multiples of 128 and 64 */
  int32_t shared;          /* 1: expert E is an always-on shared expert */
  const uint8_t* w13;      /* NVF_LAYOUT_TILED [E'*2I, H] (groups of 2I rows), rows of each expert in nvf_w13_row_map order */
  const float* gs_w13;     /* float[E'] */
  const uint8_t* w2;       /* NVF_LAYOUT_TILED [E'*H, I] (groups of H rows) */
  const float* gs_w2;      /* float[E'] */
} nvf_moe_weights;

/* Byte offsets of the forward pass' intermediates inside its workspace
 * (debug and test access; layouts as documented above). */
typedef struct nvf_moe_ws_layout {
  size_t topk_ids, topk_w, expert_offsets, tile_offsets, perm_to_src, src_to_perm, perm_token;
  size_t route_scratch;
  size_t tile_group;        /* int32[R/128 + E' + 1]: expert of each 128-row tile of A1 / A2 */
  size_t a1;                /* NVF_LAYOUT_TILED_GROUPED, K = H */
  size_t a2;                /* NVF_LAYOUT_TILED_GROUPED, K = I */
  size_t y;                 /* [R, H], row = permuted slot: float when the forward's out is NVF_F32, bf16
                               when it is NVF_BF16 (the region is sized for float) */
  size_t logits;            /* float[T, E + gated]: the router gate's output (nvfp4_moe_forward_gated only) */
  size_t total;
  int64_t R;                /* rows after permutation */
} nvf_moe_ws_layout;

nvf_status nvfp4_moe_workspace_layout(int32_t T, int32_t E, int32_t H, int32_t I, int32_t k, int32_t shared,
                                      nvf_moe_ws_layout* layout);

/* The whole layer (steps 1-7) on one stream.  The down GEMM's output y (one row per
 * permuted slot) is kept in the output's precision: FP32 with an NVF_F32 out (the
 * parity setting), BF16 with an NVF_BF16 out (half the bytes of the y round trip);
 * the combine sums the k slots in slot order in FP32 either way and rounds once.
 *   x        device bf16[T, H]; logits device float[T, E]; bias NULL or float[E].
 *   gs_a1, gs_a2 device float[E']: static activation global scales.
 *   out      device [T, H] of out_dtype (NVF_F32 | NVF_BF16).
 *   h_dump   NULL, or device float[R, I] receiving silu(gate) * up (row = perm slot).
 *   ws       device scratch of nvfp4_moe_workspace_layout().total bytes, 256-byte aligned.
 *   stage_events NULL, or NVF_MOE_STAGE_EVENTS cudaEvent_t handles recorded on `stream`
 *            before routing and after each stage (route+permute, activation quant,
 *            gate_up GEMM, down GEMM, combine), for per-stage timing.  The
 *            permutation kernel quantizes the activations, so the events after
 *            routing and after quantization are recorded together.  With events
 *            the kernels run one after the other; without, each kernel after
 *            the first may start while its predecessor finishes. */
#define NVF_MOE_STAGE_EVENTS 6
nvf_status nvfp4_moe_forward(const nvf_moe_weights* w, const void* x, const float* logits, const float* bias,
                             int32_t T, int32_t k, int32_t renormalize, const float* gs_a1, const float* gs_a2,
                             int32_t out_dtype, void* out, float* h_dump, void* ws, size_t ws_bytes,
                             void* const* stage_events, void* stream);

/* A step of the layer captured once as a CUDA graph, for serving a fixed
 * batch: the host-to-device copies of x and logits from caller-owned
 * page-locked host buffers, nvfp4_moe_forward, and the device-to-host copy of
 * out, replayed by one call.  The copies are kernels that move the bytes
 * through the device's mapping of the page-locked buffers.  It removes the per-step launch work of the
 * separate calls (a decode step's kernels take tens of microseconds; their
 * launches from a host language take as long).
 *   w, gs_a1, gs_a2, bias (NULL or device float[E]): as nvfp4_moe_forward;
 *             the device buffers they point to must outlive the graph.
 *   x_host    page-locked host bf16 [T, H]; logits_host page-locked host
 *             float [T, E]; out_host page-locked host [T, H] of out_dtype
 *             (NVF_F32 or NVF_BF16); all 16-byte aligned.  Each launch reads x_host and
 *             logits_host and writes out_host, asynchronously on the launch
 *             stream: fill the inputs before the launch, read out_host after
 *             the stream has reached the launch.  Pageable host memory:
 *             NVF_ERR_INVALID_ARG.  When logits_host starts right where
 *             x_host ends (T * H * 2 bytes on), both travel in one copy.
 *   graph     receives the handle.  The graph owns its device copies of x,
 *             logits and out and the forward's workspace (freed by
 *             nvf_moe_graph_destroy).
 * Capture does not run the step.  Errors of a launched step are reported
 * through nvf_device_status like those of the separate calls. */
typedef struct nvf_moe_graph nvf_moe_graph;
nvf_status nvf_moe_graph_create(const nvf_moe_weights* w, int32_t T, int32_t k, int32_t renormalize,
                                const float* gs_a1, const float* gs_a2, const float* bias, const void* x_host,
                                const float* logits_host, void* out_host, int32_t out_dtype, nvf_moe_graph** graph);
/* Launch the captured step on `stream` (asynchronous). */
nvf_status nvf_moe_graph_launch(nvf_moe_graph* graph, void* stream);
/* Free the graph and its device buffers (after its launches have completed).
 * NULL is a no-op. */
nvf_status nvf_moe_graph_destroy(nvf_moe_graph* graph);

/* Router gate, the step before routing: logits[t * ldl + j] = sum_h x[t, h] *
 * w_gate[j, h] for j < n, with BF16 inputs multiplied on the tensor cores and
 * summed in FP32.
 *   x       device bf16 [T, H] (row pitch H), 16-byte aligned; H a positive
 *           multiple of 128.
 *   w_gate  device bf16 [n, H]: one row per routed expert, plus, for a gated
 *           shared expert, one more row whose logit gates it.
 *   logits  device float [T, ldl], ldl >= n; columns j < n are written.
 * The pages name the experts the gate scores (FlashInfer issue #2723, "Model"
 * table: 512 routed + 1 shared expert, 10 routed per token) but give no gate
 * formula: this is the plain linear gate without bias.  Asynchronous on
 * `stream`; a bounded wait that expires is reported through nvf_device_status. */
nvf_status nvf_router_gemm(const void* x, const void* w_gate, int32_t T, int32_t H, int32_t n, float* logits,
                           int64_t ldl, void* stream);

/* The layer from the hidden states: the router gate (nvf_router_gemm with
 * w_gate bf16 [E + shared_gate, H], logits into the workspace's `logits`
 * region), then steps 1-7 as nvfp4_moe_forward.  shared_gate = 1 (the layer
 * must have a shared expert) scales the shared expert's output by
 * sigmoid(x . w_gate[E]) instead of 1 (the reading of a gated shared expert;
 * the pages give no formula).  Other arguments as nvfp4_moe_forward. */
nvf_status nvfp4_moe_forward_gated(const nvf_moe_weights* w, const void* w_gate, int32_t shared_gate, const void* x,
                                   const float* bias, int32_t T, int32_t k, int32_t renormalize, const float* gs_a1,
                                   const float* gs_a2, int32_t out_dtype, void* out, void* ws, size_t ws_bytes,
                                   void* stream);

/* ---------------------------------------------------------------------------
 * Expert parallelism (EP): the data movement around the token all-to-all the
 * pages run with DeepEP (vLLM PR #35737, CI failure logs: all2all_manager
 * get_handle, the deepep_high_throughput MoE prepare/finalize).  The pages show
 * the call sites, not the layout; the reading implemented here:
 *   G ranks, each routing its own T tokens over all E routed experts (E a
 *   multiple of G); rank r owns routed experts [r E/G, (r+1) E/G); a shared
 *   expert is replicated and every rank computes its own tokens' shared rows.
 *   A rank sends each (token, slot) row, NVFP4-quantized with the destination
 *   expert's activation global scale, to the expert's owner; the receiver
 *   groups what arrives by local expert (source by source) and runs its local
 *   experts; each y row returns to its sender at the position it was sent
 *   from, and the sender combines as on one GPU.
 * One EP layer on rank r:
 *   moe_route_permute (global expert ids) -> nvf_ep_dispatch ->
 *   exchange send_counts, then the rows (the caller's all-to-all) ->
 *   nvf_ep_receive -> nvfp4_moe_experts (local weights) -> nvf_ep_return ->
 *   exchange back -> nvf_moe_combine (with src_to_send).
 * Every call is asynchronous on `stream` and allocates nothing.
 * ------------------------------------------------------------------------- */

/* Bytes of one exchanged A1 row: H/2 code bytes (element 2j in the low nibble
 * of byte j), then H/16 E4M3 scale bytes, padded to a multiple of 16. */
size_t nvf_ep_row_bytes(int32_t H);

/* Dispatch on rank `rank` of G.  Inputs are moe_route_permute's outputs for
 * the rank's T tokens (expert_offsets [E + shared + 1], perm_token and
 * perm_to_src [R], R = T*k + shared*T), x (device bf16 [T, H], 16-byte aligned,
 * H a positive multiple of 128) and gs_a1 (device float [E + shared], global
 * expert ids).  Outputs (device, caller-owned):
 *   send_rows   [R, nvf_ep_row_bytes(H)] bytes, 16-byte aligned: the rows for
 *               rank 0, then rank 1, ...; rank r's rows are its experts' rows
 *               in routing order; the rank's own segment ends with its shared
 *               rows (by token);
 *   send_counts int32 [G, E/G + 1]: rows for each local expert of each
 *               destination; column E/G is the shared expert (own rank only);
 *   src_to_send int32 [R]: send position of assignment a (a = t*k + j, shared
 *               rows T*k + t), the row index the combine reads.
 * Errors: NVF_ERR_INVALID_ARG (G < 1, G > 1024, E % G != 0, rank out of
 * range, NULL or misaligned buffers), NVF_ERR_UNSUPPORTED_DEVICE, NVF_ERR_CUDA. */
nvf_status nvf_ep_dispatch(const void* x, int32_t T, int32_t H, int32_t E, int32_t k, int32_t shared, int32_t G,
                           int32_t rank, const int32_t* expert_offsets, const int32_t* perm_token,
                           const int32_t* perm_to_src, const float* gs_a1, void* send_rows, int32_t* send_counts,
                           int32_t* src_to_send, void* stream);

/* int32 words of scratch nvf_ep_receive needs: 2 * G * (El + 1). */
size_t nvf_ep_receive_scratch_words(int32_t G, int32_t El);

/* Receive on a rank with El local routed experts (+ the shared one when
 * shared = 1).  recv_rows: device [n_recv, nvf_ep_row_bytes(H)], the rows from
 * source 0, then source 1, ... (each source's send segment for this rank);
 * recv_counts: device int32 [G, El + 1], row s = source s's send_counts row for
 * this rank; n_recv = the sum of recv_counts (a larger n_recv is reported
 * through nvf_device_status, code 5, and the extra rows are ignored).
 * Outputs (device, caller-owned): a1, the local experts' A operand in
 * NVF_LAYOUT_TILED_GROUPED (nvfp4_tiled_bytes(n_recv, El + shared, H) bytes,
 * 16-byte aligned); local_offsets and local_tile_offsets int32
 * [El + shared + 1] (local expert j's rows: source 0's, then source 1's, ...);
 * recv_to_grp int32 [n_recv], received row i's grouped row; grp_to_recv
 * (nullable) int32 [n_recv], its inverse.  scratch: device int32
 * [nvf_ep_receive_scratch_words(G, El)].  Limits: 1 <= G <= 1024, El >= 1,
 * G * (El + 1) <= 57344 (the per-cell table is kept in shared memory);
 * otherwise NVF_ERR_INVALID_ARG. */
nvf_status nvf_ep_receive(const void* recv_rows, int64_t n_recv, const int32_t* recv_counts, int32_t G, int32_t El,
                          int32_t shared, int32_t H, uint8_t* a1, int32_t* local_offsets,
                          int32_t* local_tile_offsets, int32_t* recv_to_grp, int32_t* grp_to_recv, int32_t* scratch,
                          void* stream);

/* The expert computation of steps 4-6 on grouped rows (the layer's GEMMs
 * without routing): y[p] = alpha2_e * A2_p . W2_e^T with A2 the NVFP4 of
 * silu(gate) * up of alpha1_e * A1_p . W13_e^T, for the rows p of local
 * expert e.  w: the (local) experts' prepared weights; a1: device
 * NVF_LAYOUT_TILED_GROUPED [a_rows, H] rows grouped by offsets / tile_offsets
 * (int32 [E + shared + 1], device); gs_a1, gs_a2: device float [E + shared];
 * y: device [a_rows, H] of out_dtype (NVF_F32 | NVF_BF16), 16-byte aligned;
 * y_rows: nullable device int32 [a_rows], a permutation of [0, a_rows): grouped
 * row p is stored as y row y_rows[p] (with nvf_ep_receive's grp_to_recv, y
 * comes out in received order and nvf_ep_return is not needed); NULL stores
 * row p as row p.  ws: device scratch of nvfp4_tiled_bytes(a_rows, E + shared,
 * I) bytes (the A2 operand), 256-byte aligned. */
nvf_status nvfp4_moe_experts(const nvf_moe_weights* w, const uint8_t* a1, int64_t a_rows, const int32_t* offsets,
                             const int32_t* tile_offsets, const float* gs_a1, const float* gs_a2, int32_t out_dtype,
                             void* y, const int32_t* y_rows, void* ws, size_t ws_bytes, void* stream);

/* Return: y_ret[i] = y[recv_to_grp[i]] (rows of H elements of dtype NVF_F32 or
 * NVF_BF16, device, 16-byte aligned), the received order, which the return
 * exchange sends back segment by segment. */
nvf_status nvf_ep_return(const void* y, int64_t n_recv, int32_t H, int32_t dtype, const int32_t* recv_to_grp,
                         void* y_ret, void* stream);

/* Step 7 on its own: out[t] = sum_j w[t, j] y[src_to_row[t*k + j]] (+ the
 * shared row y[src_to_row[T*k + t]]), FP32 sums in slot order.  y: device
 * [rows, H] of dtype (NVF_F32 | NVF_BF16), 32-byte aligned rows (H a multiple
 * of 128); topk_w: device float [T, k]; src_to_row: device int32
 * [T*k + shared*T]; out: device [T, H] of dtype. */
nvf_status nvf_moe_combine(const void* y, int32_t H, int32_t dtype, const float* topk_w, const int32_t* src_to_row,
                           int32_t T, int32_t k, int32_t shared, void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H */
