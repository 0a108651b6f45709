// C ABI of the NVFP4 MoE layer: argument validation, workspace carving and the
// launch sequence.  See include/nvfp4moe.h for the contract of every entry point.
#include "../../include/nvfp4moe.h"
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>

namespace nvf {

__device__ int g_device_error[2];

namespace {

constexpr int kMaxDevices = 64;
thread_local char g_msg[512];

nvf_status fail(nvf_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

nvf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(NVF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 ok, -1 unsupported
  int sms = 0;
  int* err = nullptr;
  int major = 0, minor = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Validates the current device once (CC 10.3) and caches its SM count and the
// address of its error word.
nvf_status current_device(DeviceInfo** out) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (d < 0 || d >= kMaxDevices) return fail(NVF_ERR_UNSUPPORTED_DEVICE, "device ordinal %d out of range", d);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[d];
  if (di.checked == 0) {
    cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, d);
    cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, d);
    if (di.major != 10 || di.minor != 3) {
      di.checked = -1;
    } else {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_device_error);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
      di.err = static_cast<int*>(p);
      di.checked = 1;
    }
  }
  if (di.checked < 0)
    return fail(NVF_ERR_UNSUPPORTED_DEVICE, "device %d has compute capability %d.%d; this library is built for 10.3 (GB300)",
                d, di.major, di.minor);
  *out = &di;
  return NVF_OK;
}

thread_local int g_cur_sms = 148;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

int sm_count() { return g_cur_sms; }

void prefer_max_shared(const void* func) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  if (done.insert({dev, func}).second)
    cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}
void set_last_error(const char* msg) {
  std::snprintf(g_msg, sizeof(g_msg), "%s", msg);
}
int* device_error_word() {
  DeviceInfo* di = nullptr;
  return current_device(&di) == NVF_OK ? di->err : nullptr;
}

}  // namespace nvf

using namespace nvf;

#define NVF_BEGIN()                                 \
  g_msg[0] = 0;                                     \
  DeviceInfo* dev_ = nullptr;                       \
  {                                                 \
    nvf_status st_ = current_device(&dev_);         \
    if (st_ != NVF_OK) return st_;                  \
    g_cur_sms = dev_->sms;                          \
  }
#define NVF_REQUIRE(cond, ...) \
  do {                         \
    if (!(cond)) return fail(NVF_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define NVF_CUDA(call, what)                       \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

namespace {
RouteArgs make_route_args(const float* logits, const float* bias, int32_t T, int32_t E, int32_t k, int32_t renormalize,
                          int32_t shared, int32_t* ids, float* w, int32_t* offsets, int32_t* tile_offsets,
                          int32_t* perm_to_src, int32_t* src_to_perm, int32_t* perm_token, void* scratch) {
  RouteArgs a{};
  a.logits = logits; a.ldl = E; a.bias = bias; a.T = T; a.E = E; a.k = k; a.renormalize = renormalize ? 1 : 0;
  a.shared = shared; a.ids = ids; a.weights = w; a.offsets = offsets; a.tile_offs = tile_offsets;
  a.perm_to_src = perm_to_src; a.src_to_perm = src_to_perm; a.perm_token = perm_token;
  const size_t W = (static_cast<size_t>(T) + 31) / 32;
  a.words = static_cast<uint32_t*>(scratch);
  a.prefix = reinterpret_cast<int32_t*>(a.words + W * E);
  a.counts = a.prefix + W * E;
  return a;
}
}  // namespace

extern "C" {

const char* nvf_status_string(nvf_status s) {
  switch (s) {
    case NVF_OK: return "NVF_OK";
    case NVF_ERR_INVALID_ARG: return "NVF_ERR_INVALID_ARG";
    case NVF_ERR_UNSUPPORTED_DEVICE: return "NVF_ERR_UNSUPPORTED_DEVICE";
    case NVF_ERR_WORKSPACE: return "NVF_ERR_WORKSPACE";
    case NVF_ERR_CUDA: return "NVF_ERR_CUDA";
    case NVF_ERR_TIMEOUT: return "NVF_ERR_TIMEOUT";
    case NVF_ERR_DEVICE_CHECK: return "NVF_ERR_DEVICE_CHECK";
  }
  return "NVF_ERR_UNKNOWN";
}

const char* nvf_last_error_message(void) { return g_msg; }

int32_t nvf_abi_version(void) { return 100; }

nvf_status nvf_device_status(void* stream, int32_t* code, int32_t* detail) {
  NVF_BEGIN();
  NVF_REQUIRE(code != nullptr, "code must not be NULL");
  NVF_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  int h[2] = {0, 0};
  NVF_CUDA(cudaMemcpy(h, dev_->err, sizeof(h), cudaMemcpyDeviceToHost), "read error word");
  NVF_CUDA(cudaMemset(dev_->err, 0, sizeof(h)), "clear error word");
  *code = h[0];
  if (detail) *detail = h[1];
  if (h[0] == 0) return NVF_OK;
  if (h[0] == DEV_BAD_OFFSETS)
    return fail(NVF_ERR_DEVICE_CHECK, "a group held more rows than the GEMM layout was told (at tile %d)", h[1]);
  return fail(NVF_ERR_TIMEOUT, "a kernel pipeline wait expired (code %d, at %d)", h[0], h[1]);
}

}  // extern "C"

namespace nvf {
// Host <-> device copy done by the SMs over the device's mapping of page-locked
// host memory (16-byte pieces, grid-stride; dst and src 16-byte aligned).  In
// the captured decode step (147 KB in, 131 KB out) the two copy kernels add
// ~6 us to the layer; two copy-engine copies added ~17 us.
__global__ void __launch_bounds__(256) graph_copy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                                         size_t n) {
  // launched behind the layer's last kernel, it reads that kernel's output only
  // after it has finished; the layer's first kernel may launch meanwhile
  griddep_wait();
  griddep_launch_dependents();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x, n16 = n / 16;
  for (size_t j = i0; j < n16; j += stride) reinterpret_cast<uint4*>(dst)[j] = reinterpret_cast<const uint4*>(src)[j];
  for (size_t j = n16 * 16 + i0; j < n; j += stride) dst[j] = src[j];
}
cudaError_t copy_bytes(void* dst, const void* src, size_t n, cudaStream_t s, bool pdl) {
  const size_t n16 = (n + 15) / 16;
  const int blocks = static_cast<int>(std::min<size_t>((n16 + 255) / 256, static_cast<size_t>(4 * sm_count())));
  return launch_kernel(graph_copy_kernel, dim3(std::max(blocks, 1)), dim3(256), 0, s, pdl,
                       static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), n);
}

// One CTA waits on an mbarrier that nothing arrives on, through the pipeline's
// bounded wait; it must give up after limit_ns and record its code.
__global__ void selftest_wait_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait(smem_addr(&bar), 0, &abort_flag, err, DEV_TIMEOUT_SELFTEST, 0, limit_ns);
}
}  // namespace nvf

static nvf_status validate_route(int32_t T, int32_t E, int32_t k, int32_t shared) {
  NVF_REQUIRE(T >= 0 && T <= (1 << 24), "T=%d must be in [0, 2^24]", T);
  NVF_REQUIRE(E >= 1 && E <= 1024, "E=%d must be in [1, 1024]", E);
  NVF_REQUIRE(k >= 1 && k <= E && k <= 32, "k=%d must be in [1, min(E=%d, 32)]", k, E);
  NVF_REQUIRE(shared == 0 || shared == 1, "shared_expert=%d must be 0 or 1", shared);
  NVF_REQUIRE(static_cast<int64_t>(T) * (k + shared) < (int64_t(1) << 31), "T*(k+shared) overflows int32");
  return NVF_OK;
}

namespace nvf {
// The checks moe_route_permute_noalloc makes before it touches its fixed
// scratch: the same device check and argument checks as moe_route_permute, in
// the same order, so that both entry points return the same status for the
// same fault.
nvf_status route_precheck(int32_t T, int32_t E, int32_t k, int32_t shared) {
  NVF_BEGIN();
  (void)dev_;
  return validate_route(T, E, k, shared);
}
}  // namespace nvf

extern "C" {

nvf_status nvf_selftest_bounded_wait(uint64_t limit_ns, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(limit_ns >= 1000 && limit_ns <= 10000000000ull, "limit_ns=%llu must be in [1e3, 1e10]",
              static_cast<unsigned long long>(limit_ns));
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_->err, limit_ns);
  NVF_CUDA(cudaGetLastError(), "self-test launch");
  return NVF_OK;
}

nvf_status nvf_w13_row_map(int32_t I, int32_t* map) {
  g_msg[0] = 0;
  NVF_REQUIRE(I > 0 && I % 64 == 0, "I=%d must be a positive multiple of 64", I);
  NVF_REQUIRE(map != nullptr, "map must not be NULL");
  for (int32_t r = 0; r < 2 * I; ++r) map[r] = static_cast<int32_t>(w13_source_row(r, I));
  return NVF_OK;
}

size_t nvfp4_tiled_bytes(int64_t rows, int32_t G, int32_t K) {
  if (rows < 0 || G < 0 || K <= 0) return 0;
  return static_cast<size_t>((rows + 127) / 128 + G) * num_k_tiles(K) * TILE_BYTES;
}

nvf_status nvfp4_global_scale(const void* x, int32_t x_dtype, int64_t groups, int64_t n, float* gs_out,
                              void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(x != nullptr && gs_out != nullptr, "x and gs_out must not be NULL");
  NVF_REQUIRE(x_dtype == NVF_F32 || x_dtype == NVF_BF16, "x_dtype=%d must be NVF_F32 or NVF_BF16", x_dtype);
  NVF_REQUIRE(groups >= 1 && groups <= 65535 && n >= 1, "groups=%lld (1..65535), n=%lld (>=1)", (long long)groups,
              (long long)n);
  NVF_CUDA(launch_global_scale(x, x_dtype, groups, n, gs_out, static_cast<cudaStream_t>(stream)), "global scale");
  return NVF_OK;
}

nvf_status nvfp4_quantize(const void* x, int32_t x_dtype, int64_t rows, int32_t K, int64_t ldx,
                          const int32_t* gather_rows, const int32_t* group_offsets, const int32_t* tile_offsets,
                          int32_t G, const float* gscale, uint8_t* codes, uint8_t* scales, int32_t layout,
                          void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(layout >= NVF_LAYOUT_ROWMAJOR && layout <= NVF_LAYOUT_TILED_GROUPED, "bad layout %d", layout);
  NVF_REQUIRE(x && gscale && codes && (scales || layout != NVF_LAYOUT_ROWMAJOR),
              "x, gscale, codes (and scales for NVF_LAYOUT_ROWMAJOR) must not be NULL");
  NVF_REQUIRE(x_dtype == NVF_F32 || x_dtype == NVF_BF16, "x_dtype=%d must be NVF_F32 or NVF_BF16", x_dtype);
  NVF_REQUIRE(rows >= 0 && K > 0 && K % 64 == 0, "rows=%lld K=%d: K must be a positive multiple of 64",
              (long long)rows, K);
  NVF_REQUIRE(ldx >= K, "ldx=%lld < K=%d", (long long)ldx, K);
  const int esz = x_dtype == NVF_F32 ? 4 : 2;
  NVF_REQUIRE(aligned16(x) && (ldx * esz) % 16 == 0, "x must be 16-byte aligned with a 16-byte multiple row pitch");
  NVF_REQUIRE(aligned16(codes) && (reinterpret_cast<uintptr_t>(scales) & 3u) == 0,
              "codes must be 16-byte and scales 4-byte aligned");
  if (group_offsets) NVF_REQUIRE(G >= 1, "G=%d must be >= 1 with group_offsets", G);
  if (layout == NVF_LAYOUT_TILED_GROUPED)
    NVF_REQUIRE(group_offsets && tile_offsets, "NVF_LAYOUT_TILED_GROUPED needs group_offsets and tile_offsets");
  QuantArgs a{x, x_dtype, rows, K, ldx, gather_rows, group_offsets, tile_offsets, group_offsets ? G : 1,
              gscale, codes, scales, layout};
  if (layout == NVF_LAYOUT_TILED && group_offsets == nullptr) {
    // weights: G equal groups of rows (one expert's N rows each), gscale[g] per group
    NVF_REQUIRE(G >= 1 && rows % G == 0, "NVF_LAYOUT_TILED: rows=%lld must split into G=%d equal groups",
                (long long)rows, G);
    a.rows_per_group = rows > 0 ? static_cast<int32_t>(rows / G) : 0;
    NVF_REQUIRE(rows / G < (int64_t(1) << 31), "group too large");
  }
  NVF_CUDA(launch_quantize(a, static_cast<cudaStream_t>(stream)), "quantize launch");
  return NVF_OK;
}

nvf_status nvfp4_prepare_weights(const void* w13_src, const void* w2_src, int32_t src_dtype, int32_t e0,
                                 int32_t n_experts, int32_t H, int32_t I, uint8_t* w13, float* gs_w13, uint8_t* w2,
                                 float* gs_w2, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(w13_src && w2_src && w13 && gs_w13 && w2 && gs_w2, "weight pointers must not be NULL");
  NVF_REQUIRE(src_dtype == NVF_F32 || src_dtype == NVF_BF16, "src_dtype=%d must be NVF_F32 or NVF_BF16", src_dtype);
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(I > 0 && I % 64 == 0, "I=%d must be a positive multiple of 64", I);
  NVF_REQUIRE(e0 >= 0 && n_experts >= 1 && n_experts <= 65535, "e0=%d must be >= 0 and n_experts=%d in [1, 65535]",
              e0, n_experts);
  NVF_REQUIRE(static_cast<int64_t>(e0 + n_experts) * 2 * I * H < (int64_t(1) << 40), "weight stack too large");
  NVF_REQUIRE(aligned16(w13_src) && aligned16(w2_src) && aligned16(w13) && aligned16(w2),
              "w13_src, w2_src, w13 and w2 must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t rows13 = static_cast<int64_t>(n_experts) * 2 * I, rows2 = static_cast<int64_t>(n_experts) * H;
  // per-expert global scales gs = amax / 2688 (1 for an all-zero expert)
  NVF_CUDA(launch_global_scale(w13_src, src_dtype, n_experts, int64_t(2) * I * H, gs_w13 + e0, s), "w13 global scales");
  NVF_CUDA(launch_global_scale(w2_src, src_dtype, n_experts, int64_t(H) * I, gs_w2 + e0, s), "w2 global scales");
  // NVFP4 rows along the input dimension into the TILED layout; w13 rows in the
  // order the fused SiLU-and-mul epilogue reads them.  Expert boundaries fall on
  // 128-row tiles (2I and H are multiples of 128), so expert e starts at chunk
  // e * rows / 128 * nkt of each buffer.
  QuantArgs a13{w13_src, src_dtype, rows13, H, H, nullptr, nullptr, nullptr, 1, gs_w13 + e0,
                w13 + nvfp4_tiled_bytes(static_cast<int64_t>(e0) * 2 * I, 0, H), nullptr, LAYOUT_TILED};
  a13.rows_per_group = 2 * I;
  a13.w13_I = I;
  NVF_CUDA(launch_quantize(a13, s), "w13 quantize");
  QuantArgs a2{w2_src, src_dtype, rows2, I, I, nullptr, nullptr, nullptr, 1, gs_w2 + e0,
               w2 + nvfp4_tiled_bytes(static_cast<int64_t>(e0) * H, 0, I), nullptr, LAYOUT_TILED};
  a2.rows_per_group = H;
  NVF_CUDA(launch_quantize(a2, s), "w2 quantize");
  return NVF_OK;
}

nvf_status moe_route_permute_workspace_size(int32_t T, int32_t E, size_t* bytes) {
  g_msg[0] = 0;
  NVF_REQUIRE(bytes != nullptr && T >= 0 && E >= 1, "bad arguments");
  *bytes = align256(route_scratch_bytes(T, E));
  if (*bytes == 0) *bytes = 256;
  return NVF_OK;
}


nvf_status moe_route_permute(const float* logits, const float* bias, int32_t T, int32_t E, int32_t k,
                             int32_t renormalize, int32_t shared_expert, int32_t* topk_ids, float* topk_w,
                             int32_t* expert_offsets, int32_t* tile_offsets, int32_t* perm_to_src,
                             int32_t* src_to_perm, int32_t* perm_token, void* ws, size_t ws_bytes, void* stream) {
  NVF_BEGIN();
  {
    nvf_status s = validate_route(T, E, k, shared_expert);
    if (s != NVF_OK) return s;
  }
  NVF_REQUIRE(expert_offsets && tile_offsets, "expert_offsets and tile_offsets must not be NULL");
  if (T > 0)
    NVF_REQUIRE(logits && topk_ids && topk_w && perm_to_src && src_to_perm && perm_token,
                "logits, topk_ids, topk_w, perm_to_src, src_to_perm and perm_token must not be NULL");
  size_t need = 0;
  moe_route_permute_workspace_size(T, E, &need);
  NVF_REQUIRE(ws != nullptr || need == 0, "ws must not be NULL");
  if (ws_bytes < need) return fail(NVF_ERR_WORKSPACE, "workspace %zu bytes < %zu needed (T=%d E=%d)", ws_bytes, need, T, E);
  RouteArgs a = make_route_args(logits, bias, T, E, k, renormalize, shared_expert, topk_ids, topk_w, expert_offsets,
                                tile_offsets, perm_to_src, src_to_perm, perm_token, ws);
  NVF_CUDA(launch_route(a, static_cast<cudaStream_t>(stream)), "route launch");
  return NVF_OK;
}

static nvf_status validate_gemm(const uint8_t* A, int64_t a_rows, const uint8_t* B, int32_t G, int32_t N,
                                int32_t K) {
  NVF_REQUIRE(A && B, "A and B must not be NULL");
  NVF_REQUIRE(G >= 1 && G <= 4096, "G=%d must be in [1, 4096]", G);
  NVF_REQUIRE(N > 0 && N % 128 == 0, "N=%d must be a positive multiple of 128", N);
  NVF_REQUIRE(K > 0 && K % 64 == 0, "K=%d must be a positive multiple of 64", K);
  NVF_REQUIRE(a_rows >= 0 && a_rows < (int64_t(1) << 31), "a_rows=%lld out of range", (long long)a_rows);
  NVF_REQUIRE(static_cast<int64_t>(G) * N < (int64_t(1) << 31), "G*N overflows int32");
  NVF_REQUIRE(aligned16(A) && aligned16(B), "A and B must be 16-byte aligned");
  return NVF_OK;
}

nvf_status nvfp4_grouped_gemm(const uint8_t* A, int64_t a_rows, const uint8_t* B, const float* gs_a,
                              const float* gs_b, const int32_t* group_offsets, const int32_t* tile_offsets, int32_t G,
                              int32_t N, int32_t K, int32_t out_dtype, void* D, int64_t ldd, void* stream) {
  NVF_BEGIN();
  {
    nvf_status s = validate_gemm(A, a_rows, B, G, N, K);
    if (s != NVF_OK) return s;
  }
  NVF_REQUIRE(gs_a && gs_b && group_offsets && tile_offsets && D, "gs_a, gs_b, offsets and D must not be NULL");
  NVF_REQUIRE(out_dtype == NVF_F32 || out_dtype == NVF_BF16, "out_dtype=%d must be NVF_F32 or NVF_BF16", out_dtype);
  const int esz = out_dtype == NVF_F32 ? 4 : 2;
  NVF_REQUIRE(ldd >= N && (ldd * esz) % 16 == 0 && aligned16(D),
              "D must be 16-byte aligned with ldd >= N=%d and ldd*%d bytes a multiple of 16 (ldd=%lld)", N, esz,
              (long long)ldd);
  GemmArgs a{};
  a.a = A; a.a_rows = a_rows; a.b = B; a.gs_a = gs_a; a.gs_b = gs_b;
  a.offsets = group_offsets; a.tile_offs = tile_offsets; a.G = G; a.N = N; a.K = K;
  a.epilogue = out_dtype == NVF_F32 ? EPI_STORE_F32 : EPI_STORE_BF16;
  a.d_align32 = (reinterpret_cast<uintptr_t>(D) & 31u) == 0 && (ldd * (out_dtype == NVF_F32 ? 4 : 2)) % 32 == 0;
  a.small_a = a_rows <= 32;  // no group can hold more rows than the buffer
  a.d = D; a.ldd = ldd; a.err = dev_->err;
  const char* why = nullptr;
  cudaError_t e = launch_grouped_gemm(a, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess)
    return fail(NVF_ERR_CUDA, "grouped GEMM (G=%d M<=%lld N=%d K=%d): %s", G, (long long)a_rows, N, K,
                why ? why : cudaGetErrorString(e));
  return NVF_OK;
}

nvf_status nvfp4_moe_workspace_layout(int32_t T, int32_t E, int32_t H, int32_t I, int32_t k, int32_t shared,
                                      nvf_moe_ws_layout* L) {
  g_msg[0] = 0;
  NVF_REQUIRE(L != nullptr, "layout must not be NULL");
  {
    nvf_status s = validate_route(T, E, k, shared);
    if (s != NVF_OK) return s;
  }
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(I > 0 && I % 64 == 0, "I=%d must be a positive multiple of 64", I);
  const int64_t Et = E + shared;
  const int64_t R = static_cast<int64_t>(T) * k + (shared ? T : 0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L->R = R;
  L->topk_ids = take(sizeof(int32_t) * T * k);
  L->topk_w = take(sizeof(float) * T * k);
  L->expert_offsets = take(sizeof(int32_t) * (Et + 1));
  L->tile_offsets = take(sizeof(int32_t) * (Et + 1));
  L->perm_to_src = take(sizeof(int32_t) * R);
  L->src_to_perm = take(sizeof(int32_t) * R);
  L->perm_token = take(sizeof(int32_t) * R);
  size_t rs = 0;
  moe_route_permute_workspace_size(T, E, &rs);
  L->route_scratch = take(rs);
  L->tile_group = take(sizeof(int32_t) * (static_cast<size_t>(R) / 128 + Et + 1));
  L->a1 = take(nvfp4_tiled_bytes(R, static_cast<int32_t>(Et), H));
  L->a2 = take(nvfp4_tiled_bytes(R, static_cast<int32_t>(Et), I));
  L->y = take(sizeof(float) * static_cast<size_t>(R) * H);
  L->logits = take(sizeof(float) * static_cast<size_t>(T) * Et);
  L->total = off;
  return NVF_OK;
}

}  // extern "C"

// The layer from routing to combine.  With w_gate the router gate runs first and
// writes the logits into the workspace ([T, E + gated] rows); gated: the last
// gate row's logit gates the shared expert.
static nvf_status forward_impl(const nvf_moe_weights* w, const void* w_gate, int32_t gated, const void* x,
                               const float* logits, const float* bias, int32_t T, int32_t k, int32_t renormalize,
                               const float* gs_a1, const float* gs_a2, int32_t out_dtype, void* out, float* h_dump,
                               void* ws, size_t ws_bytes, void* const* stage_events, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(w != nullptr, "weights must not be NULL");
  nvf_moe_ws_layout L;
  {
    nvf_status s = nvfp4_moe_workspace_layout(T, w->E, w->H, w->I, k, w->shared, &L);
    if (s != NVF_OK) return s;
  }
  const int32_t E = w->E, H = w->H, I = w->I, Et = w->E + w->shared;
  NVF_REQUIRE(w->w13 && w->gs_w13 && w->w2 && w->gs_w2, "weight pointers must not be NULL");
  NVF_REQUIRE(aligned16(w->w13) && aligned16(w->w2), "weight buffers must be 16-byte aligned");
  NVF_REQUIRE(out_dtype == NVF_F32 || out_dtype == NVF_BF16, "out_dtype=%d must be NVF_F32 or NVF_BF16", out_dtype);
  NVF_REQUIRE(gated == 0 || (gated == 1 && w->shared == 1), "shared_gate=%d needs a layer with a shared expert",
              gated);
  if (T == 0) return NVF_OK;
  NVF_REQUIRE(x && (logits || w_gate) && gs_a1 && gs_a2 && out, "x, logits (or w_gate), gs_a1, gs_a2 and out must not be NULL");
  if (w_gate) NVF_REQUIRE(aligned16(w_gate), "w_gate must be 16-byte aligned");
  NVF_REQUIRE(aligned16(x) && aligned16(out) && (h_dump == nullptr || aligned16(h_dump)),
              "x, out and h_dump must be 16-byte aligned");
  NVF_REQUIRE(ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "ws must be 256-byte aligned");
  if (ws_bytes < L.total)
    return fail(NVF_ERR_WORKSPACE, "workspace %zu bytes < %zu needed (T=%d E=%d H=%d I=%d k=%d)", ws_bytes, L.total,
                T, E, H, I, k);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto i32 = [&](size_t o) { return reinterpret_cast<int32_t*>(base + o); };
  // Stage events: while the stream is being captured into a graph they are
  // recorded as external event nodes (so that the graph records them at replay);
  // otherwise they are plain records.
  unsigned int ev_flags = cudaEventRecordDefault;
  if (stage_events) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    NVF_CUDA(cudaStreamIsCapturing(s, &cs), "cudaStreamIsCapturing");
    if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
  }
  auto mark = [&](int i) -> cudaError_t {
    return stage_events ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(stage_events[i]), s, ev_flags)
                        : cudaSuccess;
  };
  int64_t ldl = E;
  if (w_gate) {
    // router gate: logits (and the shared expert's gate logit) into the workspace
    float* lg = reinterpret_cast<float*>(base + L.logits);
    NVF_CUDA(launch_router_gemm(x, w_gate, T, H, E + gated, lg, E + gated, dev_->err, s), "router gate launch");
    logits = lg;
    ldl = E + gated;
  }
  NVF_CUDA(mark(0), "cudaEventRecord");

  // routing, permutation and the activation quantization (A1) in one pass
  RouteArgs ra = make_route_args(logits, bias, T, E, k, renormalize, w->shared, i32(L.topk_ids),
                                 reinterpret_cast<float*>(base + L.topk_w), i32(L.expert_offsets),
                                 i32(L.tile_offsets), i32(L.perm_to_src), i32(L.src_to_perm), i32(L.perm_token),
                                 base + L.route_scratch);
  ra.ldl = ldl;
  ra.x = x;
  ra.H = H;
  ra.gs_a1 = gs_a1;
  ra.a1 = base + L.a1;
  ra.tile_group = i32(L.tile_group);
  // Every kernel starts while its predecessor drains (programmatic dependent
  // launch), unless stage boundaries are being timed: an event between two
  // kernels is a full dependency.  The first routing kernel too: it waits for
  // whatever ran before it on the stream (griddepcontrol.wait) before it reads
  // anything, and the kernels after it start only once it has passed that wait.
  const bool pdl = stage_events == nullptr;
  ra.pdl = pdl;
  NVF_CUDA(launch_route(ra, s), "route launch");
  NVF_CUDA(mark(1), "cudaEventRecord");

  NVF_CUDA(mark(2), "cudaEventRecord");

  const char* why = nullptr;
  GemmArgs g1{};
  g1.a = base + L.a1; g1.a_rows = L.R;
  g1.b = w->w13; g1.gs_a = gs_a1; g1.gs_b = w->gs_w13;
  g1.offsets = i32(L.expert_offsets); g1.tile_offs = i32(L.tile_offsets); g1.G = Et; g1.N = 2 * I; g1.K = H;
  g1.tile_group = i32(L.tile_group);
  g1.small_a = T <= 32;  // no expert (the shared one included) sees more rows than there are tokens
  g1.epilogue = EPI_SWIGLU_QUANT; g1.q_codes = base + L.a2; g1.gs_q = gs_a2;
  g1.h_dump = h_dump; g1.err = dev_->err; g1.pdl = pdl;
  cudaError_t e = launch_grouped_gemm(g1, s, &why);
  if (e != cudaSuccess)
    return fail(NVF_ERR_CUDA, "gate_up GEMM (E'=%d R=%lld N=%d K=%d): %s", Et, (long long)L.R, 2 * I, H,
                why ? why : cudaGetErrorString(e));
  NVF_CUDA(mark(3), "cudaEventRecord");

  GemmArgs g2{};
  g2.a = base + L.a2; g2.a_rows = L.R;
  g2.b = w->w2; g2.gs_a = gs_a2; g2.gs_b = w->gs_w2;
  g2.offsets = i32(L.expert_offsets); g2.tile_offs = i32(L.tile_offsets); g2.G = Et; g2.N = H; g2.K = I;
  g2.tile_group = i32(L.tile_group);
  g2.small_a = T <= 32;
  // y has the output's type: FP32 for parity runs, BF16 for production (half the
  // bytes of the y round trip through HBM; the combine still sums in FP32)
  g2.epilogue = out_dtype == NVF_F32 ? EPI_STORE_F32 : EPI_STORE_BF16;
  g2.d = base + L.y; g2.ldd = H; g2.err = dev_->err;
  g2.d_align32 = true;  // 256-byte aligned workspace, H a multiple of 128
  // With programmatic dependent launch the down GEMM may begin before the gate_up
  // GEMM ends and prefetch its first weight tile before its own dependency wait.
  // The group tables it reads for that come from the routing kernel, two launches
  // back; they are already complete: the gate_up GEMM executes its dependency
  // wait on the routing kernel before it allows this launch to begin.
  g2.pdl = pdl; g2.early_weights = pdl;
  e = launch_grouped_gemm(g2, s, &why);
  if (e != cudaSuccess)
    return fail(NVF_ERR_CUDA, "down GEMM (E'=%d R=%lld N=%d K=%d): %s", Et, (long long)L.R, H, I,
                why ? why : cudaGetErrorString(e));
  NVF_CUDA(mark(4), "cudaEventRecord");

  NVF_CUDA(launch_combine(base + L.y, H, reinterpret_cast<const float*>(base + L.topk_w),
                          i32(L.src_to_perm), T, k, w->shared, out_dtype, out, s, pdl,
                          gated ? logits + E : nullptr, ldl),
           "combine launch");
  NVF_CUDA(mark(5), "cudaEventRecord");
  return NVF_OK;
}

extern "C" {

nvf_status nvfp4_moe_forward(const nvf_moe_weights* w, const void* x, const float* logits, const float* bias,
                             int32_t T, int32_t k, int32_t renormalize, const float* gs_a1, const float* gs_a2,
                             int32_t out_dtype, void* out, float* h_dump, void* ws, size_t ws_bytes,
                             void* const* stage_events, void* stream) {
  return forward_impl(w, nullptr, 0, x, logits, bias, T, k, renormalize, gs_a1, gs_a2, out_dtype, out, h_dump, ws,
                      ws_bytes, stage_events, stream);
}

nvf_status nvfp4_moe_forward_gated(const nvf_moe_weights* w, const void* w_gate, int32_t shared_gate, const void* x,
                                   const float* bias, int32_t T, int32_t k, int32_t renormalize, const float* gs_a1,
                                   const float* gs_a2, int32_t out_dtype, void* out, void* ws, size_t ws_bytes,
                                   void* stream) {
  g_msg[0] = 0;
  NVF_REQUIRE(w_gate != nullptr, "w_gate must not be NULL");
  return forward_impl(w, w_gate, shared_gate, x, nullptr, bias, T, k, renormalize, gs_a1, gs_a2, out_dtype, out,
                      nullptr, ws, ws_bytes, nullptr, stream);
}

nvf_status nvfp4_w4a16_grouped_gemm(const void* A, int32_t a_dtype, int64_t a_rows, int64_t lda, const uint8_t* B,
                                    const float* gs_b, const int32_t* group_offsets, const int32_t* tile_offsets,
                                    int32_t G, int32_t N, int32_t K, int32_t out_dtype, void* D, int64_t ldd,
                                    void* stream) {
  NVF_BEGIN();
  {
    nvf_status s = validate_gemm(static_cast<const uint8_t*>(A), a_rows, B, G, N, K);
    if (s != NVF_OK) return s;
  }
  NVF_REQUIRE(gs_b && group_offsets && tile_offsets && D, "gs_b, offsets and D must not be NULL");
  NVF_REQUIRE(a_dtype == NVF_F16 || a_dtype == NVF_BF16, "a_dtype=%d must be NVF_F16 or NVF_BF16", a_dtype);
  NVF_REQUIRE(lda >= K && lda % 8 == 0, "lda=%lld must be >= K=%d and a multiple of 8", (long long)lda, K);
  NVF_REQUIRE(out_dtype == NVF_F32 || out_dtype == NVF_BF16, "out_dtype=%d must be NVF_F32 or NVF_BF16", out_dtype);
  const int esz = out_dtype == NVF_F32 ? 4 : 2;
  NVF_REQUIRE(ldd >= N && (ldd * esz) % 16 == 0 && aligned16(D),
              "D must be 16-byte aligned with ldd >= N=%d and ldd*%d bytes a multiple of 16 (ldd=%lld)", N, esz,
              (long long)ldd);
  NVF_CUDA(launch_w4a16(A, a_dtype == NVF_BF16, a_rows, lda, B, gs_b, group_offsets, tile_offsets, G, N, K,
                        out_dtype == NVF_BF16, D, ldd,
                        dev_->err, static_cast<cudaStream_t>(stream)),
           "W4A16 GEMM launch");
  return NVF_OK;
}

size_t nvf_ep_row_bytes(int32_t H) { return H > 0 ? ep_row_bytes(H) : 0; }

size_t nvf_ep_receive_scratch_words(int32_t G, int32_t El) {
  return G > 0 && El > 0 ? 2 * static_cast<size_t>(G) * (El + 1) : 0;
}

nvf_status nvf_ep_dispatch(const void* x, int32_t T, int32_t H, int32_t E, int32_t k, int32_t shared, int32_t G,
                           int32_t rank, const int32_t* expert_offsets, const int32_t* perm_token,
                           const int32_t* perm_to_src, const float* gs_a1, void* send_rows, int32_t* send_counts,
                           int32_t* src_to_send, void* stream) {
  NVF_BEGIN();
  {
    nvf_status st = validate_route(T, E, k, shared);
    if (st != NVF_OK) return st;
  }
  NVF_REQUIRE(G >= 1 && G <= 1024 && E % G == 0, "G=%d must be in [1, 1024] and divide E=%d", G, E);
  NVF_REQUIRE(rank >= 0 && rank < G, "rank=%d out of [0, %d)", rank, G);
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(expert_offsets && gs_a1 && send_counts, "expert_offsets, gs_a1 and send_counts must not be NULL");
  if (T > 0) {
    NVF_REQUIRE(x && perm_token && perm_to_src && send_rows && src_to_send,
                "x, perm_token, perm_to_src, send_rows and src_to_send must not be NULL");
    NVF_REQUIRE(aligned16(x) && aligned16(send_rows), "x and send_rows must be 16-byte aligned");
  }
  EpDispatchArgs a{};
  a.x = x; a.T = T; a.H = H; a.E = E; a.k = k; a.shared = shared; a.G = G; a.rank = rank;
  a.offsets = expert_offsets; a.perm_token = perm_token; a.perm_to_src = perm_to_src; a.gs_a1 = gs_a1;
  a.send = static_cast<uint8_t*>(send_rows); a.row_bytes = static_cast<int32_t>(ep_row_bytes(H));
  a.send_counts = send_counts; a.src_to_send = src_to_send;
  NVF_CUDA(launch_ep_dispatch(a, static_cast<cudaStream_t>(stream)), "EP dispatch launch");
  return NVF_OK;
}

nvf_status nvf_ep_receive(const void* recv_rows, int64_t n_recv, const int32_t* recv_counts, int32_t G, int32_t El,
                          int32_t shared, int32_t H, uint8_t* a1, int32_t* local_offsets,
                          int32_t* local_tile_offsets, int32_t* recv_to_grp, int32_t* grp_to_recv, int32_t* scratch,
                          void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(G >= 1 && G <= 1024 && El >= 1 && (shared == 0 || shared == 1), "G=%d, El=%d, shared=%d out of range",
              G, El, shared);
  NVF_REQUIRE(static_cast<int64_t>(G) * (El + 1) <= 57344, "G * (El + 1) = %lld exceeds 57344",
              static_cast<long long>(G) * (El + 1));
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(n_recv >= 0 && n_recv < (int64_t(1) << 31), "n_recv=%lld out of range", (long long)n_recv);
  NVF_REQUIRE(recv_counts && local_offsets && local_tile_offsets && scratch,
              "recv_counts, local_offsets, local_tile_offsets and scratch must not be NULL");
  if (n_recv > 0) {
    NVF_REQUIRE(recv_rows && a1 && recv_to_grp, "recv_rows, a1 and recv_to_grp must not be NULL");
    NVF_REQUIRE(aligned16(recv_rows) && aligned16(a1), "recv_rows and a1 must be 16-byte aligned");
  }
  NVF_CUDA(launch_ep_receive(static_cast<const uint8_t*>(recv_rows), n_recv, static_cast<int>(ep_row_bytes(H)),
                             recv_counts, G, El, shared, H, a1, local_offsets, local_tile_offsets, recv_to_grp,
                             grp_to_recv, scratch, dev_->err, static_cast<cudaStream_t>(stream)),
           "EP receive launch");
  return NVF_OK;
}

nvf_status nvfp4_moe_experts(const nvf_moe_weights* w, const uint8_t* a1, int64_t a_rows, const int32_t* offsets,
                             const int32_t* tile_offsets, const float* gs_a1, const float* gs_a2, int32_t out_dtype,
                             void* y, const int32_t* y_rows, void* ws, size_t ws_bytes, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(w != nullptr, "weights must not be NULL");
  NVF_REQUIRE(w->E >= 1 && (w->shared == 0 || w->shared == 1) && w->H > 0 && w->H % 128 == 0 && w->I > 0 &&
                  w->I % 64 == 0,
              "weights: E=%d shared=%d H=%d I=%d out of range", w->E, w->shared, w->H, w->I);
  NVF_REQUIRE(a_rows >= 0 && a_rows < (int64_t(1) << 31), "a_rows=%lld out of range", (long long)a_rows);
  NVF_REQUIRE(out_dtype == NVF_F32 || out_dtype == NVF_BF16, "out_dtype=%d must be NVF_F32 or NVF_BF16", out_dtype);
  if (a_rows == 0) return NVF_OK;
  const int32_t Et = w->E + w->shared, H = w->H, I = w->I;
  NVF_REQUIRE(a1 && offsets && tile_offsets && gs_a1 && gs_a2 && y && ws,
              "a1, offsets, tile_offsets, gs_a1, gs_a2, y and ws must not be NULL");
  NVF_REQUIRE(w->w13 && w->gs_w13 && w->w2 && w->gs_w2, "weight pointers must not be NULL");
  NVF_REQUIRE(aligned16(a1) && aligned16(y) && aligned16(w->w13) && aligned16(w->w2),
              "a1, y and the weights must be 16-byte aligned");
  NVF_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "ws must be 256-byte aligned");
  const size_t need = nvfp4_tiled_bytes(a_rows, Et, I);
  if (ws_bytes < need) return fail(NVF_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* why = nullptr;
  GemmArgs g1{};
  g1.a = a1; g1.a_rows = a_rows;
  g1.b = w->w13; g1.gs_a = gs_a1; g1.gs_b = w->gs_w13;
  g1.offsets = offsets; g1.tile_offs = tile_offsets; g1.G = Et; g1.N = 2 * I; g1.K = H;
  g1.small_a = a_rows <= 32;  // no group can hold more rows than the buffer
  g1.epilogue = EPI_SWIGLU_QUANT; g1.q_codes = static_cast<uint8_t*>(ws); g1.gs_q = gs_a2;
  g1.err = dev_->err;
  cudaError_t e = launch_grouped_gemm(g1, s, &why);
  if (e != cudaSuccess)
    return fail(NVF_ERR_CUDA, "gate_up GEMM (E'=%d rows=%lld): %s", Et, (long long)a_rows,
                why ? why : cudaGetErrorString(e));
  GemmArgs g2{};
  g2.a = static_cast<uint8_t*>(ws); g2.a_rows = a_rows;
  g2.b = w->w2; g2.gs_a = gs_a2; g2.gs_b = w->gs_w2;
  g2.offsets = offsets; g2.tile_offs = tile_offsets; g2.G = Et; g2.N = H; g2.K = I;
  g2.small_a = a_rows <= 32;
  g2.epilogue = out_dtype == NVF_F32 ? EPI_STORE_F32 : EPI_STORE_BF16;
  g2.d = y; g2.ldd = H; g2.err = dev_->err; g2.d_rows = y_rows;
  g2.d_align32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
  e = launch_grouped_gemm(g2, s, &why);
  if (e != cudaSuccess)
    return fail(NVF_ERR_CUDA, "down GEMM (E'=%d rows=%lld): %s", Et, (long long)a_rows,
                why ? why : cudaGetErrorString(e));
  return NVF_OK;
}

nvf_status nvf_ep_return(const void* y, int64_t n_recv, int32_t H, int32_t dtype, const int32_t* recv_to_grp,
                         void* y_ret, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(dtype == NVF_F32 || dtype == NVF_BF16, "dtype=%d must be NVF_F32 or NVF_BF16", dtype);
  NVF_REQUIRE(n_recv >= 0 && n_recv < (int64_t(1) << 31), "n_recv=%lld out of range", (long long)n_recv);
  if (n_recv == 0) return NVF_OK;
  NVF_REQUIRE(y && recv_to_grp && y_ret, "y, recv_to_grp and y_ret must not be NULL");
  NVF_REQUIRE(aligned16(y) && aligned16(y_ret), "y and y_ret must be 16-byte aligned");
  NVF_CUDA(launch_gather_rows(y, n_recv, static_cast<int64_t>(H) * (dtype == NVF_F32 ? 4 : 2), recv_to_grp, y_ret,
                              static_cast<cudaStream_t>(stream)),
           "EP return launch");
  return NVF_OK;
}

nvf_status nvf_moe_combine(const void* y, int32_t H, int32_t dtype, const float* topk_w, const int32_t* src_to_row,
                           int32_t T, int32_t k, int32_t shared, void* out, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(dtype == NVF_F32 || dtype == NVF_BF16, "dtype=%d must be NVF_F32 or NVF_BF16", dtype);
  NVF_REQUIRE(T >= 0 && k >= 1 && k <= 64 && (shared == 0 || shared == 1), "T=%d k=%d shared=%d out of range", T, k,
              shared);
  if (T == 0) return NVF_OK;
  NVF_REQUIRE(y && topk_w && src_to_row && out, "y, topk_w, src_to_row and out must not be NULL");
  NVF_REQUIRE((reinterpret_cast<uintptr_t>(y) & 31u) == 0 && aligned16(out), "y must be 32-byte and out 16-byte aligned");
  NVF_CUDA(launch_combine(y, H, topk_w, src_to_row, T, k, shared, dtype == NVF_BF16 ? X_BF16 : X_F32, out,
                          static_cast<cudaStream_t>(stream), false),
           "combine launch");
  return NVF_OK;
}

}  // extern "C"

struct nvf_moe_graph {
  cudaStream_t stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  void* x = nullptr;         // device x, then logits right behind it (one allocation)
  float* logits = nullptr;
  void* out = nullptr;
  void* ws = nullptr;
};

namespace {
void free_graph(nvf_moe_graph* g) {
  if (g == nullptr) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  if (g->stream) cudaStreamDestroy(g->stream);
  cudaFree(g->x);
  cudaFree(g->out);
  cudaFree(g->ws);
  delete g;
}
// The device's address of page-locked host memory, or nullptr (pageable or unmapped).
void* pinned_device_alias(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
}  // namespace

extern "C" {

nvf_status nvf_moe_graph_create(const nvf_moe_weights* w, int32_t T, int32_t k, int32_t renormalize,
                                const float* gs_a1, const float* gs_a2, const float* bias, const void* x_host,
                                const float* logits_host, void* out_host, int32_t out_dtype, nvf_moe_graph** graph) {
  NVF_BEGIN();
  NVF_REQUIRE(graph != nullptr, "graph must not be NULL");
  *graph = nullptr;
  NVF_REQUIRE(w != nullptr && T >= 1, "weights must not be NULL and T=%d must be >= 1", T);
  NVF_REQUIRE(out_dtype == NVF_F32 || out_dtype == NVF_BF16, "out_dtype=%d must be NVF_F32 or NVF_BF16", out_dtype);
  NVF_REQUIRE(x_host && logits_host && out_host, "host buffers must not be NULL");
  void* xd = pinned_device_alias(x_host);
  void* ld = pinned_device_alias(logits_host);
  void* od = pinned_device_alias(out_host);
  NVF_REQUIRE(xd && ld && od, "x_host, logits_host and out_host must be page-locked host memory");
  NVF_REQUIRE(aligned16(xd) && aligned16(ld) && aligned16(od), "host buffers must be 16-byte aligned");
  nvf_moe_ws_layout L;
  {
    nvf_status st = nvfp4_moe_workspace_layout(T, w->E, w->H, w->I, k, w->shared, &L);
    if (st != NVF_OK) return st;
  }
  const size_t xb = static_cast<size_t>(T) * w->H * 2, lb = static_cast<size_t>(T) * w->E * 4;
  const size_t ob = static_cast<size_t>(T) * w->H * (out_dtype == NVF_F32 ? 4 : 2);
  nvf_moe_graph* g = new nvf_moe_graph();
  auto bail = [&](nvf_status st) {
    free_graph(g);
    return st;
  };
  cudaError_t e = cudaStreamCreateWithFlags(&g->stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaMalloc(&g->x, xb + lb);
  g->logits = reinterpret_cast<float*>(static_cast<uint8_t*>(g->x) + xb);   // xb is a multiple of 256
  if (e == cudaSuccess) e = cudaMalloc(&g->out, ob);
  if (e == cudaSuccess) e = cudaMalloc(&g->ws, L.total);
  if (e != cudaSuccess) return bail(cuda_fail(e, "graph buffers"));
  e = cudaStreamBeginCapture(g->stream, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamBeginCapture"));
  // the inputs (one copy when logits_host directly follows x_host, as on the
  // device), then the layer, then the result back
  if (static_cast<const uint8_t*>(ld) == static_cast<const uint8_t*>(xd) + xb) {
    e = copy_bytes(g->x, xd, xb + lb, g->stream, false);
  } else {
    e = copy_bytes(g->x, xd, xb, g->stream, false);
    if (e == cudaSuccess) e = copy_bytes(g->logits, ld, lb, g->stream, true);
  }
  nvf_status st = NVF_OK;
  if (e == cudaSuccess)
    st = forward_impl(w, nullptr, 0, g->x, g->logits, bias, T, k, renormalize, gs_a1, gs_a2, out_dtype, g->out,
                      nullptr, g->ws, L.total, nullptr, g->stream);
  if (e == cudaSuccess && st == NVF_OK) e = copy_bytes(od, g->out, ob, g->stream, true);
  const cudaError_t ec = cudaStreamEndCapture(g->stream, &g->graph);
  if (st != NVF_OK) return bail(st);                     // the forward's own message stands
  if (e != cudaSuccess) return bail(cuda_fail(e, "graph capture"));
  if (ec != cudaSuccess) return bail(cuda_fail(ec, "cudaStreamEndCapture"));
  e = cudaGraphInstantiate(&g->exec, g->graph, 0);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGraphInstantiate"));
  *graph = g;
  return NVF_OK;
}

nvf_status nvf_moe_graph_launch(nvf_moe_graph* graph, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(graph != nullptr && graph->exec != nullptr, "graph must come from nvf_moe_graph_create");
  NVF_CUDA(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)), "cudaGraphLaunch");
  return NVF_OK;
}

nvf_status nvf_moe_graph_destroy(nvf_moe_graph* graph) {
  NVF_BEGIN();
  free_graph(graph);
  return NVF_OK;
}

nvf_status nvf_router_gemm(const void* x, const void* w_gate, int32_t T, int32_t H, int32_t n, float* logits,
                           int64_t ldl, void* stream) {
  NVF_BEGIN();
  NVF_REQUIRE(T >= 0 && n >= 1 && n <= 65535 * 32, "T=%d must be >= 0, n=%d in [1, 2097120]", T, n);
  NVF_REQUIRE(H > 0 && H % 128 == 0, "H=%d must be a positive multiple of 128", H);
  NVF_REQUIRE(ldl >= n, "ldl=%lld < n=%d", (long long)ldl, n);
  if (T == 0) return NVF_OK;
  NVF_REQUIRE(x && w_gate && logits, "x, w_gate and logits must not be NULL");
  NVF_REQUIRE(aligned16(x) && aligned16(w_gate), "x and w_gate must be 16-byte aligned");
  NVF_CUDA(launch_router_gemm(x, w_gate, T, H, n, logits, ldl, dev_->err, static_cast<cudaStream_t>(stream)),
           "router gate launch");
  return NVF_OK;
}

}  // extern "C"
