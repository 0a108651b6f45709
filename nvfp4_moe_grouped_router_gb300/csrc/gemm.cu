// Grouped block-scaled FP4 GEMM for sm_103a (tcgen05, kind::mxf4nvf4).
//
// For every group (expert) g with rows [offsets[g], offsets[g+1]) of A:
//     D[row, n] = alpha_g * sum_k dA[row, k] * dB_g[n, k],  alpha_g = gs_a[g] * gs_b[g]
// where dA, dB are E2M1 codes times their UE4M3 block scales (one per 16 K
// elements).  This is the grouped block-scaled FP4 GEMM the MoE expert
// computation runs on (FlashInfer issue #2723, "The Problem"; vLLM PR #29242,
// "Purpose": nvfp4_blockwise_moe_kernel.cu) with a per-expert alpha and beta = 0
// (vLLM PR #29242 review: alpha_ptr_array, beta = 0.0f).
//
// Tiles are 128 rows of one group x 256 output columns (the last tile of a row
// block is 128 wide when N % 256 == 128); one MMA per 64-element K step is
// 128 x 256 x 64.  On this part the tensor pipe charges per instruction rather
// than per FLOP: an MMA costs about the same for N = 16..128 and only a third
// more at N = 256, and a tcgen05.cp costs about as much as an MMA whatever its
// shape.  So the kernel uses the widest MMA and keeps the scale factors off the
// tensor pipe altogether: four warps, one per 32-lane quarter of TMEM, write
// them with tcgen05.st in the layout the MMA reads (each quarter holds its own
// copy of B's scales; A row r's scales sit in lane r).
//
// Roles (one CTA per SM, persistent, 512 threads = four warpgroups; setmaxnreg
// gives the epilogue warpgroups 192 registers a thread, the others 64 and 56):
//   warps 0-3   scale writers: once a stage has landed, load its scale atoms
//               from shared memory and store them into the stage's TMEM scale
//               slot (warp q writes lanes 32q..32q+31), then signal sf_ready.
//   warps 4-11  epilogue: two warps per 32-lane TMEM quarter, 128 columns
//               each.  They move their whole slice of the accumulator to
//               registers and release it before any arithmetic, so the next
//               tile's MMAs run while this tile is finished: alpha and
//               FP32/BF16 rows, or h = silu(gate) * up requantized to NVFP4
//               straight into the next GEMM's tiled operand.
//   warp 12     producer: per K tile the A chunk (one 18 KB copy of codes and
//               atoms for a full tile; the valid-row prefix and the atoms
//               otherwise) and the weight unit of the tile's 256 rows (one
//               36 KB copy: the weight layout stores it as the stage holds
//               it), moved with 1-D bulk copies into a 3- to 5-deep ring.  The
//               ring's rate is set by the number of copies, not their bytes
//               (measured: 54 KB stages as 6 copies stream 11.8 TB/s from L2,
//               as 2 copies 17.4 TB/s), hence two copies a K tile.  It issues
//               nothing else: L2 prefetches of the weights further ahead
//               competed with the ring's own loads and measured slower.
//   warp 13     MMA issuer: per K tile, once the codes have landed and the
//               scales are in TMEM, four 128x256x64 MMAs into the single
//               256-column TMEM accumulator.
//   warps 14-15 idle (they complete warpgroup 3).
// Every mbarrier wait is bounded; on timeout the kernel records an error word,
// drains what it issued, frees TMEM and returns.
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

#include <cuda_bf16.h>

namespace nvf {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int SF_WARPS = 4;               // warps 0-3 (warpgroup 0): scale writers, one per TMEM lane quarter
constexpr int EPI_WARP0 = SF_WARPS;        // warps 4-11 (warpgroups 1-2): epilogue
constexpr int EPI_WARPS = 8;
constexpr int PRODUCER_WARP = EPI_WARP0 + EPI_WARPS;  // warpgroup 3: producer, MMA issuer and two idle warps
constexpr int MMA_WARP = PRODUCER_WARP + 1;
constexpr int THREADS = 512;
// Registers per thread.  The block is launched with 65536 / 512 = 128 a thread;
// setmaxnreg then moves registers from the scale writers and the control
// warpgroup to the two epilogue warpgroups, whose threads hold a whole
// 128-column slice of the accumulator.  The shares must add up to at most the
// launch's total (a larger request would wait forever), which the host checks
// against the compiled register count before every launch.
constexpr int REG_LAUNCH = 128;
constexpr int REG_SF = 64, REG_CTRL = 56, REG_EPI = 192;
static_assert(REG_SF + REG_CTRL + 2 * REG_EPI <= 4 * REG_LAUNCH, "register split exceeds the launch's registers");
static_assert(THREADS * REG_LAUNCH <= 65536, "launch register budget");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = BN;          // scale slots after the accumulator
constexpr uint32_t SF_SLOT_COLS = 48;     // A: 16 columns, B: 32 columns
// Group tables copied to shared memory once per CTA (when G + 1 fits), so that
// decoding a tile costs a binary search in shared memory instead of a chain of
// dependent global loads on the producer's path.
constexpr int SMEM_GROUPS = 1025;

// Shared-memory layout.  A stage is [A codes][A atoms 2048][B codes 2 x 16384]
// [B atoms 2 x 2048].  When every group has at most 32 rows (a decode batch, a
// linear layer of a few rows) the A codes need 4 KB instead of 16 KB, and the
// space buys a fifth stage: a deeper ring is what lets one SM stream weights
// faster (its pace is the ring's round-trip time, not the bytes per stage).
// The MMA still reads 128 A rows; in the small layout rows 32..127 fall on the
// stage's other bytes and give accumulator rows that are never stored.
// STAGING: the store epilogue of large groups stages each warp's output through
// shared memory (4 KB a warp) so that global stores cover whole 128-byte lines;
// the space comes from a fourth ring stage (a store GEMM's K is short: the down
// GEMM has 3 K tiles a tile).
template <bool SMALL_A, bool STAGING = false>
struct Smem {
  static constexpr int STAGES = SMALL_A ? 5 : (STAGING ? 3 : 4);
  static constexpr int A_ROWS = SMALL_A ? 32 : BM;
  static constexpr int ST_A = 0;
  static constexpr int ST_ASF = A_ROWS * 128;
  static constexpr int ST_B = ST_ASF + TILE_SF_BYTES;
  static constexpr int ST_BSF = ST_B + 2 * TILE_CODE_BYTES;
  static constexpr int STAGE_BYTES = ST_BSF + 2 * TILE_SF_BYTES;
  static constexpr int OFF_GRP = STAGES * STAGE_BYTES;  // int tile_offs[SMEM_GROUPS], offsets[SMEM_GROUPS]
  static constexpr int OFF_BAR = OFF_GRP + 2 * SMEM_GROUPS * 4 + 8;
  static constexpr int NUM_BARS = 3 * STAGES + 3;  // full, empty, sf_ready per stage; acc_full/empty, drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int STG_WARP_BYTES = 4096;        // 32 rows x 128 bytes
  static constexpr int OFF_STG = (OFF_MISC + 16 + 127) & ~127;
  static constexpr int BYTES = (STAGING ? OFF_STG + EPI_WARPS * STG_WARP_BYTES : OFF_MISC + 16) + 1024;  // + alignment slack
  static_assert(SF_COL0 + STAGES * SF_SLOT_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(BYTES <= 227 * 1024, "shared memory budget");
  static_assert(STAGE_BYTES % 1024 == 0 && ST_B % 1024 == 0, "1024-byte alignment");
};

struct Tile {
  int g, mt, nt0, row0, rows;
  bool wide;  // weight tiles nt0 and nt0 + 1 (256 output columns), else nt0 only
};

// Work list of one launch.  Row block (m-tile) x 256 output columns is the
// unit; blocks are dealt to the CTAs round-robin.  When the last round would
// leave at least half of the CTAs idle, its blocks are split into two
// 128-column tiles so that the round takes half as long (only when every block
// is 256 wide, i.e. N % 256 == 0).
struct Sched {
  int nblocks;   // 256-column blocks per row block
  int first_split, total;
};

__device__ __forceinline__ Sched make_sched(const GemmArgs& p) {
  Sched s;
  s.nblocks = (p.N + BN - 1) / BN;
  const int blocks = __ldg(p.tile_offs + p.G) * s.nblocks;
  const int rem = blocks % static_cast<int>(gridDim.x);
  const int nsplit = (p.N % BN == 0 && rem > 0 && 2 * rem <= static_cast<int>(gridDim.x)) ? rem : 0;
  s.first_split = blocks - nsplit;
  s.total = blocks + nsplit;
  return s;
}

// Group tables for decode_tile: shared-memory copies when present, else global.
struct Groups {
  const int* toff;   // [G + 1] in shared memory, or nullptr
  const int* off;
};

__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& p, const Sched& sc, const Groups& gr = Groups{}) {
  Tile x;
  int b = t, half = -1;
  if (t >= sc.first_split) {
    const int u = t - sc.first_split;
    b = sc.first_split + (u >> 1);
    half = u & 1;
  }
  x.mt = b / sc.nblocks;
  const int nb = b - x.mt * sc.nblocks;
  if (gr.toff != nullptr) {
    int lo = 0, hi = p.G;  // last g with toff[g] <= mt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (gr.toff[mid] <= x.mt) lo = mid; else hi = mid;
    }
    x.g = lo;
    x.row0 = gr.off[lo] + (x.mt - gr.toff[lo]) * BM;
    x.rows = min(BM, gr.off[lo + 1] - x.row0);
  } else {
    x.g = p.tile_group != nullptr ? __ldg(p.tile_group + x.mt) : upper_group(p.tile_offs, p.G, x.mt);
    const int local = x.mt - __ldg(p.tile_offs + x.g);
    x.row0 = __ldg(p.offsets + x.g) + local * BM;
    x.rows = min(BM, __ldg(p.offsets + x.g + 1) - x.row0);
  }
  x.wide = half < 0 && (nb + 1) * BN <= p.N;
  x.nt0 = 2 * nb + (half > 0 ? 1 : 0);
  return x;
}


// The scales of one K tile (four 64-element K steps), as the MMA reads them
// from TMEM.  Scale atom (512 bytes, one per K step and 128 rows): 16 bytes per
// atom row j, word c holding the four UE4M3 scales of row j + 32 c.  Lane l of
// every 32-lane quarter receives atom row l:
//   A (128 rows):      column 4 kk + c    = A atom kk, word c (the MMA reads
//                      A row r at lane r, column 4 kk + r / 32)
//   B, 256 rows:       column 16 + 8 kk + c     = weight tile 0's atom kk, word c
//                      column 16 + 8 kk + 4 + c = weight tile 1's atom kk, word c
//   B, 128 rows:       column 16 + 4 kk + c     = the weight tile's atom kk, word c
// (the MMA reads B's scales from each quarter's own copy).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Load atoms `src + kk * 512` (kk < 4), row `lane`, into v[4 kk .. 4 kk + 3].
__device__ __forceinline__ void load_atom_rows(uint32_t (&v)[16], const uint8_t* src, int lane) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint4 w = *reinterpret_cast<const uint4*>(src + kk * 512 + lane * 16);
    v[4 * kk] = w.x;
    v[4 * kk + 1] = w.y;
    v[4 * kk + 2] = w.z;
    v[4 * kk + 3] = w.w;
  }
}

template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory"); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory"); }

template <int EPI, bool SMALL_A>
constexpr bool staged_store() { return EPI != EPI_SWIGLU_QUANT && !SMALL_A; }

// 16 bytes to / from shared memory.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

template <int EPI, bool SMALL_A>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_kernel(const GemmArgs p) {
  using SM = Smem<SMALL_A, staged_store<EPI, SMALL_A>()>;
  constexpr int STAGES = SM::STAGES;
  constexpr int ST_A = SM::ST_A, ST_ASF = SM::ST_ASF, ST_B = SM::ST_B, ST_BSF = SM::ST_BSF;
  constexpr int STAGE_BYTES = SM::STAGE_BYTES, OFF_GRP = SM::OFF_GRP;
  constexpr int OFF_BAR = SM::OFF_BAR, OFF_MISC = SM::OFF_MISC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bar0 = s_base + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto sfready_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  const uint32_t accf_bar = bar0 + 8u * (3 * STAGES);
  const uint32_t acce_bar = accf_bar + 8u;
  const uint32_t drain_mma_bar = accf_bar + 16u;
  auto stage_addr = [&](int s) { return s_base + static_cast<uint32_t>(s * STAGE_BYTES); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfready_bar(s), SF_WARPS);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, EPI_WARPS);
    mbar_init(drain_mma_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int ntiles = p.N / BM;             // 128-row weight tiles per expert
  const int k64 = p.K >> 6;
  const int nkt = (k64 + 3) >> 2;
  if (p.early_weights && threadIdx.x == 0) {
    // The previous kernel (which produces A) may still be running: start pulling
    // this CTA's first weight tile into L2 meanwhile.  The group tables read here
    // come from the routing kernel two launches back, not from the kernel this
    // one depends on: they are complete because that kernel (the gate_up GEMM)
    // executed its own dependency wait on the routing kernel before it allowed
    // this launch to begin.  The expert and weight tile are clamped to the
    // weight buffer all the same, so a prefetch can never leave it.
    const Sched sc0 = make_sched(p);
    if (static_cast<int>(blockIdx.x) < sc0.total) {
      const Tile x = decode_tile(blockIdx.x, p, sc0);
      const int g = min(max(x.g, 0), p.G - 1);
      const int nt0 = min(max(x.nt0, 0), ntiles - (x.wide ? 2 : 1));
      // the tile's weight units, all K tiles: one contiguous range of the pair
      const int pair = nt0 >> 1;
      const uint8_t* bc = p.b + (static_cast<size_t>(g) * ntiles + 2 * pair) * nkt * TILE_BYTES;
      bulk_prefetch_l2(bc, static_cast<uint32_t>((2 * pair + 1 < ntiles ? 2 : 1) * nkt) * TILE_BYTES);
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  Groups gr{};
  if (p.G + 1 <= SMEM_GROUPS) {
    int* st = reinterpret_cast<int*>(smem + OFF_GRP);
    for (int j = threadIdx.x; j <= p.G; j += blockDim.x) {
      st[j] = __ldg(p.tile_offs + j);
      st[SMEM_GROUPS + j] = __ldg(p.offsets + j);
    }
    __syncthreads();
    gr.toff = st;
    gr.off = st + SMEM_GROUPS;
  }
  const Sched sc = make_sched(p);
  const int total = sc.total;

  // Roles by warpgroup; each warpgroup first takes its share of the register
  // file (every thread of the warpgroup executes the same setmaxnreg).
  const int wg = warp >> 2;
  if (wg == 3) {
    regs_dec<REG_CTRL>();
    if (warp == PRODUCER_WARP) {
      if (lane == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t ph = 0;
        uint32_t pending = 0, pend_par = 0;  // per stage: load issued, parity of that phase
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
          const Tile x = decode_tile(t, p, sc, gr);
          const uint8_t* a_chunk = p.a + static_cast<size_t>(x.mt) * nkt * TILE_BYTES;
          // Weights (TILED, groups of N rows): a 256-column tile reads one
          // 36864-byte unit per K tile, [codes of both 128-row halves][their
          // atoms], straight into the stage's [B codes][B atoms]; a 128-column
          // tile reads its half's codes and atoms with two copies.
          const int pair = x.nt0 >> 1, half = x.nt0 & 1;
          const bool paired = 2 * pair + 1 < ntiles;
          const uint8_t* b_pair = p.b + (static_cast<size_t>(x.g) * ntiles + 2 * pair) * nkt * TILE_BYTES;
          const size_t b_unit = static_cast<size_t>(paired ? 2 : 1) * TILE_BYTES;
          const size_t b_codes = paired ? static_cast<size_t>(half) * TILE_CODE_BYTES : 0;
          const size_t b_atoms = paired ? 2 * TILE_CODE_BYTES + static_cast<size_t>(half) * TILE_SF_BYTES : TILE_CODE_BYTES;
          // rows of A to fetch: the valid ones, rounded up to the 8-row swizzle group
          int a_rows = x.rows;
          if (a_rows > SM::A_ROWS) {  // the caller promised at most 32 rows per group
            report_error(p.err, DEV_BAD_OFFSETS, t);
            a_rows = SM::A_ROWS;
          }
          const uint32_t a_code_bytes = static_cast<uint32_t>((a_rows + 7) & ~7) * 128u;
          const bool a_whole = !SMALL_A && a_rows == BM;    // codes and atoms in one copy
          const uint32_t stage_tx = a_code_bytes + TILE_SF_BYTES + (x.wide ? 2 : 1) * TILE_BYTES;
          for (int kt = 0; kt < nkt; ++kt) {
            if (!mbar_wait(empty_bar(stage), ph ^ 1u, abort_flag, p.err, DEV_TIMEOUT_PRODUCER, t)) {
              ok = false;
              break;
            }
            const uint32_t st = stage_addr(stage);
            const uint32_t fb = full_bar(stage);
            const uint8_t* ac = a_chunk + static_cast<size_t>(kt) * TILE_BYTES;
            const uint8_t* bu = b_pair + kt * b_unit;
            mbar_arrive_expect_tx(fb, stage_tx);
            if (a_whole) {
              bulk_load(st + ST_A, ac, TILE_BYTES, fb);        // ST_ASF follows ST_A's 16 KB
            } else {
              bulk_load(st + ST_A, ac, a_code_bytes, fb);
              bulk_load(st + ST_ASF, ac + TILE_CODE_BYTES, TILE_SF_BYTES, fb);
            }
            if (x.wide) {
              bulk_load(st + ST_B, bu, 2 * TILE_BYTES, fb);    // ST_BSF follows ST_B's 32 KB
            } else {
              bulk_load(st + ST_B, bu + b_codes, TILE_CODE_BYTES, fb);
              bulk_load(st + ST_BSF, bu + b_atoms, TILE_SF_BYTES, fb);
            }
            pending |= 1u << stage;
            pend_par = (pend_par & ~(1u << stage)) | (ph << stage);
            if (++stage == STAGES) {
              stage = 0;
              ph ^= 1u;
            }
          }
        }
        if (!ok || *abort_flag) {
          // Let every copy this thread issued land before the CTA goes away.
          for (int s = 0; s < STAGES; ++s)
            if ((pending >> s) & 1u) mbar_wait_drain(full_bar(s), (pend_par >> s) & 1u, p.err, s);
        }
      }
    } else if (warp == MMA_WARP) {
      if (lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int i = 0;  // K tiles consumed so far (ring position)
        int tile_i = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tile_i) {
          const Tile x = decode_tile(t, p, sc, gr);
          const uint32_t idesc = mxf4nvf4_idesc(BM, x.wide ? 256 : 128);
          for (int kt = 0; kt < nkt; ++kt, ++i) {
            const int s = i % STAGES;
            // Stage landed and its scales are in TMEM slot s (written after the
            // MMAs of K tile i - STAGES, which last read the slot, completed).
            if (!mbar_wait(full_bar(s), (i / STAGES) & 1, abort_flag, p.err, DEV_TIMEOUT_MMA, t) ||
                !mbar_wait(sfready_bar(s), (i / STAGES) & 1, abort_flag, p.err, DEV_TIMEOUT_MMA, t)) {
              ok = false;
              break;
            }
            if (kt == 0) {
              // the epilogue has moved the previous tile out of TMEM
              if (!mbar_wait(acce_bar, (tile_i & 1) ^ 1u, abort_flag, p.err, DEV_TIMEOUT_MMA, t)) {
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const int na = min(4, k64 - kt * 4);
            const uint32_t st = stage_addr(s);
            const uint32_t sf = tmem + SF_COL0 + s * SF_SLOT_COLS;
            // Descriptors once per K tile: K step kk starts 32 bytes further into
            // the swizzled rows (start address field + 2).  The issuing thread
            // shares its scheduler with busy epilogue warps, so the fewer
            // instructions between the MMAs the better.
            const uint64_t da = operand_desc_sw128(st + ST_A), db = operand_desc_sw128(st + ST_B);
            const uint32_t sfb_step = x.wide ? 8u : 4u;
            if (na == 4) {
              tc_mma_nvfp4(tmem, da, db, idesc, sf, sf + 16, kt != 0 ? 1u : 0u);
              tc_mma_nvfp4(tmem, da + 2, db + 2, idesc, sf + 4, sf + 16 + sfb_step, 1u);
              tc_mma_nvfp4(tmem, da + 4, db + 4, idesc, sf + 8, sf + 16 + 2 * sfb_step, 1u);
              tc_mma_nvfp4(tmem, da + 6, db + 6, idesc, sf + 12, sf + 16 + 3 * sfb_step, 1u);
            } else {
              for (int kk = 0; kk < na; ++kk)
                tc_mma_nvfp4(tmem, da + 2 * kk, db + 2 * kk, idesc, sf + kk * 4, sf + 16 + kk * sfb_step,
                             (kt | kk) != 0 ? 1u : 0u);
            }
            tc_commit(empty_bar(s));
          }
          if (ok) tc_commit(accf_bar);
        }
        // Every MMA this thread issued must finish before TMEM is freed.
        tc_commit(drain_mma_bar);
        mbar_wait_drain(drain_mma_bar, 0, p.err, -1);
      }
    }  // warps 14-15 have no role
  } else if (wg == 0) {
    regs_dec<REG_SF>();
    // -------------------------------------------------------------- scale writers
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;  // this warp's TMEM lane quarter
    int i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile x = decode_tile(t, p, sc, gr);
      for (int kt = 0; kt < nkt; ++kt, ++i) {
        const int s = i % STAGES;
        // The stage landed (atoms arrive with the codes).  The MMAs of K tile i - STAGES, the last to
        // read TMEM slot s, completed before the producer refilled the stage.
        // Every lane waits (and acquires); the warp leaves together if any lane gave up.
        const bool got = mbar_wait(full_bar(s), (i / STAGES) & 1, abort_flag, p.err, DEV_TIMEOUT_PRODUCER, t);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + s * STAGE_BYTES;
        const uint32_t col = tmem + lanes + SF_COL0 + s * SF_SLOT_COLS;
        uint32_t v[16];
        load_atom_rows(v, st + ST_ASF, lane);
        tmem_st16(col, v);
        if (x.wide) {
          // 8 columns per K step: tile 0's atom row, then tile 1's
          uint32_t w[16];
          load_atom_rows(v, st + ST_BSF, lane);
          load_atom_rows(w, st + ST_BSF + TILE_SF_BYTES, lane);
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              lo[8 * kk + c] = v[4 * kk + c];
              lo[8 * kk + 4 + c] = w[4 * kk + c];
              hi[8 * kk + c] = v[4 * (kk + 2) + c];
              hi[8 * kk + 4 + c] = w[4 * (kk + 2) + c];
            }
          tmem_st16(col + 16, lo);
          tmem_st16(col + 32, hi);
        } else {
          load_atom_rows(v, st + ST_BSF, lane);
          tmem_st16(col + 16, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfready_bar(s));
      }
    }
  } else {
    regs_inc<REG_EPI>();
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = (warp - EPI_WARP0) >> 2;  // which 128 of the tile's 256 columns
    const int r = q * 32 + lane;            // tile row handled by this thread
    int tile_i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tile_i) {
      const Tile x = decode_tile(t, p, sc, gr);
      const bool active = q * 32 < x.rows && (half == 0 || x.wide);
      // per-tile constants, fetched while the tile's MMAs run
      const float alpha = active ? __fmul_rn(__ldg(p.gs_a + x.g), __ldg(p.gs_b + x.g)) : 0.0f;
      float gsq = 0.0f;
      if constexpr (EPI == EPI_SWIGLU_QUANT) gsq = active ? __ldg(p.gs_q + x.g) : 0.0f;
      if (!mbar_wait(accf_bar, tile_i & 1, abort_flag, p.err, DEV_TIMEOUT_EPILOGUE, t)) break;
      tc_fence_after();
      const uint32_t tb = tmem + half * 128 + (static_cast<uint32_t>(q * 32) << 16);
      const bool valid = r < x.rows;
      const int64_t row = static_cast<int64_t>(x.row0) + r;
      const int nt = x.nt0 + half;          // 128-column weight tile of this warp
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar);  // accumulator is in registers: release it
      };
      // The whole 128-column slice of the accumulator moves to registers (128
      // values a thread: the epilogue warpgroups run with REG_EPI registers) and
      // the accumulator is released before any arithmetic, so the next tile's
      // MMAs run while this tile is scaled, quantized and stored.
      uint32_t v[4][32];
      if (active) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tb + c * 32, v[c]);
        tmem_ld_wait();
      }
      release();
      if (!active) continue;
      if constexpr (EPI == EPI_SWIGLU_QUANT) {
        // Prepared w13 rows: in every 32-column chunk c of weight tile nt, the
        // first 16 columns are gate rows and the last 16 the matching up rows
        // of intermediate indices nt * 64 + 16 c .. + 15.
        const int I = p.N >> 1;
        const float six_gsq = __fmul_rn(6.0f, gsq);
        uint32_t cw[8];
        uint32_t sfw = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float h[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // rows past the group's end carry whatever their scale bytes held: use zeros
            const float g = valid ? __fmul_rn(__uint_as_float(v[c][j]), alpha) : 0.0f;
            const float u = valid ? __fmul_rn(__uint_as_float(v[c][16 + j]), alpha) : 0.0f;
            h[j] = __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u);
          }
          if (p.h_dump != nullptr && valid) {
            float4* hd = reinterpret_cast<float4*>(p.h_dump + row * I + nt * 64 + c * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) hd[j] = make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
          }
          sfw |= quant_block16(h, gsq, six_gsq, cw[2 * c], cw[2 * c + 1]) << (8 * c);
        }
        // A2 is the down GEMM's A operand (TILED_GROUPED, K = I): weight tile
        // nt's 64 h values are MMA step nt % 4 of K tile nt / 4: 32 code bytes
        // and 4 scale bytes of row r.
        uint8_t* chunk = p.q_codes + (static_cast<size_t>(x.mt) * num_k_tiles(I) + (nt >> 2)) * TILE_BYTES;
        if (valid) {
          *reinterpret_cast<uint4*>(chunk + tiled_code_offset(r, (nt & 3) * 32)) =
              make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint4*>(chunk + tiled_code_offset(r, (nt & 3) * 32 + 16)) =
              make_uint4(cw[4], cw[5], cw[6], cw[7]);
        }
        *reinterpret_cast<uint32_t*>(chunk + TILE_CODE_BYTES + (nt & 3) * 512 + sf_atom_offset(r, 0)) = sfw;
      } else if constexpr (staged_store<EPI, SMALL_A>()) {
        // Each 128-byte column chunk of the warp's 32 rows goes through its 4 KB
        // of shared memory: lane l writes its row's eight 16-byte pieces (piece j
        // at l * 128 + ((j ^ (l % 8)) * 16), so that the writes and the reads
        // below hit distinct banks), then each store instruction writes four
        // whole rows' 128 bytes: lane l takes piece l % 8 of row 4 i + l / 8.
        constexpr bool F32 = EPI == EPI_STORE_F32;
        constexpr int CHUNK_COLS = F32 ? 32 : 64;             // 128 bytes of a row
        const uint32_t stg = s_base + SM::OFF_STG + static_cast<uint32_t>((warp - EPI_WARP0) * SM::STG_WARP_BYTES);
        const int rows_here = min(32, x.rows - q * 32);       // valid rows of this warp's quarter
        // with a row map, lane l holds the output row of the quarter's row l
        const int32_t out_row = p.d_rows != nullptr && lane < rows_here
                                    ? __ldg(p.d_rows + x.row0 + q * 32 + lane) : 0;
#pragma unroll
        for (int ch = 0; ch < 128 / CHUNK_COLS; ++ch) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t w[4];
            if constexpr (F32) {
              const int c = ch, e0 = 4 * j;                     // columns 32 ch + 4 j .. + 3
#pragma unroll
              for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(__fmul_rn(__uint_as_float(v[c][e0 + e]), alpha));
            } else {
              const int c = 2 * ch + (j >> 2), e0 = 8 * (j & 3);  // columns 64 ch + 8 j .. + 7
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[c][e0 + 2 * e]), alpha),
                                                         __fmul_rn(__uint_as_float(v[c][e0 + 2 * e + 1]), alpha));
                w[e] = *reinterpret_cast<uint32_t*>(&b);
              }
            }
            st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) * 16), w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
          const int pc = lane & 7;
          // this lane's 16-byte piece of the chunk; rows 4 i + lane / 8 of the quarter
          constexpr int ESZ = F32 ? 4 : 2;
          const int64_t pitch = p.ldd * ESZ;
          uint8_t* dst = static_cast<uint8_t*>(p.d) + (static_cast<int64_t>(nt) * 128 + ch * CHUNK_COLS) * ESZ + pc * 16;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);                 // row within the warp's quarter
            const uint4 d = ld_shared_v4(stg + rr * 128 + ((pc ^ (rr & 7)) * 16));
            // output row: the grouped row itself, or where the row map sends it
            const int64_t orow = p.d_rows == nullptr ? static_cast<int64_t>(x.row0) + q * 32 + rr
                                                     : static_cast<int64_t>(__shfl_sync(0xffffffffu, out_row, rr));
            if (rr < rows_here) *reinterpret_cast<uint4*>(dst + orow * pitch) = d;
          }
          __syncwarp();
        }
      } else {
        if (!valid) continue;
        const int64_t orow = p.d_rows == nullptr ? row : static_cast<int64_t>(__ldg(p.d_rows + row));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t col = static_cast<int64_t>(nt) * 128 + c * 32;
          if constexpr (EPI == EPI_STORE_F32) {
            float* drow = static_cast<float*>(p.d) + orow * p.ldd + col;
            if (p.d_align32) {
              // whole 32-byte sectors per instruction
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(__fmul_rn(__uint_as_float(v[c][8 * j + e]), alpha));
                st_global_v8(drow + 8 * j, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(drow);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(__fmul_rn(__uint_as_float(v[c][4 * j]), alpha),
                                     __fmul_rn(__uint_as_float(v[c][4 * j + 1]), alpha),
                                     __fmul_rn(__uint_as_float(v[c][4 * j + 2]), alpha),
                                     __fmul_rn(__uint_as_float(v[c][4 * j + 3]), alpha));
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.d) + orow * p.ldd + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int h2 = 0; h2 < 4; ++h2) {
                __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[c][8 * j + 2 * h2]), alpha),
                                                         __fmul_rn(__uint_as_float(v[c][8 * j + 2 * h2 + 1]), alpha));
                w[h2] = *reinterpret_cast<uint32_t*>(&b);
              }
              dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

template <int EPI, bool SMALL_A>
cudaError_t launch_layout(const GemmArgs& a, int grid, cudaStream_t s, const char** why) {
  auto k = grouped_gemm_kernel<EPI, SMALL_A>;
  constexpr int bytes = Smem<SMALL_A, staged_store<EPI, SMALL_A>()>::BYTES;
  // The register split assumes the block is launched with REG_LAUNCH registers a
  // thread; with fewer, the epilogue's setmaxnreg.inc could never be granted.
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, k);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * THREADS < (REG_SF + REG_CTRL + 2 * REG_EPI) * 128 || fa.numRegs > REG_LAUNCH) {
    *why = "the GEMM kernel was compiled with a register count its register split does not fit";
    return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  prefer_max_shared(reinterpret_cast<const void*>(k));
  return launch_kernel(k, dim3(grid), dim3(THREADS), bytes, s, a.pdl, a);
}

template <int EPI>
cudaError_t launch_epi(const GemmArgs& a, int grid, cudaStream_t s, const char** why) {
  return a.small_a ? launch_layout<EPI, true>(a, grid, s, why) : launch_layout<EPI, false>(a, grid, s, why);
}

}  // namespace

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s, const char** why) {
  *why = nullptr;
  if (a.a_rows <= 0) return cudaSuccess;
  const int64_t max_tiles = ((a.a_rows + BM - 1) / BM + a.G) * ((a.N + BN - 1) / BN);
  int grid = a.max_ctas > 0 ? a.max_ctas : sm_count();
  if (grid > max_tiles) grid = static_cast<int>(max_tiles);
  if (grid < 1) grid = 1;
  switch (a.epilogue) {
    case EPI_STORE_F32: return launch_epi<EPI_STORE_F32>(a, grid, s, why);
    case EPI_STORE_BF16: return launch_epi<EPI_STORE_BF16>(a, grid, s, why);
    case EPI_SWIGLU_QUANT: return launch_epi<EPI_SWIGLU_QUANT>(a, grid, s, why);
    default: *why = "unknown epilogue"; return cudaErrorInvalidValue;
  }
}

}  // namespace nvf
