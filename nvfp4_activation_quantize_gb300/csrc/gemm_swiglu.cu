// gemm_swiglu.cu -- the FFN-up projection as a block-scaled NVFP4 GEMM on the
// fifth-generation tensor cores, with the SwiGLU and the NVFP4 quantize of its
// output fused into the epilogue.
//
// (FastVideo compare "fasth3-spark-exact-perf", minimax_h3_swiglu_gemm.cu:
// launch_gemm_swiglu takes NVFP4 A [m, k] and B [n, k] with value/gate-paired
// columns, alpha and the output's global scale as device pointers;
// h3_epilogue::Store forms value = bf16(alpha * acc[2j]) and gate =
// bf16(alpha * acc[2j + 1]), the SwiGLU, and the block quantize with the
// swizzled scale store.  That kernel is a CUTLASS SM120 collective; this one is
// written for sm_103a directly.)
//
// Work: persistent CTAs, one per SM, in clusters of two on neighbouring 128-row
// tiles of A that share one 256-row tile of B (128 outputs): each CTA loads half
// of B's tile and of its scales with a cluster multicast into both CTAs'
// shared memory, so a CTA moves a third fewer bytes from L2 than alone.  Units
// go in a grouped order (32 row-tile pairs sweep all of B's column tiles), so a
// group's A stays in L2 while B streams.
// Warp roles inside a CTA of 14 warps:
//   warp 12, one lane  TMA producer: per 256-element k stage, a 2-D tensor copy
//                      of A (128 rows x 128 bytes) and of B (256 x 128), 128-byte
//                      swizzle, and 1-D bulk copies of the stage's 128x4 scale
//                      atoms, all completing on the stage's mbarrier; three
//                      stages.
//   warps 0..3         (warp 1 also allocates the 512 TMEM columns) write each
//                      stage's scale atoms into the stage's TMEM scale slot with
//                      tcgen05.st -- each thread its own TMEM lane, the layout
//                      tcgen05.cp .32x128b.warpx4 would write, but without
//                      occupying the tensor pipe, where those copies took as
//                      long as the MMAs -- and signal the stage ready.
//   warp 13, one lane  issues four tcgen05.mma per stage (kind::mxf4nvf4,
//                      block_scale, 16-element blocks, M = 128, N = 256, K = 64)
//                      accumulating in TMEM columns 0..255, and tcgen05.commit
//                      to free the stage; after the last stage a commit tells
//                      the epilogue the accumulator is complete.
//   warps 4..11        the epilogue: warp w reads TMEM lane quarter w % 4 (one
//                      accumulator row per thread) and half of the tile's
//                      columns, forms the bf16 value and gate pairs in registers
//                      and hands the accumulator back (the next tile's MMAs
//                      start); then per 16 outputs y by the SiLU table (or
//                      directly) and the NVFP4 block of y: 8 code bytes and one
//                      scale byte, all in the thread's own registers.
// Every wait is bounded: a wait that runs out sets a device flag, tells the
// other roles to stop, and the CTA drains what it has in flight, frees its TMEM
// and returns (h3q_kernel_error_flag reads and clears the flag).
#include <cuda.h>  // CUtensorMap; the encode function is fetched at run time

#include <mutex>

#include "h3q_async.cuh"
#include "h3q_device.cuh"
#include "h3q_internal.h"
#include "h3q_silu.cuh"

namespace h3q {
namespace {

constexpr int kTileM = 128;                       // acc rows per tile (the MMA's M)
constexpr int kTileN = 256;                       // acc columns per tile (the MMA's N)
constexpr int kStageK = 256;                      // K elements per pipeline stage (128 bytes a row)
constexpr int kKSteps = kStageK / 64;             // tcgen05.mma per stage (K = 64 each)
constexpr int kStages = 4;
constexpr int kThreads = 448;                     // 14 warps
constexpr int kSfThreads = 128;                   // warps 0..3: the scale fill
constexpr int kEpiWarp0 = 4;                      // first epilogue warp
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kEpiThreads = 256;
constexpr int kCluster = 2;                       // CTAs per cluster, on neighbouring row tiles
constexpr int kGroupPairs = 32;                   // row-tile pairs of A per raster group

constexpr int kABytes = kTileM * kStageK / 2;     // 16 KB
constexpr int kBBytes = kTileN * kStageK / 2;     // 32 KB
constexpr int kSfaBytes = kKSteps * 512;          // one 128x4 atom per K = 64 step
constexpr int kSfbBytes = 2 * kKSteps * 512;      // two row tiles of B x one atom per step
constexpr uint32_t kStageTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;

// TMEM columns: the fp32 accumulator at 0..255, then one scale slot per stage:
// A's scales of the stage's K = 64 steps (4 columns each) and B's (8 each).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfSlot0 = 256;
constexpr uint32_t kSfSlotCols = 12 * kKSteps;
static_assert(kSfSlot0 + kStages * kSfSlotCols <= kTmemCols, "TMEM columns");

// Shared memory carve-up (offsets from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSfa = kOffB + kStages * kBBytes;
constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr int kOffInv = kOffSfb + kStages * kSfbBytes;
constexpr int kOffBar = kOffInv + 128 * 4;
constexpr int kBars = 3 * kStages + 3;            // full[], empty[], sf_ready[], acc_full, acc_empty, drain
constexpr int kOffMisc = kOffBar + kBars * 8;     // TMEM base address, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4: A and B E2M1 (format
// 1 at bits 7-9 and 10-12), both K-major (bits 15, 16 clear), N >> 3 at bits
// 17-22, scale type UE4M3 (bit 23 clear), M >> 4 at bits 24-28, scale factor
// ids 0 (bits 4-5, 29-30), dense K = 64 (bit 31 clear).
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (uint32_t(kTileN >> 3) << 17) |
                            (uint32_t(kTileM >> 4) << 24);


// Set when a bounded wait ran out (read and cleared by h3q_kernel_error_flag).
__device__ int g_gemm_fault;

struct GemmArgs {
  const uint8_t* sfa;    // A's scales, 128x4 layout [pad128(m), k/16]
  const uint8_t* sfb;    // B's scales, 128x4 layout [n, k/16]
  int64_t m, n, k;
  const float* alpha;
  const float* gsf;
  uint8_t* codes;        // [m, n/4]
  uint8_t* scales;       // [pad128(m), n/32], 128x4 layout
  uint16_t* y;           // optional bf16 [m, n/2]
  float* acc;            // optional fp32 [m, n]
  const float* silu;     // the SiLU table (g_silu_table), filled on the stream before the launch
};

// s = fl(g * sigma(g)) of every bf16 gate in the SiLU table's window (h3q_silu.cuh),
// 32 KB: shared memory is taken by the operand stages, so the table lives here
// (read through L1) and silu_table_kernel writes it before each GEMM launch on
// the same stream -- the same values every time.
__device__ __align__(16) float g_silu_table[2 * kTabHalf];

__global__ void __launch_bounds__(1024) silu_table_kernel(float* table) { fill_silu_table(table); }

// --- PTX wrappers ---------------------------------------------------------------

// Wait for the phase of parity `parity` of the barrier to complete.  Gives up
// (false) when another role has raised the abort flag, or after kWaitNs, which
// raises it and the device fault flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;  // the common case, without reading the timer
  const uint64_t start = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (now_ns() - start > kWaitNs) break;
    }
  }
  *abort = 1;
  atomicExch(&g_gemm_fault, 1);
  return false;
}

// The same wait with no abort flag (the drain after an abort), bounded the same way.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) { (void)wait_bounded(bar, parity); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The same copy delivered to every CTA of the cluster (same shared-memory offset
// and the same barrier offset in each).
constexpr uint16_t kClusterMask = (1u << kCluster) - 1;

__device__ __forceinline__ void tma_load_2d_all(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(kClusterMask)
      : "memory");
}

__device__ __forceinline__ void bulk_load_all(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "h"(kClusterMask)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}


__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared memory matrix descriptor: start address, leading and stride byte
// offsets (all >> 4), the descriptor version 1 at bits 46-47, the layout at
// bits 61-63 (0 none, 2 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  return static_cast<uint64_t>((addr >> 4) & 0x3fffu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(layout) << 61);
}

// A or B stage operand: K-major rows of 128 bytes, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr) { return smem_desc(addr, 16, 1024, 2); }

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::
          "r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Arrives on the barrier at this offset in every CTA of the cluster once the
// issued tcgen05 operations have completed.
__device__ __forceinline__ void tc_commit_all(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(kClusterMask)
      : "memory");
}

// 32 consecutive fp32 columns of this warp's TMEM lane quarter, one row per thread.
__device__ __forceinline__ void tc_load32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_load() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 and 32 consecutive 32-bit columns of this warp's TMEM lane quarter, one
// lane per thread (the thread's own row).
__device__ __forceinline__ void tc_store16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tc_store32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tc_wait_store() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// --- tile order ---------------------------------------------------------------------

// Unit u of the grouped order: a pair of neighbouring row tiles of A (one per
// CTA of the cluster) and one column tile of B.  Groups of kGroupPairs pairs;
// inside a group the pair varies fastest, so clusters working at the same time
// share B's tile and the group's A stays in L2 while B's column tiles go by.
__device__ __forceinline__ void unit_of(int64_t u, int64_t pairs, int64_t tiles_n, int64_t& mp, int64_t& nt) {
  const int64_t per_group = int64_t{kGroupPairs} * tiles_n;
  const int64_t group = u / per_group;
  const int64_t rest = u - group * per_group;
  const int64_t first = group * kGroupPairs;
  const int64_t rows = pairs - first < kGroupPairs ? pairs - first : kGroupPairs;
  mp = first + rest % rows;
  nt = rest / rows;
}

// --- the kernel ---------------------------------------------------------------------

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
gemm_swiglu_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  const uint32_t base = smem_u32(smem);
  const uint32_t bar_full = base + kOffBar;                 // + 8 * stage
  const uint32_t bar_empty = bar_full + 8 * kStages;        // + 8 * stage
  const uint32_t bar_sf = bar_empty + 8 * kStages;          // + 8 * stage
  const uint32_t bar_acc_full = bar_sf + 8 * kStages;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  const uint32_t bar_drain = bar_acc_empty + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  float* inv_table = reinterpret_cast<float*>(smem + kOffInv);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work: units of (row-tile pair, column tile); this CTA takes row tile
  // 2 * pair + rank of each unit of its cluster.  With an odd number of row
  // tiles the last pair's second tile lies past the matrix: its A reads as zero
  // and its outputs are not stored.
  const uint32_t rank = cluster_rank();
  const int64_t cluster = blockIdx.x / kCluster;
  const int64_t clusters = gridDim.x / kCluster;
  const int64_t tiles_m = (args.m + kTileM - 1) / kTileM;
  const int64_t pairs = (tiles_m + kCluster - 1) / kCluster;
  const int64_t tiles_n = args.n / kTileN;
  const int64_t units = pairs * tiles_n;
  const int stages_k = static_cast<int>(args.k / kStageK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kCluster);  // both CTAs' MMAs must be done with the stage
      mbar_init(bar_sf + 8 * s, kSfThreads);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, kEpiThreads);
    mbar_init(bar_drain, 1);
    *abort = 0;
    mbar_init_fence();
  }
  if (warp == 1) {  // the whole warp allocates the CTA's TMEM (one CTA per SM)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const float gsf = *args.gsf;
  fill_inverse_scales(inv_table, gsf);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the partner's barriers are initialised before any copy lands in them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ---- TMA producer (one lane; the others wait at the __syncwarp below so the
    // warp reaches the final, aligned barrier converged)
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
      const int64_t atoms_k = args.k / 64;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per stage: ever issued, parity of the last issue
      bool ok = true;
      for (int64_t u = cluster; u < units && ok; u += clusters) {
        int64_t mp, nt;
        unit_of(u, pairs, tiles_n, mp, nt);
        const int64_t mt = mp * kCluster + rank;
        const int64_t mt_sf = mt < tiles_m ? mt : tiles_m - 1;  // a phantom tile reads real scales
        const uint8_t* sfa = args.sfa + mt_sf * atoms_k * 512;
        // this CTA's share of B: rows 128 * rank .. of the column tile, and their scales
        const uint8_t* sfb = args.sfb + (nt * 2 + rank) * atoms_k * 512;
        for (int kt = 0; kt < stages_k; ++kt) {
          if (!(ok = mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort))) break;
          const uint32_t full = bar_full + 8 * stage;
          constexpr uint32_t kSfChunk = kKSteps * 512;  // one row tile's atoms of the stage
          mbar_expect_tx(full, kStageTx);
          tma_load_2d(base + kOffA + stage * kABytes, &map_a, kt * (kStageK / 2), static_cast<int>(mt * kTileM),
                      full);
          bulk_load(base + kOffSfa + stage * kSfaBytes, sfa + kt * kSfChunk, kSfChunk, full);
          tma_load_2d_all(base + kOffB + stage * kBBytes + rank * (kBBytes / kCluster), &map_b, kt * (kStageK / 2),
                          static_cast<int>(nt * kTileN + rank * (kTileN / kCluster)), full);
          bulk_load_all(base + kOffSfb + stage * kSfbBytes + rank * kSfChunk, sfb + kt * kSfChunk, kSfChunk, full);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Before the cluster may exit: every stage's last use must be released by
      // both CTAs' MMAs (their commits arrive on this CTA's empty barriers), and on
      // an abort every copy issued must have landed (bounded waits).
      for (int s = 0; s < kStages; ++s) {
        if (!(issued & (1u << s))) continue;
        if (!ok) mbar_drain(bar_full + 8 * s, (issued_parity >> s) & 1u);
        mbar_drain(bar_empty + 8 * s, (issued_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (warp < kSfThreads / 32) {
    // ---- scale fill (warps 0..3, one TMEM lane quarter each).  Per stage every
    // thread copies its row (m mod 32) of each of the stage's 12 scale atoms from
    // shared memory into its own TMEM lane with tcgen05.st -- the layout
    // tcgen05.cp .32x128b.warpx4 would write, without taking the tensor pipe --
    // and arrives on the stage's sf_ready barrier.  It runs up to kStages stages
    // ahead of the MMAs: a stage's slot is rewritten only after its full barrier
    // completes again, which needs the MMAs that read the slot to have finished.
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t u = cluster; u < units; u += clusters) {
      bool ok = true;
      for (int kt = 0; kt < stages_k; ++kt) {
        // one decision per warp (tcgen05.st is warp-aligned)
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * stage, phase, abort)))) break;
        tc_fence_after();
        const uint32_t slot = kSfSlot0 + kSfSlotCols * stage;
        const uint8_t* sfa = smem + kOffSfa + stage * kSfaBytes + 16 * lane;
        const uint8_t* sfb = smem + kOffSfb + stage * kSfbBytes + 16 * lane;
        uint32_t va[16], vb[32];
#pragma unroll
        for (int j = 0; j < kKSteps; ++j) {
          const uint4 x = *reinterpret_cast<const uint4*>(sfa + 512 * j);
          const uint4 y0 = *reinterpret_cast<const uint4*>(sfb + 512 * j);                 // B rows 0..127
          const uint4 y1 = *reinterpret_cast<const uint4*>(sfb + kKSteps * 512 + 512 * j);  // rows 128..255
          va[4 * j] = x.x; va[4 * j + 1] = x.y; va[4 * j + 2] = x.z; va[4 * j + 3] = x.w;
          vb[8 * j] = y0.x; vb[8 * j + 1] = y0.y; vb[8 * j + 2] = y0.z; vb[8 * j + 3] = y0.w;
          vb[8 * j + 4] = y1.x; vb[8 * j + 5] = y1.y; vb[8 * j + 6] = y1.z; vb[8 * j + 7] = y1.w;
        }
        // slot: A's scales of step j at columns 4j, B's at 4 * kKSteps + 8j (its
        // rows 0..127 in the first four columns, 128..255 in the next four)
        tc_store16(lane_base + slot, va);
        tc_store32(lane_base + slot + 4 * kKSteps, vb);
        tc_wait_store();
        tc_fence_before();
        mbar_arrive(bar_sf + 8 * stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issue (one lane)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t u = cluster; u < units && ok; u += clusters) {
        if (!(ok = mbar_wait(bar_acc_empty, acc_phase ^ 1u, abort))) break;
        tc_fence_after();
        for (int kt = 0; kt < stages_k; ++kt) {
          // the stage's operands are in shared memory once its scales are in TMEM
          if (!(ok = mbar_wait(bar_sf + 8 * stage, phase, abort))) break;
          tc_fence_after();
          const uint32_t slot = tmem + kSfSlot0 + kSfSlotCols * stage;
          const uint32_t a = base + kOffA + stage * kABytes;
          const uint32_t b = base + kOffB + stage * kBBytes;
#pragma unroll
          for (int j = 0; j < kKSteps; ++j)
            tc_mma(tmem, operand_desc(a + 32 * j), operand_desc(b + 32 * j), slot + 4 * j,
                   slot + 4 * kKSteps + 8 * j, (kt > 0 || j > 0) ? 1u : 0u);
          tc_commit_all(bar_empty + 8 * stage);  // both CTAs: this CTA's MMAs are done with the stage
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(bar_acc_full);
        acc_phase ^= 1u;
      }
      // On an abort, let the tcgen05 operations already issued finish before the
      // TMEM is freed (a barrier of its own; bounded).  Otherwise the epilogue's
      // wait for the last tile has already seen them all complete.
      if (!ok) {
        tc_commit(bar_drain);
        mbar_drain(bar_drain, 0);
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ---- epilogue
    const int quarter = warp & 3;
    const int half = (warp - kEpiWarp0) >> 2;
    const int64_t f = args.n / 2;
    const int64_t quads = f / 64;
    const float alpha = *args.alpha;
    const float2 alpha2 = make_float2(alpha, alpha);
    const char* table = reinterpret_cast<const char*>(args.silu);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t acc_phase = 0;
    for (int64_t u = cluster; u < units; u += clusters) {
      // one decision per warp: lanes could see an abort and the barrier at different polls
      if (!__all_sync(0xffffffffu, mbar_wait(bar_acc_full, acc_phase, abort))) break;
      tc_fence_after();
      int64_t mp, nt;
      unit_of(u, pairs, tiles_n, mp, nt);
      const int64_t mt = mp * kCluster + rank;
      const int64_t row = mt * kTileM + quarter * 32 + lane;
      const bool in_rows = row < args.m;
      // Drain: the thread's 128 accumulator columns (four blocks of 16 outputs) as
      // bf16 value and gate pairs in registers, then the accumulator is handed
      // back so the next tile's MMAs run while this one's SwiGLU and quantize do.
      uint32_t uw[4][8], gw[4][8];
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) {
        const int blk = half * 4 + bi;  // 16 outputs = 32 accumulator columns
        uint32_t r[32];
        __syncwarp();  // tcgen05.ld is warp-aligned
        tc_load32(lane_base + 32 * blk, r);
        tc_wait_load();
        if (args.acc != nullptr && in_rows) {
          float* dst = args.acc + row * args.n + nt * kTileN + 32 * blk;
#pragma unroll
          for (int i = 0; i < 32; i += 4) store16(dst + i, make_uint4(r[i], r[i + 1], r[i + 2], r[i + 3]));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // outputs 2i, 2i+1: values in columns 4i, 4i+2, gates in 4i+1, 4i+3
          uw[bi][i] = float2_to_bf16x2(
              mul2(make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 2])), alpha2));
          gw[bi][i] = float2_to_bf16x2(
              mul2(make_float2(__uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 3])), alpha2));
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acc_empty);
      acc_phase ^= 1u;

      uint32_t sf_word = 0;
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) {
        const int blk = half * 4 + bi;
        Block16 ub, gb;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ub.w[i] = uw[bi][i];
          gb.w[i] = gw[bi][i];
        }
        Block16 y;
        uint32_t dw[8];
        if (__all_sync(0xffffffffu, table_words(gb, dw))) {
          swiglu_block_table(dw, ub, y, table);
        } else if (__all_sync(0xffffffffu, block_amax(gb) <= kFastLimit)) {
          swiglu_block<true>(gb, ub, y);
        } else {
          swiglu_block<false>(gb, ub, y);
        }
        const Quantized q = quantize_block<true>(y, gsf, inv_table);
        const int64_t out_col = nt * (kTileN / 2) + 16 * blk;
        if (in_rows) {
          store_codes(args.codes + row * (f / 2) + out_col / 2, q.codes_lo, q.codes_hi);
          if (args.y != nullptr) {
            uint16_t* dst = args.y + row * f + out_col;
            store16(dst, make_uint4(y.w[0], y.w[1], y.w[2], y.w[3]));
            store16(dst + 8, make_uint4(y.w[4], y.w[5], y.w[6], y.w[7]));
          }
          sf_word |= q.sf << (8 * bi);
        }
      }
      // the thread's four blocks are one scale quad; rows past m (padding) get 0
      if (mt < tiles_m)  // a phantom row tile has no scale rows
        store_word(args.scales + scale_word_offset(row, nt * 2 + half, quads), sf_word);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
  cluster_sync();  // no copy or commit of the partner may still be headed for this CTA
}

// --- host side ----------------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult found;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &found) ==
            cudaSuccess &&
        found == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}

// Row-major bytes [rows, row_bytes] loaded in boxes of 128 bytes x box_rows with
// the 128-byte swizzle; rows past the end read as zero.
cudaError_t byte_map(CUtensorMap* map, const void* p, int64_t rows, int64_t row_bytes, uint32_t box_rows) {
  EncodeTiled enc = encode_tiled();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {kStageK / 2, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(p), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Clusters of kCluster CTAs that fit the GPU at once (one CTA per SM), per CUDA
// context; the first query also raises the kernel's shared-memory limit.
cudaError_t resident_clusters(int* clusters) {
  static std::mutex mu;
  static unsigned long long cached_context = 0;
  static int cached = 0;
  unsigned long long context = 0;
  cudaError_t err = current_context_id(&context);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  if (context != cached_context || cached == 0) {
    const void* kernel = reinterpret_cast<const void*>(&gemm_swiglu_kernel);
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};  // the cluster size is the kernel's own (__cluster_dims__)
    cfg.gridDim = dim3(kCluster, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (err != cudaSuccess) return err;
    if (n < 1) return cudaErrorInvalidConfiguration;
    cached = n;
    cached_context = context;
  }
  *clusters = cached;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_swiglu(const uint8_t* a, const uint8_t* sfa, int64_t m, int64_t k, const uint8_t* b,
                               const uint8_t* sfb, int64_t n, const float* alpha, const float* gsf,
                               uint8_t* codes, uint8_t* scales, uint16_t* y, float* acc, cudaStream_t stream) {
  CUtensorMap map_a, map_b;
  cudaError_t err = byte_map(&map_a, a, m, k / 2, kTileM);
  if (err == cudaSuccess) err = byte_map(&map_b, b, n, k / 2, kTileN / kCluster);  // each CTA loads half
  if (err != cudaSuccess) return err;
  const int64_t units = ((m + kTileM - 1) / kTileM + kCluster - 1) / kCluster * (n / kTileN);
  int clusters = 0;
  err = resident_clusters(&clusters);
  if (err != cudaSuccess) return err;
  const int64_t grid = (units < clusters ? units : clusters) * kCluster;
  void* silu = nullptr;
  if ((err = cudaGetSymbolAddress(&silu, g_silu_table)) != cudaSuccess) return err;
  silu_table_kernel<<<1, 1024, 0, stream>>>(static_cast<float*>(silu));
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const GemmArgs args{sfa, sfb, m, n, k, alpha, gsf, codes, scales, y, acc, static_cast<const float*>(silu)};
  gemm_swiglu_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(map_a, map_b, args);
  return cudaGetLastError();
}

cudaError_t gemm_error_flag(int* flag) {
  int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(flag, g_gemm_fault, sizeof(int));
  if (err == cudaSuccess) err = cudaMemcpyToSymbol(g_gemm_fault, &zero, sizeof(int));
  return err;
}

}  // namespace h3q
