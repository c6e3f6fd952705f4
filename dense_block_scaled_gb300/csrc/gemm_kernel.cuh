// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D[m][n] = alpha_eff * sum_k a(m,k) * b(n,k)      (A: M x K, B: N x K, K-major)
//
// FP32 accumulation in tensor memory, BF16 output.  Three operand formats:
//   BF16  : kind::f16
//   MXFP8 : kind::mxf8f6f4.block_scale.scale_vec::1X  (E4M3 values, E8M0 scale / 32 K)
//   NVFP4 : kind::mxf4nvf4.block_scale.scale_vec::4X  (E2M1 values, UE4M3 scale / 16 K)
// named by "ThunderKittens 2.0 GPU Kernel优化" (opening section: BF16/MXFP8/NVFP4
// GEMMs) and recapped in "To Infinity and Beyond: ThunderKittens Now on NVIDIA Vera
// Rubin NVL72!" (section "起点：NVIDIA HGX B200 GEMM").
//
// Structure (one CTA per SM, CG CTAs per cluster share one MMA when CG == 2):
//   warp 0      TMA producer: A, B and scale tiles into a STAGES-deep ring, each
//               stage gated by a full/empty mbarrier pair with explicit phase bits
//               ("异步Tensor Core原理与实战", §3.2).
//   warp 1      MMA issuer (pair leader only when CG == 2): waits for a stage,
//               copies its scales to tensor memory with tcgen05.cp and issues the
//               tcgen05.mma that read them from the same thread, so the copy and
//               the MMA pipeline with no fence or barrier between them ("ThunderKittens
//               2.0", §二 2.1).  No tcgen05.fence::after_thread_sync or
//               fence.proxy.async sits between the stage wait and the MMA: the TMA
//               data reaches the MMA through the complete_tx release / try_wait
//               acquire of the same thread (§一 1.2).
//   warp 2      tensor-memory allocation and release; with cluster launch
//               control, the tile scheduler (try_cancel of clusters not yet run).
//   warp 3      with device-resident group sizes, builds the group table.
//   warps 4-11  epilogue: tcgen05.ld of the accumulator, release of the
//               accumulator buffer, alpha scale, BF16 round-to-nearest-even, TMA
//               store (row-masked stores where a grouped GEMM's group ends).
//
// Tensor memory (512 columns): BF16 either double-buffers a 256-column
// accumulator, so the next tile's MMAs overlap the drain, or runs dual
// accumulate on 256 x 512 pair tiles (two N=256 MMAs per K step share the A
// tile, "ThunderKittens 2.0" §二 2.2); MXFP8 / NVFP4 use one 256-column
// accumulator and a ring of scale regions.  Tiles of odd waves walk K
// backwards (serpentine order) to reuse the operand slices still in L2.
//
// Every wait is bounded: past the limit a role sets the device status word and
// an abort flag, all roles leave their loops, in-flight copies and MMAs are
// drained, tensor memory is freed and the kernel returns.
#pragma once
#include <cuda.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace tkg {

enum : int { FMT_BF16 = 0, FMT_MXFP8 = 1, FMT_NVFP4 = 2 };
enum : uint32_t { DEV_ERR_TIMEOUT = 1u, DEV_ERR_CHECK = 2u };

// Check builds (compiled with TKG_CHECK=1): an invariant that does not hold
// sets DEV_ERR_CHECK in the status word, and the caller skips the access the
// invariant guards (a skipped load ends in a bounded wait that runs out); no
// trap, no assert.  In other builds the check compiles to nothing.
#ifndef TKG_CHECK
#define TKG_CHECK 0
#endif
__device__ __forceinline__ bool invariant(bool ok, unsigned int* status) {
#if TKG_CHECK
  if (!ok) atomicOr(status, DEV_ERR_CHECK);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}

struct GemmParams {
  int m, n, k;
  int num_kstages;           // ceil(K / K-per-stage)
  int tiles_m, tiles_n, num_tiles;
  float alpha;
  const float* ta;           // NVFP4 per-tensor scales (device, may be null)
  const float* tb;
  unsigned int* status;      // device status word (error bits)
  unsigned long long timeout_ns;
  int inject_stall;          // test hook: the MMA role waits on a barrier nothing arrives on
  int raster_group;          // M-blocks per raster band (see tile_coords)
  int wave;                  // tiles per wave (resident clusters); 0: every tile walks K forwards
  uint32_t tx_bytes;         // bytes landing on the (leader's) full barrier per stage; the A and B boxes
                             // may be shorter than the tile (rows past them feed only unstored results)
  uint32_t idesc;            // MMA instruction descriptor (N may be narrower than the tile for narrow B)
  int b_cta_rows;            // B rows each CTA of the pair supplies to one MMA
  // Half-width tiles (plain GEMMs): tiles at or past tail_start are halves of
  // the last original tiles, two per tile (the last partial wave, split so it
  // runs in about half the time); tail_start == num_tiles when there are none.
  int tail_start;
  uint32_t tx_half;          // stage bytes of a half tile
  uint32_t idesc_half;       // its MMA descriptor (N halved; dual accumulate: one of its two MMAs)
  int b_cta_rows_half;       // B rows each CTA supplies to a half tile's MMA
  // Plain GEMMs: the epilogue writes D from registers with 16-byte stores
  // (direct_store != 0; rows and columns masked at m and n) instead of staging
  // 32 x 32 boxes in shared memory for TMA stores.
  int direct_store;
  void* d;                   // D (for direct stores)
  int ldd;                   // its row pitch in elements
};

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<FMT_BF16> {
  static constexpr int kStageK = 64;      // K elements per stage (128 bytes of a row)
  static constexpr int kMmaK = 16;        // K elements per MMA (32 bytes)
  static constexpr int kSfAtoms = 0;      // 512-byte scale atoms per 128 rows per stage
};
template <>
struct FmtTraits<FMT_MXFP8> {
  static constexpr int kStageK = 128;
  static constexpr int kMmaK = 32;
  static constexpr int kSfAtoms = 1;      // 4 blocks of 32 = one atom per stage
};
template <>
struct FmtTraits<FMT_NVFP4> {
  static constexpr int kStageK = 256;
  static constexpr int kMmaK = 64;
  static constexpr int kSfAtoms = 4;      // 16 blocks of 16 = four atoms, one per MMA
};

// The same instruction descriptor with N (bits 17-22, N >> 3) replaced.
__host__ __device__ constexpr uint32_t idesc_with_n(uint32_t idesc, int N) {
  return (idesc & ~(0x3Fu << 17)) | (uint32_t(N >> 3) << 17);
}

// Instruction descriptor, kind::f16: D = F32, A = B = BF16, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
// Instruction descriptor, block-scaled kinds.  fmt: 0 = E4M3 (mxf8f6f4), 1 = E2M1
// (mxf4nvf4); scale: 1 = UE8M0, 0 = UE4M3; sf ids pick the byte of a scale word.
__host__ __device__ constexpr uint32_t idesc_bs(int M, int N, uint32_t fmt, uint32_t scale_e8m0, uint32_t a_sf_id,
                                                uint32_t b_sf_id) {
  return (b_sf_id << 4) | (fmt << 7) | (fmt << 10) | (uint32_t(N >> 3) << 17) | (scale_e8m0 << 23) |
         (uint32_t(M >> 4) << 24) | (a_sf_id << 29);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  return uint64_t((addr >> 4) & 0x3FFF) | (uint64_t(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Scale atom for tcgen05.cp 32x128b: 32 rows of 16 bytes, no swizzle, 8-row groups 128 B apart.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t addr) {
  return uint64_t((addr >> 4) & 0x3FFF) | (uint64_t(128 >> 4) << 32) | (1ull << 46);
}

// Tile order: bands of `group` M-blocks; within a band consecutive tiles step
// through its M-blocks for one N-block, then move to the next N-block, so the
// clusters running together share A rows and B columns in L2, and a band's A
// panels stay in L2 while B streams past (the host sizes the band from the L2
// capacity and the panel size).
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group, int& mb, int& nb) {
  const int group_size = group * tiles_n;
  const int band = t / group_size;
  const int first_m = band * group;
  const int gm = min(tiles_m - first_m, group);
  const int r = t - band * group_size;
  mb = first_m + r % gm;
  nb = r / gm;
}

enum : int { SCHED_STATIC = 0, SCHED_CLC = 1 };

// Grouped GEMM (groups of rows of A, each against its own B): group g owns
// rows [row0[g], row0[g] + rows[g]) of A and D and the N x K matrix g of the
// stacked B.  Its output tiles are tile_start[g] .. tile_start[g + 1] - 1, in
// the same banded order as a plain GEMM of rows[g] x N.  A group's scales
// start on a 128-row block of their own: SFA block sfa_block0[g], SFB block
// g * n_blocks.
constexpr int kMaxGroups = 128;
// static shared memory of the table a launch with device-resident group sizes
// builds (first tile, first row, rows and first SFA block per group, the tile count)
constexpr int kDevGroupTableBytes = (4 * kMaxGroups + 2) * 4 + 16;
struct GroupTable {
  int count;
  int n_blocks;                       // 128-row scale blocks per group of B
  int ldd;                            // D row pitch (elements)
  void* d;                            // D, for the row-masked stores at group ends
  const float* tb;                    // NVFP4: per-group tensor scales of B (or null)
  int tile_start[kMaxGroups + 1];
  int row0[kMaxGroups];
  int rows[kMaxGroups];
  int sfa_block0[kMaxGroups];
};
// Grouped GEMM with the group sizes in device memory (written by an earlier
// kernel, e.g. a router): the kernel builds the table above in shared memory
// after its dependency wait.  Negative sizes count as 0; rows past the
// capacity of A and D (GemmParams::m) are neither read into results nor stored.
struct GroupDev {
  const int* sizes;                   // device, `count` entries
  int count;
  int n_blocks;
  int ldd;
  void* d;
  const float* tb;
};
struct NoGroups {
  int unused;
};
// A list of independent GEMMs in one launch (GROUPED == 3): GEMM e has its
// own shape, operands, scales, output and alpha, given by its tensor maps and
// the per-GEMM fields below; its output tiles are tile_start[e] ..
// tile_start[e + 1] - 1 in the usual banded order.  Small GEMMs -- the
// projections of one decode step, a batch of 512^3 products -- then share one
// launch's fixed cost and fill the SMs together.
constexpr int kMaxList = 16;
struct GemmList {
  CUtensorMap maps[kMaxList][5];      // A, B, SFA, SFB, D of each GEMM
  int count;
  int tile_start[kMaxList + 1];
  int tiles_m[kMaxList];
  int tiles_n[kMaxList];
  int raster[kMaxList];               // M-blocks per raster band
  int m[kMaxList];
  int k[kMaxList];
  int kstages[kMaxList];
  int b_cta_rows[kMaxList];           // B rows each CTA of a pair supplies to one MMA
  uint32_t tx_bytes[kMaxList];        // bytes per stage on the (leader's) full barrier
  uint32_t idesc[kMaxList];           // MMA instruction descriptor (N narrowed for narrow GEMMs)
  float alpha[kMaxList];
  const float* ta[kMaxList];          // NVFP4 per-tensor scales (device, may be null)
  const float* tb[kMaxList];
};
template <int GROUPED>
using GroupArg = std::conditional_t<
    GROUPED == 1, GroupTable,
    std::conditional_t<GROUPED == 2, GroupDev, std::conditional_t<GROUPED == 3, GemmList, NoGroups>>>;

// Where one output tile's operands and results live.
struct TileCoord {
  int half;          // -1: a whole tile; 0 / 1: the first or second half (columns) of one
  int n0;            // first column of the tile (or half)
  int mb, nb;        // M-block (of kMmaM rows) and N-block of the tile
  int a_row;         // first row of this CTA's A rows (and D rows)
  int row_limit;     // rows at or past this one are not stored
  int b_row;         // first row of this CTA's B rows
  int sfa_block;     // 128-row scale block of this CTA's A rows
  int sfb_block0;    // first 128-row scale block of the tile's B rows
  int group;
};

// EXTRA_SMEM: static shared memory the kernel takes besides this layout (the
// device-size group table), counted when choosing the epilogue staging buffers.
template <int FMT, int CG, int BN, int STAGES, int ACC, int SCHED = SCHED_STATIC, int EXTRA_SMEM = 0>
struct GemmConfig {
  using T = FmtTraits<FMT>;
  static constexpr bool kScaled = FMT != FMT_BF16;
  static constexpr int kThreads = 384;
  static constexpr int kEpiWarps = 8;
  static constexpr int kCtaM = 128;                 // accumulator rows per CTA
  static constexpr int kMmaM = 128 * CG;
  static constexpr int kBRows = BN / CG;            // B rows loaded by each CTA
  // Dual accumulate (BN = 512, BF16): two N=256 MMAs per K step share the A
  // tile ("ThunderKittens 2.0" §二 2.2); each CTA loads two 128-row boxes of B,
  // one per half of the 512-column tile
  static constexpr bool kDual = BN == 512;
  static constexpr int kBBox = kDual ? kBRows / 2 : kBRows;
  static constexpr int kMmaN = kDual ? 256 : BN;
  static constexpr int kRowBytes = 128;             // K bytes per stage row
  static constexpr int kABytes = kCtaM * kRowBytes;
  static constexpr int kBBytes = kBRows * kRowBytes;
  static constexpr int kSfaBytes = T::kSfAtoms * 512;
  // B scales come in 128-row blocks of the tiled layout; every CTA holds the
  // whole N tile's scales (the MMA's B scales live in each CTA's tensor memory)
  static constexpr int kSfbBlocks = BN / 128;
  static constexpr int kSfbBytes = kScaled ? kSfbBlocks * T::kSfAtoms * 512 : 0;
  static constexpr int kStageBytes = ((kABytes + kBBytes + kSfaBytes + kSfbBytes + 1023) / 1024) * 1024;
  static constexpr int kMmasPerStage = T::kStageK / T::kMmaK;
  static constexpr int kEpiBufBytes = 32 * 64;      // 32 rows x 32 BF16
  static constexpr int kNumBars = 2 * STAGES + 2 * ACC + 2 + 4;
  // barriers, two tile-scheduler answers, alignment slack
  static constexpr int kFixedBytes = kNumBars * 8 + 2 * 16 + 16 + 1024;
  static constexpr bool kClc = SCHED == SCHED_CLC;
  // arrivals that free one scheduler answer: producer, epilogue warps, per CTA;
  // plus the MMA issuer and the scheduler itself in the pair leader
  static constexpr int kClcConsumers = CG * (1 + kEpiWarps) + 2;
  // two staging buffers per epilogue warp when they fit, else one
  static constexpr int kEpiBufs =
      STAGES * kStageBytes + kEpiWarps * 2 * kEpiBufBytes + kFixedBytes + EXTRA_SMEM <= 232448 ? 2 : 1;
  static constexpr int kEpiBytes = kEpiWarps * kEpiBufs * kEpiBufBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes + kEpiBytes;
  static constexpr int kSmemBytes = kBarOffset + kFixedBytes;
  // bytes landing on the leader's full barrier per stage (all CTAs of the pair),
  // for A boxes of a_rows rows and b_rows rows of B per CTA (both halves when dual)
  static constexpr uint32_t tx_bytes(int a_rows, int b_rows) {
    return uint32_t(CG * (a_rows * kRowBytes + b_rows * kRowBytes + kSfaBytes + kSfbBytes));
  }
  // tensor memory: ACC accumulators of BN columns, then a ring of scale
  // regions (4 columns of A scales + 4 per 128-row block of B scales), one
  // region per stage (MXFP8) or per MMA (NVFP4)
  static constexpr int kAccCols = BN;
  static constexpr int kScaleBase = ACC * kAccCols;
  static constexpr int kRegionCols = 4 + 4 * kSfbBlocks;
  static constexpr int kRegions = kScaled ? (512 - kScaleBase) / kRegionCols : 0;
  static constexpr int kTmemCols = 512;
  static_assert(!kScaled || kRegions >= 2, "tensor memory overflow");
  static_assert(ACC * kAccCols <= kTmemCols, "tensor memory overflow");
  static_assert(BN == 128 || BN == 256 || (BN == 512 && !kScaled && ACC == 1 && CG == 2),
                "B tiles must cover whole 128-row scale blocks; dual accumulate is BF16 pairs only");
  static_assert(kSmemBytes <= 232448, "shared memory overflow");
  static constexpr uint32_t kIdescBase =
      FMT == FMT_BF16 ? idesc_f16(kMmaM, kMmaN)
                      : idesc_bs(kMmaM, kMmaN, FMT == FMT_NVFP4 ? 1u : 0u, FMT == FMT_MXFP8 ? 1u : 0u, 0u, 0u);
};

struct Ctl {
  volatile int* abort_flag;   // this CTA's flag (shared memory)
  uint32_t abort_smem;        // its shared-memory address (same offset in every CTA)
  uint32_t rank;              // this CTA's rank in the cluster
  uint32_t ncta;              // CTAs in the cluster
  unsigned int* status;
  unsigned long long timeout_ns;
};

// Mark the kernel as aborting: this CTA's flag, every other CTA of the
// cluster, and the device status word the host reads.
__device__ __forceinline__ void raise_abort(const Ctl& c) {
  *c.abort_flag = 1;
  for (uint32_t r = 0; r < c.ncta; ++r)
    if (r != c.rank) ptx::st_shared_cluster_u32(ptx::map_to_rank(c.abort_smem, r), 1u);
  atomicOr(c.status, DEV_ERR_TIMEOUT);
}

// Bounded wait for the phase of parity `parity` of barrier `bar` to complete.
// Returns false when the kernel is aborting (timeout here or elsewhere).
// Each try sleeps until the phase completes or kWaitSleepNs pass; the abort
// flag and the time limit are checked between tries, so an abort raised
// elsewhere is seen within about kWaitSleepNs.
constexpr uint32_t kWaitSleepNs = 200000u;
template <bool kClusterScope>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (kClusterScope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
  while (true) {
    if (kClusterScope ? ptx::mbar_try_wait_cluster_sleep(bar, parity, kWaitSleepNs)
                      : ptx::mbar_try_wait_sleep(bar, parity, kWaitSleepNs))
      return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer() - t0 > c.timeout_ns) {
      raise_abort(c);
      return false;
    }
  }
}

// The same wait made by a whole converged warp; the answer is the same in
// every lane (an abort seen by one lane ends the wait for all).
template <bool kClusterScope>
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Ctl& c) {
  return __all_sync(0xffffffffu, wait_bar<kClusterScope>(bar, parity, c));
}

// GROUPED: 0 plain GEMM, 1 grouped with a host-built table, 2 grouped with
// device-resident group sizes (static schedule only), 3 a list of GEMMs.
template <int FMT, int CG, int BN, int STAGES, int ACC, int SCHED = SCHED_STATIC, int GROUPED = 0>
__global__ void __launch_bounds__(384, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmBh, const GemmParams p,
                const __grid_constant__ GroupArg<GROUPED> gt) {
  using C = GemmConfig<FMT, CG, BN, STAGES, ACC, SCHED, GROUPED == 2 ? kDevGroupTableBytes : 0>;
  using T = FmtTraits<FMT>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  static_assert(GROUPED != 2 || SCHED == SCHED_STATIC, "device group sizes need the static schedule");
  static_assert(GROUPED != 2 || C::kSmemBytes + kDevGroupTableBytes <= 232448,
                "dynamic shared memory and the group table exceed an SM's shared memory");
  // GROUPED == 2: first tile, first row, rows and first SFA block of each
  // group, then the tile count
  __shared__ int s_gtab[GROUPED == 2 ? 4 * kMaxGroups + 2 : 1];

  // Programmatic dependent launch: the next kernel may be scheduled onto free
  // SMs from here on (its own dependency wait still holds it until this grid
  // has completed); measured 1-1.5% faster on launch-bound skinny GEMMs than
  // releasing after the set-up.
  ptx::pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;

  // 1024-byte aligned carve-up (identical in both CTAs of a pair)
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  auto stage_a = [&](int s) { return base + uint32_t(s * C::kStageBytes); };
  auto stage_b = [&](int s) { return base + uint32_t(s * C::kStageBytes + C::kABytes); };
  auto stage_sfa = [&](int s) { return base + uint32_t(s * C::kStageBytes + C::kABytes + C::kBBytes); };
  // B scales: block a (of the loaded ones), atom g at stage_sfb + (a * kSfAtoms + g) * 512
  auto stage_sfb = [&](int s) {
    return base + uint32_t(s * C::kStageBytes + C::kABytes + C::kBBytes + C::kSfaBytes);
  };
  const uint32_t epi_base = base + uint32_t(STAGES * C::kStageBytes);
  const uint32_t bars = base + uint32_t(C::kBarOffset);
  auto full_bar = [&](int s) { return bars + uint32_t(8 * s); };
  auto empty_bar = [&](int s) { return bars + uint32_t(8 * (STAGES + s)); };
  auto accf_bar = [&](int a) { return bars + uint32_t(8 * (2 * STAGES + a)); };
  auto acce_bar = [&](int a) { return bars + uint32_t(8 * (2 * STAGES + ACC + a)); };
  const uint32_t drain_bar = bars + uint32_t(8 * (2 * STAGES + 2 * ACC));
  const uint32_t never_bar = drain_bar + 8;
  auto clc_full = [&](uint32_t i) { return never_bar + 8u + 8u * i; };     // answer i landed
  auto clc_empty = [&](uint32_t i) { return never_bar + 24u + 8u * i; };   // answer i read by all (leader)
  auto clc_resp = [&](uint32_t i) { return ((never_bar + 40u + 15u) & ~15u) + 16u * i; };   // 16-byte answers

  // group table: the host-built parameter, or the shared-memory copy built
  // from device sizes (filled after the dependency wait, read only after it)
  auto tab_tile_start = [&](int g) {
    if constexpr (GROUPED == 2) return s_gtab[g]; else if constexpr (GROUPED == 1) return gt.tile_start[g]; else return 0;
  };
  auto tab_row0 = [&](int g) {
    if constexpr (GROUPED == 2) return s_gtab[kMaxGroups + 1 + g]; else if constexpr (GROUPED == 1) return gt.row0[g]; else return 0;
  };
  auto tab_rows = [&](int g) {
    if constexpr (GROUPED == 2) return s_gtab[2 * kMaxGroups + 1 + g]; else if constexpr (GROUPED == 1) return gt.rows[g]; else return 0;
  };
  auto tab_sfa0 = [&](int g) {
    if constexpr (GROUPED == 2) return s_gtab[3 * kMaxGroups + 1 + g]; else if constexpr (GROUPED == 1) return gt.sfa_block0[g]; else return 0;
  };

  constexpr bool kList = GROUPED == 3;
  auto gt_count = [&]() -> int { if constexpr (GROUPED != 0) return gt.count; else return 1; };
  // tensor maps of the GEMM a tile belongs to (a list) or of the launch
  auto map_a = [&](int e) -> const void* { if constexpr (kList) return &gt.maps[e][0]; else { (void)e; return &tmA; } };
  auto map_b = [&](int e) -> const void* { if constexpr (kList) return &gt.maps[e][1]; else { (void)e; return &tmB; } };
  auto map_sfa = [&](int e) -> const void* { if constexpr (kList) return &gt.maps[e][2]; else { (void)e; return &tmSFA; } };
  auto map_sfb = [&](int e) -> const void* { if constexpr (kList) return &gt.maps[e][3]; else { (void)e; return &tmSFB; } };
  auto map_d = [&](int e) -> const void* { if constexpr (kList) return &gt.maps[e][4]; else { (void)e; return &tmD; } };
  // per-GEMM K stages, K, MMA descriptor and stage bytes
  auto kstages_of = [&](int e) { if constexpr (kList) return gt.kstages[e]; else { (void)e; return p.num_kstages; } };
  auto k_of = [&](int e) { if constexpr (kList) return gt.k[e]; else { (void)e; return p.k; } };
  auto idesc_of = [&](int e) { if constexpr (kList) return gt.idesc[e]; else { (void)e; return p.idesc; } };
  auto tx_of = [&](int e) { if constexpr (kList) return gt.tx_bytes[e]; else { (void)e; return p.tx_bytes; } };

  // Tile t -> operand coordinates for this CTA.
  auto coords = [&](int t) {
    TileCoord tc;
    if constexpr (kList) {
      int lo = 0, hi = gt.count;
#pragma unroll 1
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (gt.tile_start[mid] <= t) lo = mid; else hi = mid;
      }
      const int e = lo;
      tile_coords(t - gt.tile_start[e], gt.tiles_m[e], gt.tiles_n[e], gt.raster[e], tc.mb, tc.nb);
      tc.a_row = tc.mb * C::kMmaM + int(rank) * C::kCtaM;
      tc.row_limit = gt.m[e];
      tc.b_row = tc.nb * BN + int(rank) * gt.b_cta_rows[e];
      tc.sfa_block = tc.a_row / 128;
      tc.sfb_block0 = (tc.nb * BN) / 128;
      tc.group = e;
      tc.half = -1;
      tc.n0 = tc.nb * BN;
    } else if constexpr (GROUPED != 0) {
      // last group whose first tile is <= t (empty groups are skipped)
      int lo = 0, hi = gt.count;
#pragma unroll 1
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tab_tile_start(mid) <= t) lo = mid; else hi = mid;
      }
      const int g = lo;
      const int tiles_m_g = (tab_tile_start(g + 1) - tab_tile_start(g)) / p.tiles_n;
      tile_coords(t - tab_tile_start(g), tiles_m_g, p.tiles_n, p.raster_group, tc.mb, tc.nb);
      const int local_row = tc.mb * C::kMmaM + int(rank) * C::kCtaM;
      tc.a_row = tab_row0(g) + local_row;
      tc.row_limit = tab_row0(g) + tab_rows(g);
      if (tc.row_limit > p.m) tc.row_limit = p.m;   // never past the capacity of D
      tc.b_row = g * p.n + tc.nb * BN + int(rank) * p.b_cta_rows;
      tc.sfa_block = tab_sfa0(g) + local_row / 128;
      tc.sfb_block0 = g * gt.n_blocks + (tc.nb * BN) / 128;
      tc.group = g;
      tc.half = -1;
      tc.n0 = tc.nb * BN;
    } else {
      // tiles past tail_start are halves of the last tiles: tile tail_start + u / 2, half u % 2
      int o = t;
      tc.half = -1;
      if (t >= p.tail_start) {
        const int u = t - p.tail_start;
        o = p.tail_start + (u >> 1);
        tc.half = u & 1;
      }
      tile_coords(o, p.tiles_m, p.tiles_n, p.raster_group, tc.mb, tc.nb);
      tc.n0 = tc.nb * BN + (tc.half > 0 ? BN / 2 : 0);
      tc.a_row = tc.mb * C::kMmaM + int(rank) * C::kCtaM;
      tc.row_limit = p.m;
      tc.b_row = tc.n0 + int(rank) * (tc.half >= 0 ? p.b_cta_rows_half : p.b_cta_rows);
      tc.sfa_block = tc.a_row / 128;
      tc.sfb_block0 = tc.n0 / 128;
      tc.group = 0;
    }
    return tc;
  };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC; ++a) {
      ptx::mbar_init(accf_bar(a), 1);
      ptx::mbar_init(acce_bar(a), CG * C::kEpiWarps);   // every epilogue warp of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    ptx::mbar_init(never_bar, 1);
    for (uint32_t i = 0; i < 2; ++i) {
      ptx::mbar_init(clc_full(i), 1);
      ptx::mbar_init(clc_empty(i), C::kClcConsumers);
    }
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmD);
    if (C::kScaled) {
      ptx::prefetch_tmap(&tmSFA);
      ptx::prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 2) {
    ptx::tmem_alloc<CG>(ptx::smem_u32(&s_tmem_base), C::kTmemCols);
    ptx::tmem_relinquish<CG>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // The peer's barriers are initialised before anything reaches them: the
  // initialisations are published by fence.mbarrier_init (release, cluster
  // scope), so the arrive itself is relaxed (0.25-0.4 us per launch shorter
  // than a release arrive on 2048^3 GEMMs).  The one other word a peer writes
  // here, the abort flag, is written only after a wait has run out its time
  // limit, long after this CTA cleared it.
  if (CG == 2) ptx::cluster_sync_relaxed();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  // Warm L2 with the first stages of this cluster's first tile while the
  // previous kernel may still be running (prefetches read nothing back; see
  // ptx::tma_prefetch_2d).
  if (warp == 0) {
    if (GROUPED != 2 && ptx::elect_one() && int(blockIdx.x) / CG < p.num_tiles) {
      const TileCoord tc = coords(int(blockIdx.x) / CG);
      const int npf = min(kstages_of(tc.group), STAGES);
#pragma unroll 1
      for (int ks = 0; ks < npf; ++ks) {
        const int kx = ks * C::kRowBytes / (FMT == FMT_BF16 ? 2 : 1);
        ptx::tma_prefetch_2d(map_a(tc.group), kx, tc.a_row);
        ptx::tma_prefetch_2d(map_b(tc.group), kx, tc.b_row);
      }
    }
    if constexpr (GROUPED == 2) {
      // The group sizes may only be read after the dependency wait.  Prefetch
      // the B tile (and its scales) this cluster's first tile has when every
      // group holds one row block, the decode regime; a wrong guess costs only
      // L2 bandwidth (8 experts x 16 rows, N=4096, K=7168: 1.3-1.8 us less).
      if (ptx::elect_one()) {
        const int t = int(blockIdx.x) / CG;
        const int g = t / p.tiles_n;
        if (g < gt.count) {
          const int nb = t - g * p.tiles_n;
          const int b_row = g * p.n + nb * BN + int(rank) * p.b_cta_rows;
          const int npf = min(p.num_kstages, STAGES);
#pragma unroll 1
          for (int ks = 0; ks < npf; ++ks) {
            const int kx = ks * C::kRowBytes / (FMT == FMT_BF16 ? 2 : 1);
            ptx::tma_prefetch_2d(&tmB, kx, b_row);
            if constexpr (C::kScaled) {
#pragma unroll
              for (int a = 0; a < C::kSfbBlocks; ++a)
                ptx::tma_prefetch_3d(&tmSFB, 0, ks * T::kSfAtoms, g * gt.n_blocks + (nb * BN) / 128 + a);
            }
          }
        }
      }
    }
    __syncwarp();
  }
  // Programmatic dependent launch: the set-up above overlapped the previous
  // kernel's tail.  Only the roles that read global memory, or hand out work,
  // wait for the previous grid to complete (griddepcontrol.wait): the producer
  // right before its first load, the epilogue before it reads the tensor
  // scales, the scheduler before it takes tiles of clusters not yet launched
  // (before the release only the clusters resident early would get them).
  // The MMA issuer touches only shared and tensor memory, and every store of D
  // follows the producer's first load (through the stage and accumulator
  // barriers), hence the previous grid's completion.  The producer's set-up
  // runs before its wait (0.1-0.25 us per launch on 2048^3 and 4096^3 GEMMs).
  // Device-side group sizes are read by the whole CTA: it waits here.
  if constexpr (GROUPED == 2) ptx::pdl_wait();

  int num_tiles = p.num_tiles;
  if constexpr (GROUPED == 2) {
    // group table from the device sizes: one warp scans 32 groups at a time
    if (warp == 3) {
      int carry_t = 0, carry_r = 0, carry_b = 0;
#pragma unroll 1
      for (int g0 = 0; g0 < gt.count; g0 += 32) {
        const int g = g0 + lane;
        int mg = g < gt.count ? __ldg(gt.sizes + g) : 0;
        if (mg < 0) mg = 0;
        int tl = ((mg + C::kMmaM - 1) / C::kMmaM) * p.tiles_n, rw = mg, bl = (mg + 127) / 128;
        // inclusive scans over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int a = __shfl_up_sync(0xffffffffu, tl, o), b = __shfl_up_sync(0xffffffffu, rw, o),
                    c = __shfl_up_sync(0xffffffffu, bl, o);
          if (lane >= o) {
            tl += a;
            rw += b;
            bl += c;
          }
        }
        const int tiles_g = ((mg + C::kMmaM - 1) / C::kMmaM) * p.tiles_n;
        if (g < gt.count) {
          s_gtab[g] = carry_t + tl - tiles_g;
          s_gtab[kMaxGroups + 1 + g] = carry_r + rw - mg;
          s_gtab[2 * kMaxGroups + 1 + g] = mg;
          s_gtab[3 * kMaxGroups + 1 + g] = carry_b + bl - (mg + 127) / 128;
        }
        carry_t += __shfl_sync(0xffffffffu, tl, 31);
        carry_r += __shfl_sync(0xffffffffu, rw, 31);
        carry_b += __shfl_sync(0xffffffffu, bl, 31);
      }
      if (lane == 0) {
        s_gtab[gt.count] = carry_t;
        s_gtab[4 * kMaxGroups + 1] = carry_t;
      }
    }
    __syncthreads();
    num_tiles = s_gtab[4 * kMaxGroups + 1];
  }

  Ctl ctl;
  ctl.abort_flag = &s_abort;
  ctl.abort_smem = ptx::smem_u32(&s_abort);
  ctl.rank = rank;
  ctl.ncta = CG;
  ctl.status = p.status;
  ctl.timeout_ns = p.timeout_ns;

  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  const int first_tile = cluster_id < num_tiles ? cluster_id : -1;   // static grids may outnumber the tiles

  // Next tile for this cluster.  Static: a fixed stride over the tile list.
  // Cluster launch control: the grid holds one cluster per tile; a running
  // cluster takes over a cluster that has not started yet (its tile is that
  // cluster's index).  The pair leader's scheduler lane asks; every role reads
  // the answer from its own CTA's copy and releases it.  Returns -1 when no
  // tile is left, -2 when the kernel is aborting.  next_tile is called by a
  // whole converged warp (every lane waits and reads, lane 0 releases),
  // next_tile_lane by a role that runs in one elected lane.
  auto next_tile = [&](int t, uint32_t& cslot, uint32_t& cphase) -> int {
    if constexpr (!C::kClc) {
      (void)cslot;
      (void)cphase;
      return t + num_clusters < num_tiles ? t + num_clusters : -1;
    } else {
      if (!wait_bar_warp<false>(clc_full(cslot), cphase, ctl)) return -2;
      uint32_t x = 0;
      const bool got = ptx::clc_read(clc_resp(cslot), x);
      __syncwarp();
      if (lane == 0) {
        if (leader)
          ptx::mbar_arrive(clc_empty(cslot));
        else
          ptx::mbar_arrive_relaxed_cluster(ptx::map_to_rank(clc_empty(cslot), 0));
      }
      if (++cslot == 2) {
        cslot = 0;
        cphase ^= 1u;
      }
      return got ? int(x) / CG : -1;
    }
  };

  auto next_tile_lane = [&](int t, uint32_t& cslot, uint32_t& cphase) -> int {
    if constexpr (!C::kClc) {
      (void)cslot;
      (void)cphase;
      return t + num_clusters < num_tiles ? t + num_clusters : -1;
    } else {
      if (!wait_bar<false>(clc_full(cslot), cphase, ctl)) return -2;
      uint32_t x = 0;
      const bool got = ptx::clc_read(clc_resp(cslot), x);
      if (leader)
        ptx::mbar_arrive(clc_empty(cslot));
      else
        ptx::mbar_arrive_relaxed_cluster(ptx::map_to_rank(clc_empty(cslot), 0));
      if (++cslot == 2) {
        cslot = 0;
        cphase ^= 1u;
      }
      return got ? int(x) / CG : -1;
    }
  };

  // ------------------------------------------------------------------ producer
  if (warp == 0) {
    if (ptx::elect_one()) {
      // A panels are reused across the raster band; B streams through (measured
      // 3% faster than evict_normal for B at 16384^3, BF16 and MXFP8)
      const uint64_t pol_a = ptx::policy_evict_last();
      const uint64_t pol_b = ptx::policy_evict_first();
      // barrier the operand loads complete on: the pair leader's full barrier
      const uint32_t lead_full0 = (CG == 2) ? ptx::map_to_rank(full_bar(0), 0) : full_bar(0);
      uint32_t stage = 0, phase = 0;
      bool waited = GROUPED == 2;  // past griddepcontrol.wait
      uint32_t armed = 0;          // stages whose last arming is not yet known complete
      uint32_t armed_par = 0;      // parity of that arming
      bool ok = true;
      uint32_t cslot = 0, cphase = 0;
#pragma unroll 1
      for (int t = first_tile; t >= 0 && ok;) {
        const TileCoord tc = coords(t);
        const int a_row = tc.a_row;
        const int b_row = tc.b_row;
        const int sfb_block0 = tc.sfb_block0;
        const void* mA = map_a(tc.group);
        const bool half = tc.half >= 0;
        // a half tile's B box: half the rows per CTA (a second map), or for dual
        // accumulate one of its two boxes
        const void* mB = (half && !C::kDual) ? static_cast<const void*>(&tmBh) : map_b(tc.group);
        const void* mSFA = map_sfa(tc.group);
        const void* mSFB = map_sfb(tc.group);
        const int nks = kstages_of(tc.group);
        const uint32_t txb = half ? p.tx_half : tx_of(tc.group);
        // Serpentine K order: tiles of odd waves walk K backwards, so that they
        // start on the operand slices the previous wave read last, which are
        // still in L2 (BF16 16384^3: 13% fewer DRAM bytes).
        const bool rev = p.wave > 0 && ((t / p.wave) & 1);
#pragma unroll 1
        for (int it = 0; it < nks; ++it) {
          const int ks = rev ? nks - 1 - it : it;
          if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, ctl)) {
            ok = false;
            break;
          }
          armed &= ~(1u << stage);   // its previous load was consumed, hence complete
          const uint32_t fb = lead_full0 + 8u * stage;
          if (leader) {
            ptx::mbar_arrive_expect_tx(full_bar(stage), txb);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          const int kx = ks * C::kRowBytes / (FMT == FMT_BF16 ? 2 : 1);   // TMA x coordinate (elements)
          // a tile of this launch, a ring slot, a 16-byte aligned x (TMA's rule)
          if (!invariant(t < num_tiles && stage < uint32_t(STAGES) && ks >= 0 && ks < nks &&
                             (kx * (FMT == FMT_BF16 ? 2 : 1)) % 16 == 0 && (GROUPED == 0 || tc.group >= 0),
                         p.status)) {
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!waited) {
            ptx::pdl_wait();
            waited = true;
          }
          ptx::tma_load_2d<CG>(stage_a(stage), mA, kx, a_row, fb, pol_a);
          ptx::tma_load_2d<CG>(stage_b(stage), mB, kx, b_row, fb, pol_b);
          if constexpr (C::kDual) {   // second half of the 512-column tile
            if (!half)
              ptx::tma_load_2d<CG>(stage_b(stage) + uint32_t(C::kBBytes / 2), mB, kx, b_row + BN / 2, fb, pol_b);
          }
          if constexpr (C::kScaled) {
            const int atom0 = ks * T::kSfAtoms;
            // SFA: this CTA's 128 rows = scale block (a_row / 128)
            ptx::tma_load_3d<CG>(stage_sfa(stage), mSFA, 0, atom0, tc.sfa_block, fb, pol_a);
            // SFB: every CTA of the pair holds the whole N tile's scales (the
            // MMA reads B scales from each CTA's tensor memory), so each CTA
            // loads every 128-row block itself; plain loads, no multicast.
#pragma unroll
            for (int a = 0; a < C::kSfbBlocks; ++a)
              ptx::tma_load_3d<CG>(stage_sfb(stage) + uint32_t(a * T::kSfAtoms * 512), mSFB, 0, atom0,
                                   sfb_block0 + a, fb, pol_b);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        t = next_tile_lane(t, cslot, cphase);
        if (t == -2) ok = false;
      }
      if (!ok && leader) {
        // drain: every armed stage completes once its bytes land
        Ctl quiet = ctl;
        int dummy = 0;
        quiet.abort_flag = &dummy;   // keep waiting through the abort, still bounded
#pragma unroll 1
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) wait_bar<false>(full_bar(s), (armed_par >> s) & 1u, quiet);
      }
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ MMA issuer
  else if (warp == 1) {
    if (leader && ptx::elect_one()) {
      uint32_t stage = 0, phase = 0, acc = 0, accph = 0;
      uint32_t region = 0;        // next scale region in tensor memory (ring of kRegions)
      bool ok = true;
      if (p.inject_stall) ok = wait_bar<false>(never_bar, 0u, ctl);
      const uint16_t mask = (CG == 2) ? uint16_t(0x3) : uint16_t(0x1);
      uint32_t cslot = 0, cphase = 0;
      uint32_t committed = 0;     // tiles whose accumulator went to the epilogue
#pragma unroll 1
      for (int t = first_tile; t >= 0 && ok;) {
        if (!wait_bar<CG == 2>(acce_bar(acc), accph ^ 1u, ctl)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(acc * C::kAccCols);
        const bool rev = p.wave > 0 && ((t / p.wave) & 1);   // the producer's K order
        int e = 0;
        bool half = false;
        if constexpr (kList) {
          e = coords(t).group;
        } else if constexpr (GROUPED == 0) {
          half = t >= p.tail_start;
        }
        const int nks = kstages_of(e);
        const int kk = k_of(e);
        const uint32_t idesc0 = half ? p.idesc_half : idesc_of(e);
#pragma unroll 1
        for (int it = 0; it < nks; ++it) {
          const int ks = rev ? nks - 1 - it : it;
          if (!wait_bar<false>(full_bar(stage), phase, ctl)) {
            ok = false;
            break;
          }
          const uint64_t adesc = sdesc_sw128(stage_a(stage));
          const uint64_t bdesc = sdesc_sw128(stage_b(stage));
          // the accumulator columns this stage's MMAs write lie inside the allocation
          const uint32_t n_mma = ((idesc0 >> 17) & 0x3Fu) << 3;
          const bool stage_ok = invariant(stage < uint32_t(STAGES) && acc < uint32_t(ACC) &&
                                              acc * uint32_t(C::kAccCols) + n_mma +
                                                      ((C::kDual && !half) ? 256u : 0u) <= uint32_t(C::kTmemCols),
                                          p.status);
#pragma unroll
          for (int j = 0; j < C::kMmasPerStage; ++j) {
            const int k0 = ks * T::kStageK + j * T::kMmaK;
            if (k0 >= kk || !stage_ok) break;
            const uint64_t koff = uint64_t((j * 32) >> 4);   // 32 bytes of K per MMA
            const uint32_t accum = (it > 0 || j > 0) ? 1u : 0u;
            if constexpr (FMT == FMT_BF16) {
              ptx::mma_f16<CG>(d_tmem, adesc + koff, bdesc + koff, idesc0, accum);
              if constexpr (C::kDual) {
                if (!half) {
                  const uint64_t bdesc1 = sdesc_sw128(stage_b(stage) + uint32_t(C::kBBytes / 2));
                  ptx::mma_f16<CG>(d_tmem + 256u, adesc + koff, bdesc1 + koff, idesc0, accum);
                }
              }
            } else {
              // scales -> tensor memory from this thread, right before the MMAs that
              // read them: one region per stage (MXFP8: MMA j reads byte j of each
              // word) or per MMA (NVFP4: MMA j reads atom j)
              const int g = (FMT == FMT_NVFP4) ? j : 0;
              // the scale region lies between the accumulators and the end of the allocation
              if (!invariant(region < uint32_t(C::kRegions) &&
                                 uint32_t(C::kScaleBase) + (region + 1u) * uint32_t(C::kRegionCols) <=
                                     uint32_t(C::kTmemCols),
                             p.status))
                break;
              if (FMT == FMT_NVFP4 || j == 0) {
                const uint32_t reg = tmem + uint32_t(C::kScaleBase + region * C::kRegionCols);
                ptx::tmem_cp_32x128b_x4<CG>(reg, sdesc_sf(stage_sfa(stage) + uint32_t(512 * g)));
#pragma unroll
                for (int a = 0; a < C::kSfbBlocks; ++a)
                  ptx::tmem_cp_32x128b_x4<CG>(reg + uint32_t(4 + 4 * a),
                                              sdesc_sf(stage_sfb(stage) + uint32_t((a * T::kSfAtoms + g) * 512)));
              }
              const uint32_t reg = tmem + uint32_t(C::kScaleBase + region * C::kRegionCols);
              if constexpr (FMT == FMT_MXFP8) {
                const uint32_t idesc = idesc0 | (uint32_t(j) << 29) | (uint32_t(j) << 4);
                ptx::mma_mxf8<CG>(d_tmem, adesc + koff, bdesc + koff, idesc, reg, reg + 4u, accum);
              } else {
                ptx::mma_nvf4<CG>(d_tmem, adesc + koff, bdesc + koff, idesc0, reg, reg + 4u, accum);
              }
              if (FMT == FMT_NVFP4 || j == C::kMmasPerStage - 1 || k0 + T::kMmaK >= kk) {
                if (++region == uint32_t(C::kRegions)) region = 0;
              }
            }
          }
          ptx::tc_commit<CG>(empty_bar(stage), mask);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit<CG>(accf_bar(acc), mask);
        ++committed;
        if (++acc == ACC) {
          acc = 0;
          accph ^= 1u;
        }
        t = next_tile_lane(t, cslot, cphase);
        if (t == -2) ok = false;
      }
      // every MMA this thread issued has finished before tensor memory goes away
      ptx::tc_commit<CG>(drain_bar, uint16_t(1u << rank));
      Ctl quiet = ctl;
      int dummy = 0;
      quiet.abort_flag = &dummy;
      wait_bar<false>(drain_bar, 0u, quiet);
      // Every hand-back of an accumulator has landed before the pair may leave:
      // a follower's epilogue warps hand back with remote arrives on this CTA's
      // barrier, so none may still be in flight when the CTA exits (and the
      // teardown barrier below then needs no memory ordering).  Use u of
      // buffer a completes phase u - 1 of its barrier.
      if (ok) {
#pragma unroll 1
        for (uint32_t a = 0; a < uint32_t(ACC); ++a) {
          const uint32_t uses = committed / uint32_t(ACC) + (a < committed % uint32_t(ACC) ? 1u : 0u);
          if (uses) wait_bar<CG == 2>(acce_bar(a), (uses & 1u) ^ 1u, quiet);
        }
      }
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ tile scheduler
  else if (warp == 2) {
    if constexpr (C::kClc) {
      if constexpr (GROUPED != 2) ptx::pdl_wait();
      if (leader && ptx::elect_one()) {
        uint32_t slot = 0, ph = 0;
#pragma unroll 1
        while (true) {
          // the answer slot is free once every role has read its last answer
          if (!wait_bar<CG == 2>(clc_empty(slot), ph ^ 1u, ctl)) break;
          ptx::mbar_arrive_expect_tx(clc_full(slot), 16u);
          if (CG == 2) ptx::mbar_expect_tx_relaxed_cluster(ptx::map_to_rank(clc_full(slot), 1), 16u);
          ptx::clc_try_cancel<CG == 2>(clc_resp(slot), clc_full(slot));
          // read the answer too: a failed request ends the schedule
          if (!wait_bar<false>(clc_full(slot), ph, ctl)) break;
          uint32_t x = 0;
          const bool got = ptx::clc_read(clc_resp(slot), x);
          ptx::mbar_arrive(clc_empty(slot));
          if (++slot == 2) {
            slot = 0;
            ph ^= 1u;
          }
          if (!got) break;
        }
      }
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ epilogue
  else if (warp >= 4) {
    const int e = warp - 4;
    const int q = warp & 3;              // accumulator lane quadrant this warp may read
    const int h = e >> 2;                // column half of the tile: [0, BN/2) or [BN/2, BN)
    constexpr int kWarpChunks = BN / 64;               // 32-column accumulator chunks per warp
    constexpr int kPasses = (kWarpChunks + 3) / 4;     // four chunks (128 registers) per pass
    const uint32_t my_buf0 = epi_base + uint32_t(e * C::kEpiBufs * C::kEpiBufBytes);
    const uint32_t acce_lead0 = (CG == 2) ? ptx::map_to_rank(acce_bar(0), 0) : acce_bar(0);
    if constexpr (GROUPED != 2) ptx::pdl_wait();
    float alpha0 = p.alpha;
    if (p.ta) alpha0 = alpha0 * __ldg(p.ta);
    if (p.tb) alpha0 = alpha0 * __ldg(p.tb);
    uint32_t acc = 0, accph = 0;
    uint32_t cslot = 0, cphase = 0;
#pragma unroll 1
    for (int t = first_tile; t >= 0;) {
      const TileCoord tc = coords(t);
      float alpha = alpha0;
      if constexpr (GROUPED == 1 || GROUPED == 2) {
        if (gt.tb) alpha = alpha * __ldg(gt.tb + tc.group);
      } else if constexpr (kList) {
        // fp32(fp32(alpha * tA) * tB), as for the single GEMM
        alpha = gt.alpha[tc.group];
        if (gt.ta[tc.group]) alpha = alpha * __ldg(gt.ta[tc.group]);
        if (gt.tb[tc.group]) alpha = alpha * __ldg(gt.tb[tc.group]);
      }
      const void* mD = map_d(tc.group);
      // All 32 lanes wait, converged.  The issuing roles above run in one
      // elected lane (a producer or MMA warp whose 32 lanes ran the loop, with
      // one lane issuing, measured 5% and 2x slower on NVFP4), but eight
      // epilogue warps each waiting in lane 0 with 31 lanes parked cost 2-3%
      // on NVFP4 and BF16 (branch and convergence units busy the whole tile).
      if (!wait_bar_warp<false>(accf_bar(acc), accph, ctl)) break;
      ptx::tc_fence_after();
      const int row0 = tc.a_row + q * 32;
      // a 32-row box that crosses the end of a group (grouped GEMM) is stored
      // row by row so that the next group's rows are left alone
      const bool masked = ((GROUPED == 1 || GROUPED == 2) && row0 + 32 > tc.row_limit) ||
                          (GROUPED == 0 && p.direct_store != 0);
      const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + uint32_t(acc * C::kAccCols + h * (BN / 2));
      // a half tile holds BN / 2 columns: the warps of the second column half
      // only hand the accumulator back (as does every warp if a check fails)
      const bool idle = (tc.half >= 0 && h == 1) ||
                        !invariant(acc < uint32_t(ACC) && acc * uint32_t(C::kAccCols) + uint32_t(BN) <= uint32_t(C::kTmemCols) &&
                                       t < num_tiles && (!kList || tc.group < gt_count()),
                                   p.status);
#pragma unroll
      for (int pass = 0; pass < kPasses; ++pass) {
        const int nch = kWarpChunks - 4 * pass < 4 ? kWarpChunks - 4 * pass : 4;
        uint32_t v[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < nch && !idle) ptx::tmem_ld_32x32b_x32(tbase + uint32_t(pass * 128 + c * 32), v[c]);
        ptx::tmem_ld_wait();
        if (pass == kPasses - 1) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            // Accumulator buffer free.  The loads above have completed (wait::ld
            // returned), so nothing has to be ordered before the signal: leader
            // warps arrive on the MMA issuer's barrier directly, follower warps
            // with a relaxed remote arrive.  (A release arrive costs a
            // cluster-wide fence; a 16-byte copy completing on the barrier, used
            // before, measured 0.05-0.4 us per launch slower on 2048^3 to 8192^3
            // and 1-3% at 16384^3.)
            if (CG == 1 || leader)
              ptx::mbar_arrive(acce_bar(acc));
            else
              ptx::mbar_arrive_relaxed_cluster(acce_lead0 + 8u * acc);
          }
          if (++acc == ACC) {
            acc = 0;
            accph ^= 1u;
          }
        }
        if (idle) continue;
        const int col0 = tc.n0 + h * (BN / 2) + pass * 128;
        if (masked) {
          if constexpr (GROUPED != 3) {
            uint16_t* dbase;
            size_t ldd;
            if constexpr (GROUPED == 1 || GROUPED == 2) {
              dbase = static_cast<uint16_t*>(gt.d);
              ldd = size_t(gt.ldd);
            } else {
              dbase = static_cast<uint16_t*>(p.d);
              ldd = size_t(p.ldd);
            }
            const int r = row0 + lane;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (c >= nch) break;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t w[4];
#pragma unroll
                for (int x = 0; x < 4; ++x)
                  w[x] = ptx::pack_bf16x2(__uint_as_float(v[c][8 * j + 2 * x]) * alpha,
                                          __uint_as_float(v[c][8 * j + 2 * x + 1]) * alpha);
                const int col = col0 + c * 32 + j * 8;
                if (r < tc.row_limit && col < p.n) {
                  uint4* dst = reinterpret_cast<uint4*>(dbase + size_t(r) * ldd + col);
                  *dst = make_uint4(w[0], w[1], w[2], w[3]);
                }
              }
            }
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c >= nch || masked) break;
          const uint32_t buf = my_buf0 + uint32_t((C::kEpiBufs == 2 ? (c & 1) : 0) * C::kEpiBufBytes);
          if (lane == 0) {
            if (C::kEpiBufs == 2)
              ptx::bulk_wait_group_read<1>();
            else
              ptx::bulk_wait_group_read<0>();
          }
          __syncwarp();
          const uint32_t row_addr = buf + uint32_t(lane * 64);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float lo = __uint_as_float(v[c][8 * j + 2 * x]) * alpha;
              const float hi = __uint_as_float(v[c][8 * j + 2 * x + 1]) * alpha;
              w[x] = ptx::pack_bf16x2(lo, hi);
            }
            const uint32_t chunk = uint32_t(j) ^ ((uint32_t(lane) >> 1) & 3u);   // 64-byte swizzle
            ptx::st_shared_v4(row_addr + chunk * 16u, w[0], w[1], w[2], w[3]);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(mD, buf, col0 + c * 32, row0);
            ptx::bulk_commit_group();
          }
        }
      }
      t = __shfl_sync(0xffffffffu, next_tile(t, cslot, cphase), 0);
    }
    // the stores need only have read their shared memory before this CTA goes;
    // their global writes are part of the grid's work the next kernel waits for
    if (lane == 0) ptx::bulk_wait_group_read<0>();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (s_abort && threadIdx.x == 0) {
    // let any copy still in flight land before this CTA's shared memory is released
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 50000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA of a pair leaves (or frees tensor memory) before the other is
  // done with it; nothing is published here, so the arrive is relaxed
  // (0.4-0.6 us per launch shorter than a release arrive, measured on 2048^3
  // to 8192^3 GEMMs of every format)
  if (CG == 2) ptx::cluster_sync_relaxed();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<CG>(tmem, C::kTmemCols);
  }
}

}  // namespace tkg
