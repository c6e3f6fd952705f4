// host_common.cuh -- host-side plumbing shared by the launchers: tensor-map
// encoding through the driver entry point, per-device state (status word, SM
// count), process-wide options, and the persistent cluster launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../../include/tkg_gemm.h"
#include "gemm_kernel.cuh"
#include "gemm_splitk.cuh"

namespace tkg {

struct Problem {
  int m, n, k;               // grouped: m = rows of A and D (at least the sum of the group sizes)
  const void* A;
  const void* B;
  const void* sfa;
  const void* sfb;
  const float* ta;
  const float* tb;           // grouped NVFP4: one per group
  void* D;
  float alpha;
  int groups = 0;            // grouped GEMM: number of groups, and their sizes (host)
  const int* m_sizes = nullptr;
  int ldd = 0;               // row stride of D in elements (0: n); plain GEMMs only
  uint64_t lda_bytes = 0;    // row pitch of A and B in bytes (0: contiguous rows); plain GEMMs only
  uint64_t ldb_bytes = 0;
  unsigned int* status = nullptr;   // device status word to use (null: the library's, allocated on first use)
};

// row stride of D in bytes
inline uint64_t d_row_bytes(const Problem& pr) { return uint64_t(pr.ldd > 0 ? pr.ldd : pr.n) * 2; }
// row pitches of A and B in bytes, given the contiguous pitch for the format
inline uint64_t a_row_bytes(const Problem& pr, uint64_t contiguous) { return pr.lda_bytes ? pr.lda_bytes : contiguous; }
inline uint64_t b_row_bytes(const Problem& pr, uint64_t contiguous) { return pr.ldb_bytes ? pr.ldb_bytes : contiguous; }

// ---- options and per-device state (tkg_api.cu)
int option(tkg_option o);
tkg_status device_status_word(unsigned int** out);   // lazily allocated per device
unsigned int* existing_status_word();                // the current device's word if allocated, else null
// allocation-free entry point (gemm_noalloc.cu): reads and clears its status
// word on the current device (0 when it was never set up there)
tkg_status noalloc_take_status(cudaStream_t stream, unsigned int* out);
tkg_status device_sm_count(int* out);
tkg_status device_l2_bytes(int* out);
// clusters of `size` (2 or 3) CTAs that can be resident at once when each CTA
// takes more than half of an SM's shared memory
tkg_status device_max_clusters(int size, int* out);

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// M-blocks per raster band: as many as let the band's A panels (rows x K
// bytes each) fill about a quarter of L2, between 4 and 32 (measured best at
// 16384^3 on GB300: BF16 4-8, MXFP8 8, NVFP4 16 bands; at half of L2 NVFP4
// loses 9%).  With dual accumulate the B panels are twice as wide, and bands
// three times as tall (capped at 12) measured best (BF16 16384^3: 12).
inline int raster_group(int block_rows, int k, int fmt, int tiles_m, bool dual = false) {
  const int forced = option(TKG_OPT_RASTER_GROUP);
  if (forced > 0) return forced < tiles_m ? forced : (tiles_m > 0 ? tiles_m : 1);
  int l2 = 0;
  if (device_l2_bytes(&l2) != TKG_OK || l2 <= 0) l2 = 96 << 20;
  const double bytes_per_elem = fmt == 0 ? 2.0 : (fmt == 1 ? 1.0 : 0.5);
  const double panel = double(block_rows) * double(k) * bytes_per_elem;
  int g = int((dual ? 0.75 : 0.25) * double(l2) / (panel > 1.0 ? panel : 1.0) + 0.5);
  if (g < 4) g = 4;
  if (g > (dual ? 12 : 32)) g = dual ? 12 : 32;
  if (g > tiles_m) g = tiles_m > 0 ? tiles_m : 1;
  return g;
}

// The last partial round of tiles is split into half-width tiles when its
// halves fit one round and at most this many full rounds precede it.  With
// more, cluster launch control has staggered the clusters enough that the last
// round is already short (measured at 8192^3: NVFP4 unchanged, MXFP8 2-4%
// slower split; at 4096^3, 3 full rounds: BF16 +4.8%, MXFP8 +1.8%, NVFP4 +2.3%).
constexpr int kTailSplitMaxRounds = 4;
inline bool split_tail(long long tiles, int clusters) {
  const long long full = tiles / clusters, r = tiles % clusters;
  return r > 0 && 2 * r <= clusters && full <= kTailSplitMaxRounds;
}

// Rounds of `tiles` equal tiles on `clusters` resident clusters, in units of
// one tile's time; a split last round counts as half a round.
inline double tile_rounds(long long tiles, int clusters, bool tail_split) {
  const long long full = tiles / clusters, r = tiles % clusters;
  if (r == 0) return double(full);
  return double(full) + ((tail_split && split_tail(tiles, clusters)) ? 0.5 : 1.0);
}

// BF16 dual accumulate (256 x 512 pair tiles) unless 256 x 256 tiles finish
// sooner: each option's time is its rounds of tiles times the tile width, and
// dual accumulate does the same work about 2-4% faster (measured: 16384^3
// 1711 -> 1755 TFLOP/s, 8192^3 1715 -> 1750, and 1895-1914 against 1863-1879
// for 256-wide tiles with a split tail).  At 16384^3 and 8192^3 that is dual,
// at 4096^3 256-wide tiles (3.5 rounds with the split tail against 2 rounds of
// twice the width: 1805 against 1723 TFLOP/s).
// TKG_OPT_BF16_TILE_N forces 256 or 512.
inline bool use_dual_bf16(const Problem& pr) {
  const int forced = option(TKG_OPT_BF16_TILE_N);
  if (forced == 512) return true;
  if (forced == 256) return false;
  int sms = 0;
  if (device_sm_count(&sms) != TKG_OK || sms < 2) return false;
  const int pairs = sms / 2;
  const bool split = option(TKG_OPT_TAIL_SPLIT) != 1;
  const long long tm = ceil_div(pr.m, 256);
  // at most half a wave of 512-wide tiles would all run as 256-wide halves,
  // which the double-buffered 256-wide kernel runs better (2048^3)
  if (2 * tm * ceil_div(pr.n, 512) <= pairs) return false;
  const double t512 = 2.0 * tile_rounds(tm * ceil_div(pr.n, 512), pairs, split) / 1.04;
  const double t256 = tile_rounds(tm * ceil_div(pr.n, 256), pairs, split);
  return t512 <= t256;
}

// ---- tensor maps (tkg_api.cu)
tkg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                     uint64_t row_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz);
tkg_status encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                     uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                     uint32_t box2);


// Launch one instantiation of the persistent GEMM (or, with GROUPED, of the
// grouped GEMM over pr.groups groups of rows).
template <int FMT, int CG, int BN, int STAGES, int ACC, int SCHED, int GROUPED = 0>
tkg_status launch_gemm(const Problem& pr, cudaStream_t stream) {
  using C = GemmConfig<FMT, CG, BN, STAGES, ACC, SCHED, GROUPED == 2 ? kDevGroupTableBytes : 0>;
  using T = FmtTraits<FMT>;
  auto kern = gemm_kernel<FMT, CG, BN, STAGES, ACC, SCHED, GROUPED>;
  // Request at least just over half an SM's shared memory so that no two CTAs
  // ever share an SM: each allocates all 512 tensor-memory columns.
  constexpr int kLaunchSmem = C::kSmemBytes > 118784 ? C::kSmemBytes : 118784;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TKG_ERR_CUDA;
  static bool attr_set[64] = {};   // per instantiation and device (idempotent if two threads race)
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLaunchSmem) != cudaSuccess)
      return TKG_ERR_CUDA;
    if (CG == 2 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
    }
    attr_set[dev] = true;
  }

  // group table: tiles, rows and scale blocks of each group
  GroupArg<GROUPED> gt{};
  int b_rows = pr.n, sfa_blocks = ceil_div(pr.m, 128), sfb_blocks = ceil_div(pr.n, 128);
  int total_tiles = ceil_div(pr.m, C::kMmaM) * ceil_div(pr.n, BN), max_tiles_m = ceil_div(pr.m, C::kMmaM);
  if constexpr (GROUPED == 2) {
    // sizes live on the device: size the tensor maps and the grid for the
    // capacity pr.m (the kernel finds the real tile count itself)
    if (pr.groups < 1 || pr.groups > kMaxGroups || !pr.m_sizes) return TKG_ERR_INVALID_ARG;
    gt.sizes = pr.m_sizes;
    gt.count = pr.groups;
    gt.n_blocks = ceil_div(pr.n, 128);
    gt.ldd = pr.n;
    gt.d = pr.D;
    gt.tb = pr.tb;
    b_rows = pr.groups * pr.n;
    sfa_blocks = ceil_div(pr.m, 128) + pr.groups;
    sfb_blocks = pr.groups * gt.n_blocks;
    total_tiles = (ceil_div(pr.m, C::kMmaM) + pr.groups) * ceil_div(pr.n, BN);
  } else if constexpr (GROUPED == 1) {
    if (pr.groups < 1 || pr.groups > kMaxGroups || !pr.m_sizes) return TKG_ERR_INVALID_ARG;
    const int tiles_n = ceil_div(pr.n, BN);
    gt.count = pr.groups;
    gt.n_blocks = ceil_div(pr.n, 128);
    gt.ldd = pr.n;
    gt.d = pr.D;
    gt.tb = pr.tb;
    long long row = 0, blk = 0, tiles = 0;
    max_tiles_m = 1;
    for (int g = 0; g < pr.groups; ++g) {
      const int mg = pr.m_sizes[g];
      gt.tile_start[g] = int(tiles);
      gt.row0[g] = int(row);
      gt.rows[g] = mg;
      gt.sfa_block0[g] = int(blk);
      const int tm = ceil_div(mg, C::kMmaM);
      if (tm > max_tiles_m) max_tiles_m = tm;
      tiles += (long long)tm * tiles_n;
      row += mg;
      blk += ceil_div(mg, 128);
    }
    gt.tile_start[pr.groups] = int(tiles);
    if (row > pr.m || tiles > 0x7fffffff) return TKG_ERR_INVALID_ARG;
    b_rows = pr.groups * pr.n;
    sfa_blocks = int(blk) > 0 ? int(blk) : 1;
    sfb_blocks = pr.groups * gt.n_blocks;
    total_tiles = int(tiles);
    if (total_tiles == 0) return TKG_OK;
  }

  // operand tensor maps: 128-byte K rows per stage, 128-byte swizzle
  CUtensorMap tmA, tmB, tmSFA, tmSFB, tmD;
  const bool bf16 = FMT == FMT_BF16;
  const CUtensorMapDataType vt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint64_t kdim = FMT == FMT_NVFP4 ? uint64_t(pr.k) / 2 : uint64_t(pr.k);   // elements along dim0
  const uint64_t row_bytes = FMT == FMT_BF16 ? uint64_t(pr.k) * 2 : kdim;
  const uint32_t boxk = bf16 ? 64 : 128;
  tkg_status st;
  // A box: the CTA's 128 rows, or all of M when M is shorter (measured: a box
  // that runs mostly past the last row slows the load stream, by a third at
  // M=1).  A grouped tile starts at its group's first row, so its box may still
  // run past the end, by fewer rows than M.
  const int a_rows = pr.m < C::kCtaM ? pr.m : C::kCtaM;
  if ((st = encode_2d(&tmA, vt, pr.A, kdim, pr.m, a_row_bytes(pr, row_bytes), boxk, uint32_t(a_rows),
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  // Narrow B (N at most half the MMA width; not dual, not grouped): the MMA runs
  // half as wide, each CTA of a pair supplying half its columns, so the tensor
  // pipe does not compute columns that do not exist; the B box is clipped to N
  // rows as the A box is to M.
  const bool narrow = GROUPED == 0 && !C::kDual && pr.n <= C::kMmaN / 2;
  const int mma_n = narrow ? C::kMmaN / 2 : C::kMmaN;
  const int b_cta_rows = C::kDual ? C::kBBox : mma_n / CG;
  const int b_box = (GROUPED == 0 && pr.n < b_cta_rows) ? pr.n : b_cta_rows;
  if ((st = encode_2d(&tmB, vt, pr.B, kdim, b_rows, b_row_bytes(pr, row_bytes), boxk, uint32_t(b_box),
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  // half tiles (the split last wave): an MMA half as wide, each CTA supplying
  // half as many B rows (dual accumulate: one of its two N = 256 MMAs and boxes)
  const int b_cta_rows_half = C::kDual ? C::kBBox : (C::kMmaN / 2) / CG;
  CUtensorMap tmBh = tmB;
  const bool can_split = GROUPED == 0 && !narrow;
  if (can_split && !C::kDual &&
      (st = encode_2d(&tmBh, vt, pr.B, kdim, b_rows, b_row_bytes(pr, row_bytes), boxk, uint32_t(b_cta_rows_half),
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  if ((st = encode_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pr.D, pr.n, pr.m, d_row_bytes(pr), 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B)) != TKG_OK)
    return st;
  if constexpr (C::kScaled) {
    const int bs = FMT == FMT_MXFP8 ? 32 : 16;
    const int ka = ceil_div(ceil_div(pr.k, bs), 4);   // 512-byte atoms per 128-row block
    if ((st = encode_3d(&tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, pr.sfa, 128, ka, sfa_blocks, 512,
                        uint64_t(ka) * 512, 128, T::kSfAtoms, 1)) != TKG_OK)
      return st;
    if ((st = encode_3d(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, pr.sfb, 128, ka, sfb_blocks, 512,
                        uint64_t(ka) * 512, 128, T::kSfAtoms, 1)) != TKG_OK)
      return st;
  } else {
    tmSFA = tmD;
    tmSFB = tmD;
  }

  GemmParams p;
  p.m = pr.m;
  p.n = pr.n;
  p.k = pr.k;
  p.num_kstages = ceil_div(pr.k, T::kStageK);
  p.tiles_m = ceil_div(pr.m, C::kMmaM);
  p.tiles_n = ceil_div(pr.n, BN);
  p.num_tiles = total_tiles;
  p.alpha = pr.alpha;
  p.ta = pr.ta;
  p.tb = GROUPED ? nullptr : pr.tb;
  if (pr.status)
    p.status = pr.status;
  else if ((st = device_status_word(&p.status)) != TKG_OK)
    return st;
  const int tmo = option(TKG_OPT_TIMEOUT_MS);
  p.timeout_ns = 1000000ull * (unsigned long long)(tmo > 0 ? tmo : 1000);
  p.inject_stall = option(TKG_OPT_INJECT_STALL);
  p.raster_group = raster_group(C::kMmaM, pr.k, FMT, max_tiles_m, C::kDual);

  int sms = 0;
  if ((st = device_sm_count(&sms)) != TKG_OK) return st;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = kLaunchSmem;
  cfg.stream = stream;
  int nattr = 0;
  if (CG == 2) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = CG;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  cfg.attrs = attr;
  cfg.numAttrs = nattr;

  // persistent grid: as many clusters as can be resident at once, no more than tiles
  static int max_clusters_dev[64] = {};
  int& max_clusters = max_clusters_dev[dev];
  if (max_clusters == 0) {
    if (CG == 2) {
      cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess || nc <= 0) {
        cudaGetLastError();
        nc = sms / 2;
      }
      max_clusters = nc;
    } else {
      max_clusters = sms;
    }
  }
  const int cap = option(TKG_OPT_MAX_CLUSTERS);
  const int resident = (SCHED == SCHED_STATIC && cap > 0 && cap < max_clusters) ? cap : max_clusters;

  // Split the last partial wave: with T tiles on P resident clusters the last
  // round holds r = T mod P tiles and takes as long as a full one; when its
  // 2r half-width tiles still fit one round, it takes about half as long
  // (split_tail also asks for few full rounds before it).
  p.tail_start = p.num_tiles;
  const int split_opt = option(TKG_OPT_TAIL_SPLIT);
  if (can_split && split_opt != 1 && p.num_tiles > 0) {
    if (split_opt == 2)
      p.tail_start = 0;   // every tile in halves (a test of the half-tile path)
    else if (split_tail(p.num_tiles, resident))
      p.tail_start = p.num_tiles - p.num_tiles % resident;
    p.num_tiles += p.num_tiles - p.tail_start;
  }
  p.b_cta_rows_half = b_cta_rows_half;
  // Epilogue stores: TMA boxes (1) or 16-byte stores from registers (2); plain
  // GEMMs only.  Automatic: direct stores for dual accumulate with many tiles per
  // cluster.  Its single 512-column accumulator drains in two passes and is
  // released only after the second pass's loads; direct stores do not hold
  // those loads up behind staging-buffer waits (16384^3, 27 rounds of tiles:
  // 1766 -> 1790 and 1778 -> 1805 TFLOP/s; 8192^3, 7 rounds: equal).  With one
  // tile per cluster the final drain is all that counts and TMA stores are
  // faster (M=1024, N=K=8192: 78.7 against 82.3 us), as they are for every other
  // tile shape (2048^3 BF16 12%, NVFP4 16384^3 5%).
  const int store_opt = option(TKG_OPT_EPILOGUE_STORE);
  const bool many_rounds = p.num_tiles >= 8 * resident;
  p.direct_store = (GROUPED == 0 && (store_opt == 2 || (store_opt == 0 && C::kDual && many_rounds))) ? 1 : 0;
  p.d = pr.D;
  p.ldd = pr.ldd > 0 ? pr.ldd : pr.n;
  p.tx_half = C::tx_bytes(a_rows, C::kDual ? b_box : b_cta_rows_half);
  p.idesc_half = C::kDual ? idesc_with_n(C::kIdescBase, mma_n) : idesc_with_n(C::kIdescBase, C::kMmaN / 2);

  int clusters = resident < p.num_tiles ? resident : p.num_tiles;
  // cluster launch control: one cluster per tile; running clusters take over
  // the ones that have not started
  if (SCHED == SCHED_CLC) clusters = p.num_tiles;
  cfg.gridDim = dim3(clusters * CG, 1, 1);

  p.wave = max_clusters;   // the serpentine K order flips every wave of resident clusters
  p.tx_bytes = C::tx_bytes(a_rows, C::kDual ? 2 * b_box : b_box);
  p.idesc = idesc_with_n(C::kIdescBase, mma_n);
  p.b_cta_rows = b_cta_rows;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSFA, tmSFB, tmD, tmBh, p, gt);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}

// Split-K launch: one cluster of SPLIT CTAs per 128 x 128 output tile.
template <int FMT, int SPLIT, int STAGES, int AROWS = 128>
tkg_status launch_splitk(const Problem& pr, cudaStream_t stream) {
  using C = SplitKConfig<FMT, SPLIT, STAGES, AROWS>;
  using T = FmtTraits<FMT>;
  auto kern = gemm_splitk_kernel<FMT, SPLIT, STAGES, AROWS>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TKG_ERR_CUDA;
  static bool attr_set[64] = {};
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return TKG_ERR_CUDA;
    attr_set[dev] = true;
  }
  CUtensorMap tmA, tmB, tmSFA, tmSFB, tmD;
  const bool bf16 = FMT == FMT_BF16;
  const CUtensorMapDataType vt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint64_t kdim = FMT == FMT_NVFP4 ? uint64_t(pr.k) / 2 : uint64_t(pr.k);
  const uint64_t row_bytes = FMT == FMT_BF16 ? uint64_t(pr.k) * 2 : kdim;
  const uint32_t boxk = bf16 ? 64 : 128;
  tkg_status st;
  const int a_rows = pr.m < AROWS ? pr.m : AROWS;   // no A box partly past the last row (see launch_gemm)
  if ((st = encode_2d(&tmA, vt, pr.A, kdim, pr.m, a_row_bytes(pr, row_bytes), boxk, uint32_t(a_rows),
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  // narrow B: an MMA of N = 64 (the tile's 128 columns would be mostly absent), box clipped to N rows
  const int mma_n = pr.n <= C::BN / 2 ? C::BN / 2 : C::BN;
  const int b_box = pr.n < mma_n ? pr.n : mma_n;
  if ((st = encode_2d(&tmB, vt, pr.B, kdim, pr.n, b_row_bytes(pr, row_bytes), boxk, uint32_t(b_box),
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  if ((st = encode_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pr.D, pr.n, pr.m, d_row_bytes(pr), 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B)) != TKG_OK)
    return st;
  if constexpr (C::kScaled) {
    const int bs = FMT == FMT_MXFP8 ? 32 : 16;
    const int ka = ceil_div(ceil_div(pr.k, bs), 4);
    if ((st = encode_3d(&tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, pr.sfa, 128, ka, ceil_div(pr.m, 128), 512,
                        uint64_t(ka) * 512, 128, T::kSfAtoms, 1)) != TKG_OK)
      return st;
    if ((st = encode_3d(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, pr.sfb, 128, ka, ceil_div(pr.n, 128), 512,
                        uint64_t(ka) * 512, 128, T::kSfAtoms, 1)) != TKG_OK)
      return st;
  } else {
    tmSFA = tmD;
    tmSFB = tmD;
  }
  GemmParams p;
  p.m = pr.m;
  p.n = pr.n;
  p.k = pr.k;
  p.num_kstages = ceil_div(pr.k, T::kStageK);
  p.tiles_m = ceil_div(pr.m, C::BM);
  p.tiles_n = ceil_div(pr.n, C::BN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.alpha = pr.alpha;
  p.ta = pr.ta;
  p.tb = pr.tb;
  if ((st = device_status_word(&p.status)) != TKG_OK) return st;
  const int tmo = option(TKG_OPT_TIMEOUT_MS);
  p.timeout_ns = 1000000ull * (unsigned long long)(tmo > 0 ? tmo : 1000);
  p.inject_stall = option(TKG_OPT_INJECT_STALL);
  p.wave = 0;
  p.tx_bytes = C::tx_bytes(a_rows, b_box);
  p.idesc = idesc_with_n(C::kIdesc, mma_n);
  p.b_cta_rows = mma_n;
  p.raster_group = raster_group(C::BM, pr.k, FMT, p.tiles_m);

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.gridDim = dim3(p.num_tiles * SPLIT, 1, 1);
  int nattr = 0;
  if (SPLIT > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = SPLIT;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSFA, tmSFB, tmD, p) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}

// K split for problems with few 128 x 128 output tiles: 2 or 3 CTAs per tile
// when that still fits one wave, 0 to use the persistent kernel.  Every CTA's
// stretch of K (ceil(stages / split) stages) must be non-empty, and the tiles'
// clusters must all be resident at once: SMs group into GPCs, so fewer clusters
// of 3 fit than a third of the SMs (M=16, N=6400, K=8192: 50 clusters of 3 ran
// in two waves, twice as long as 50 clusters of 2).
inline int choose_split(const Problem& pr, int stage_k) {
  const int forced = option(TKG_OPT_SPLIT_K);
  if (forced == 1) return 0;
  int sms = 0;
  if (device_sm_count(&sms) != TKG_OK) return 0;
  const int tiles = ceil_div(pr.m, 128) * ceil_div(pr.n, 128);
  const int stages = ceil_div(pr.k, stage_k);
  int split = forced >= 2 ? forced : (tiles * 2 <= sms ? (sms / tiles < 3 ? sms / tiles : 3) : 0);
  while (split >= 2 && (split - 1) * ceil_div(stages, split) >= stages) --split;
  if (forced < 2) {
    while (split >= 2) {
      int fit = 0;
      if (device_max_clusters(split, &fit) != TKG_OK || tiles <= fit) break;
      --split;
    }
  }
  return split >= 2 ? split : 0;
}

// Cluster launch control unless TKG_OPT_SCHEDULER asks for the static schedule.
template <int FMT, int CG, int BN, int STAGES, int ACC, int GROUPED = 0>
tkg_status launch_sched(const Problem& pr, cudaStream_t s) {
  if constexpr (GROUPED == 2) {
    return launch_gemm<FMT, CG, BN, STAGES, ACC, SCHED_STATIC, GROUPED>(pr, s);
  } else {
    if (option(TKG_OPT_SCHEDULER) == 1) return launch_gemm<FMT, CG, BN, STAGES, ACC, SCHED_STATIC, GROUPED>(pr, s);
    return launch_gemm<FMT, CG, BN, STAGES, ACC, SCHED_CLC, GROUPED>(pr, s);
  }
}

tkg_status launch_bf16(const Problem& pr, cudaStream_t s);
tkg_status launch_mxfp8(const Problem& pr, cudaStream_t s);
tkg_status launch_nvfp4(const Problem& pr, cudaStream_t s);
tkg_status launch_grouped_bf16(const Problem& pr, cudaStream_t s);
tkg_status launch_grouped_mxfp8(const Problem& pr, cudaStream_t s);
tkg_status launch_grouped_nvfp4(const Problem& pr, cudaStream_t s);
tkg_status launch_grouped_dev_bf16(const Problem& pr, cudaStream_t s);
tkg_status launch_grouped_dev_mxfp8(const Problem& pr, cudaStream_t s);
tkg_status launch_grouped_dev_nvfp4(const Problem& pr, cudaStream_t s);

}  // namespace tkg
