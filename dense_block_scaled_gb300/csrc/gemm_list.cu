// gemm_list.cu -- tkg_gemm_list_*: a list of independent GEMMs run by one
// persistent launch (the GROUPED == 3 instantiations of gemm_kernel).
//
// Each GEMM keeps its own tensor maps (A, B, scales, D), K, MMA descriptor and
// alpha in a kernel parameter table; the output tiles of all of them form one
// tile list that the persistent clusters walk (cluster launch control by
// default), so several small GEMMs fill the SMs together and pay one launch's
// fixed cost.
#include <cstdint>

#include "host_common.cuh"

namespace tkg {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The plain entry point's checks for one entry.  *skip: nothing to compute
// (empty, or k == 0 with D already zeroed -- done by the caller once every
// entry has passed).
tkg_status check_entry(int fmt, const tkg_gemm_desc& g, bool* skip) {
  *skip = false;
  if (g.m < 0 || g.n < 0 || g.k < 0) return TKG_ERR_INVALID_ARG;
  if (g.m == 0 || g.n == 0) {
    *skip = true;
    return TKG_OK;
  }
  if (!g.D) return TKG_ERR_INVALID_ARG;
  if (!aligned16(g.D) || (g.n % 8) != 0) return TKG_ERR_ALIGNMENT;
  if (g.k == 0) {
    *skip = true;
    return TKG_OK;
  }
  if (!g.A || !g.B) return TKG_ERR_INVALID_ARG;
  const int k_multiple = fmt == FMT_BF16 ? 8 : 32;
  if (!aligned16(g.A) || !aligned16(g.B) || (g.k % k_multiple) != 0) return TKG_ERR_ALIGNMENT;
  if (fmt != FMT_BF16) {
    if (!g.sfa || !g.sfb) return TKG_ERR_INVALID_ARG;
    if (!aligned16(g.sfa) || !aligned16(g.sfb)) return TKG_ERR_ALIGNMENT;
  }
  if (fmt == FMT_NVFP4 && ((g.tensor_scale_a && (reinterpret_cast<uintptr_t>(g.tensor_scale_a) & 3u)) ||
                           (g.tensor_scale_b && (reinterpret_cast<uintptr_t>(g.tensor_scale_b) & 3u))))
    return TKG_ERR_ALIGNMENT;
  return TKG_OK;
}

template <int FMT, int CG, int BN, int STAGES, int ACC, int SCHED>
tkg_status launch_list(const tkg_gemm_desc* const* gemms, int count, cudaStream_t stream) {
  using C = GemmConfig<FMT, CG, BN, STAGES, ACC, SCHED>;
  using T = FmtTraits<FMT>;
  static_assert(!C::kDual, "lists run 128- or 256-column tiles");
  auto kern = gemm_kernel<FMT, CG, BN, STAGES, ACC, SCHED, 3>;
  constexpr int kLaunchSmem = C::kSmemBytes > 118784 ? C::kSmemBytes : 118784;   // one CTA per SM

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TKG_ERR_CUDA;
  static bool attr_set[64] = {};
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLaunchSmem) != cudaSuccess)
      return TKG_ERR_CUDA;
    attr_set[dev] = true;
  }

  // the table is a kernel parameter (about 11 KB): kept per thread, off the stack
  static thread_local GemmList gl;
  gl.count = count;
  const bool bf16 = FMT == FMT_BF16;
  const CUtensorMapDataType vt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t boxk = bf16 ? 64 : 128;
  long long tiles = 0;
  tkg_status st;
  for (int e = 0; e < count; ++e) {
    const tkg_gemm_desc& g = *gemms[e];
    const uint64_t kdim = FMT == FMT_NVFP4 ? uint64_t(g.k) / 2 : uint64_t(g.k);
    const uint64_t row_bytes = bf16 ? uint64_t(g.k) * 2 : kdim;
    // boxes clipped to the GEMM (A to m rows, B to n rows) and a half-width
    // MMA for narrow GEMMs, as in the single-GEMM launch
    const int a_rows = g.m < C::kCtaM ? g.m : C::kCtaM;
    const bool narrow = g.n <= C::kMmaN / 2;
    const int mma_n = narrow ? C::kMmaN / 2 : C::kMmaN;
    const int b_cta_rows = mma_n / CG;
    const int b_box = g.n < b_cta_rows ? g.n : b_cta_rows;
    CUtensorMap* mp = gl.maps[e];
    if ((st = encode_2d(&mp[0], vt, g.A, kdim, g.m, row_bytes, boxk, uint32_t(a_rows), CU_TENSOR_MAP_SWIZZLE_128B)) !=
        TKG_OK)
      return st;
    if ((st = encode_2d(&mp[1], vt, g.B, kdim, g.n, row_bytes, boxk, uint32_t(b_box), CU_TENSOR_MAP_SWIZZLE_128B)) !=
        TKG_OK)
      return st;
    if ((st = encode_2d(&mp[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.D, g.n, g.m, uint64_t(g.n) * 2, 32, 32,
                        CU_TENSOR_MAP_SWIZZLE_64B)) != TKG_OK)
      return st;
    if constexpr (C::kScaled) {
      const int bs = FMT == FMT_MXFP8 ? 32 : 16;
      const int ka = ceil_div(ceil_div(g.k, bs), 4);
      if ((st = encode_3d(&mp[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, g.sfa, 128, ka, ceil_div(g.m, 128), 512,
                          uint64_t(ka) * 512, 128, T::kSfAtoms, 1)) != TKG_OK)
        return st;
      if ((st = encode_3d(&mp[3], CU_TENSOR_MAP_DATA_TYPE_UINT32, g.sfb, 128, ka, ceil_div(g.n, 128), 512,
                          uint64_t(ka) * 512, 128, T::kSfAtoms, 1)) != TKG_OK)
        return st;
    } else {
      mp[2] = mp[4];
      mp[3] = mp[4];
    }
    gl.tile_start[e] = int(tiles);
    gl.tiles_m[e] = ceil_div(g.m, C::kMmaM);
    gl.tiles_n[e] = ceil_div(g.n, BN);
    gl.raster[e] = raster_group(C::kMmaM, g.k, FMT, gl.tiles_m[e]);
    gl.m[e] = g.m;
    gl.k[e] = g.k;
    gl.kstages[e] = ceil_div(g.k, T::kStageK);
    gl.b_cta_rows[e] = b_cta_rows;
    gl.tx_bytes[e] = C::tx_bytes(a_rows, b_box);
    gl.idesc[e] = idesc_with_n(C::kIdescBase, mma_n);
    gl.alpha[e] = g.alpha;
    gl.ta[e] = FMT == FMT_NVFP4 ? g.tensor_scale_a : nullptr;
    gl.tb[e] = FMT == FMT_NVFP4 ? g.tensor_scale_b : nullptr;
    tiles += (long long)gl.tiles_m[e] * gl.tiles_n[e];
  }
  if (tiles > 0x7fffffff) return TKG_ERR_UNSUPPORTED;
  gl.tile_start[count] = int(tiles);

  GemmParams p{};
  p.num_tiles = int(tiles);
  p.tail_start = p.num_tiles;   // lists keep whole tiles and TMA stores
  p.direct_store = 0;
  p.alpha = 1.0f;
  p.ta = nullptr;
  p.tb = nullptr;
  if ((st = device_status_word(&p.status)) != TKG_OK) return st;
  const int tmo = option(TKG_OPT_TIMEOUT_MS);
  p.timeout_ns = 1000000ull * (unsigned long long)(tmo > 0 ? tmo : 1000);
  p.inject_stall = option(TKG_OPT_INJECT_STALL);
  // fields the list replaces per GEMM (kept consistent with the first one)
  p.m = gemms[0]->m;
  p.n = gemms[0]->n;
  p.k = gemms[0]->k;
  p.num_kstages = gl.kstages[0];
  p.tiles_m = gl.tiles_m[0];
  p.tiles_n = gl.tiles_n[0];
  p.raster_group = gl.raster[0];
  p.tx_bytes = gl.tx_bytes[0];
  p.idesc = gl.idesc[0];
  p.b_cta_rows = gl.b_cta_rows[0];

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
  int clusters = max_clusters < p.num_tiles ? max_clusters : p.num_tiles;
  const int cap = option(TKG_OPT_MAX_CLUSTERS);
  if (cap > 0 && clusters > cap) clusters = cap;
  if (SCHED == SCHED_CLC) clusters = p.num_tiles;
  cfg.gridDim = dim3(clusters * CG, 1, 1);
  p.wave = max_clusters;
  cudaError_t err =
      cudaLaunchKernelEx(&cfg, kern, gl.maps[0][0], gl.maps[0][1], gl.maps[0][2], gl.maps[0][3], gl.maps[0][4],
                         gl.maps[0][1], p, gl);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}

template <int FMT, int CG, int BN, int STAGES, int ACC>
tkg_status launch_list_sched(const tkg_gemm_desc* const* gemms, int count, cudaStream_t s) {
  if (option(TKG_OPT_SCHEDULER) == 1) return launch_list<FMT, CG, BN, STAGES, ACC, SCHED_STATIC>(gemms, count, s);
  return launch_list<FMT, CG, BN, STAGES, ACC, SCHED_CLC>(gemms, count, s);
}

// Tile shape of a list: 256 x 256 CTA pairs when the list has at least one
// wave of them; else single-CTA 128 x 256 tiles (pairs would leave as many SMs
// idle and gain nothing from sharing B); and 128 x 128 single-CTA tiles when
// even twice as many of those still fit one wave (a batch of 512^3 GEMMs: the
// narrower tiles put twice the SMs to work on the same FLOPs).
enum ListTiles { kPair256, kSingle256, kSingle128 };
ListTiles list_tiles(const tkg_gemm_desc* const* gemms, int count) {
  const int cg = option(TKG_OPT_CTA_GROUP);
  int sms = 0;
  if (device_sm_count(&sms) != TKG_OK) sms = 148;
  long long pair_tiles = 0, single_tiles = 0;
  for (int e = 0; e < count; ++e) {
    pair_tiles += (long long)ceil_div(gemms[e]->m, 256) * ceil_div(gemms[e]->n, 256);
    single_tiles += (long long)ceil_div(gemms[e]->m, 128) * ceil_div(gemms[e]->n, 256);
  }
  if (cg == 2 || (cg == 0 && pair_tiles >= sms / 2)) return kPair256;
  return 2 * single_tiles <= sms ? kSingle128 : kSingle256;
}

tkg_status gemm_list(int fmt, int count, const tkg_gemm_desc* gemms, cudaStream_t stream) {
  if (!gemms || count < 1) return TKG_ERR_INVALID_ARG;
  if (count > kMaxList) return TKG_ERR_UNSUPPORTED;
  const tkg_gemm_desc* run[kMaxList];
  int nrun = 0;
  bool zero[kMaxList] = {};
  for (int e = 0; e < count; ++e) {
    bool skip = false;
    const tkg_status st = check_entry(fmt, gemms[e], &skip);
    if (st != TKG_OK) return st;
    if (!skip) run[nrun++] = &gemms[e];
    else if (gemms[e].m > 0 && gemms[e].n > 0) zero[e] = true;   // k == 0: an empty sum
  }
  for (int e = 0; e < count; ++e)
    if (zero[e] && cudaMemsetAsync(gemms[e].D, 0, size_t(gemms[e].m) * size_t(gemms[e].n) * 2, stream) != cudaSuccess)
      return TKG_ERR_CUDA;
  if (nrun == 0) return TKG_OK;
  const ListTiles tiles = list_tiles(run, nrun);
  if (fmt == FMT_BF16) {
    if (tiles == kSingle128) return launch_list_sched<FMT_BF16, 1, 128, 6, 2>(run, nrun, stream);
    if (tiles == kSingle256) return launch_list_sched<FMT_BF16, 1, 256, 4, 2>(run, nrun, stream);
    return launch_list_sched<FMT_BF16, 2, 256, 6, 2>(run, nrun, stream);
  }
  if (fmt == FMT_MXFP8) {
    if (tiles == kSingle128) return launch_list_sched<FMT_MXFP8, 1, 128, 6, 1>(run, nrun, stream);
    if (tiles == kSingle256) return launch_list_sched<FMT_MXFP8, 1, 256, 4, 1>(run, nrun, stream);
    return launch_list_sched<FMT_MXFP8, 2, 256, 6, 1>(run, nrun, stream);
  }
  if (tiles == kSingle128) return launch_list_sched<FMT_NVFP4, 1, 128, 5, 1>(run, nrun, stream);
  if (tiles == kSingle256) return launch_list_sched<FMT_NVFP4, 1, 256, 3, 1>(run, nrun, stream);
  return launch_list_sched<FMT_NVFP4, 2, 256, 5, 1>(run, nrun, stream);
}

}  // namespace
}  // namespace tkg

extern "C" {

tkg_status tkg_gemm_list_bf16(int count, const tkg_gemm_desc* gemms, cudaStream_t stream) {
  return tkg::gemm_list(tkg::FMT_BF16, count, gemms, stream);
}

tkg_status tkg_gemm_list_mxfp8(int count, const tkg_gemm_desc* gemms, cudaStream_t stream) {
  return tkg::gemm_list(tkg::FMT_MXFP8, count, gemms, stream);
}

tkg_status tkg_gemm_list_nvfp4(int count, const tkg_gemm_desc* gemms, cudaStream_t stream) {
  return tkg::gemm_list(tkg::FMT_NVFP4, count, gemms, stream);
}

}  // extern "C"
