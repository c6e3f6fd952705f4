// gemm_noalloc.cu -- tkg_gemm_bf16_noalloc: the BF16 GEMM for callers that
// cannot allocate device memory.
//
// The regular entry points keep their one piece of scratch -- the status word
// a kernel sets when one of its bounded waits runs out -- in a buffer the
// library obtains with cudaMalloc on first use.  A runtime that reserves all
// of its device memory up front, or runs under a budget where a hidden
// allocation must not happen, cannot accept that.  This entry point runs the
// same kernel with its scratch in a fixed array that is part of the library
// image: every GPU that loads the library holds the array until the process
// exits, and no call allocates or frees anything.
//
// The array's name is only a host-side stand-in for the symbol; a kernel
// handed that name would fault (or, where the GPU can reach host memory,
// silently use the wrong bytes).  The device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first
// call made on it.
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.cuh"

namespace tkg {
namespace {

constexpr int kScratchBytes = 256;   // the array's fixed size
constexpr int kScratchWords = kScratchBytes / 4;
constexpr int kStatusWord = 0;       // the kernel's only scratch: one status word
constexpr size_t kScratchNeeded = sizeof(unsigned int);

static __device__ __align__(256) unsigned int g_noalloc_scratch[kScratchWords];

std::mutex g_mu;
unsigned int* g_scratch_dev[64] = {};   // device address of the array, per device
bool g_attr_set[64] = {};

// One-time set-up for the current device.  Returns the array's device address.
tkg_status scratch_for_current_device(unsigned int** out, int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TKG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    g_scratch_dev[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_scratch_dev[dev];
  *dev_out = dev;
  return TKG_OK;
}

}  // namespace
}  // namespace tkg

using namespace tkg;

extern "C" tkg_status tkg_gemm_bf16_noalloc(int m, int n, int k, const void* A, const void* B, void* D, float alpha,
                                            cudaStream_t stream) {
  // The scratch this kernel needs does not grow with m, n or k; the check
  // below keeps the stated limit explicit should that ever change.
  static_assert(kScratchNeeded <= size_t(kScratchBytes), "scratch exceeds the fixed array");
  if (m < 0 || n < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (kScratchNeeded > size_t(kScratchBytes)) return TKG_ERR_UNSUPPORTED;
  if (m == 0 || n == 0) return TKG_OK;
  if (!D) return TKG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(D) & 15u) || (n % 8) != 0) return TKG_ERR_ALIGNMENT;
  if (k == 0) return cudaMemsetAsync(D, 0, size_t(m) * size_t(n) * 2, stream) == cudaSuccess ? TKG_OK : TKG_ERR_CUDA;
  if (!A || !B) return TKG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) || (k % 8) != 0)
    return TKG_ERR_ALIGNMENT;

  using C = GemmConfig<FMT_BF16, 2, 256, 6, 2>;
  auto kern = gemm_kernel<FMT_BF16, 2, 256, 6, 2>;
  unsigned int* scratch = nullptr;
  int dev = 0;
  tkg_status st = scratch_for_current_device(&scratch, &dev);
  if (st != TKG_OK) return st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
        return TKG_ERR_CUDA;
      g_attr_set[dev] = true;
    }
  }

  CUtensorMap tmA, tmB, tmD;
  if ((st = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, k, m, uint64_t(k) * 2, 64, C::kCtaM,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  if ((st = encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, k, n, uint64_t(k) * 2, 64, C::kBRows,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != TKG_OK)
    return st;
  if ((st = encode_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, n, m, uint64_t(n) * 2, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B)) != TKG_OK)
    return st;

  GemmParams p;
  p.m = m;
  p.n = n;
  p.k = k;
  p.num_kstages = ceil_div(k, FmtTraits<FMT_BF16>::kStageK);
  p.tiles_m = ceil_div(m, C::kMmaM);
  p.tiles_n = ceil_div(n, 256);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.alpha = alpha;
  p.ta = nullptr;
  p.tb = nullptr;
  p.status = scratch + kStatusWord;
  const int tmo = option(TKG_OPT_TIMEOUT_MS);
  p.timeout_ns = 1000000ull * (unsigned long long)(tmo > 0 ? tmo : 1000);
  p.inject_stall = 0;
  p.raster_group = 8;
  p.wave = 0;
  p.tx_bytes = C::tx_bytes(C::kCtaM, C::kBRows);
  p.idesc = C::kIdescBase;
  p.b_cta_rows = C::kBBox;

  int sms = 0;
  if ((st = device_sm_count(&sms)) != TKG_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
    cudaGetLastError();
    clusters = sms / 2;
  }
  if (clusters > p.num_tiles) clusters = p.num_tiles;
  cfg.gridDim = dim3(2 * clusters, 1, 1);

  // The array keeps the previous call's contents: the status word must start at zero.
  if (cudaMemsetAsync(p.status, 0, kScratchNeeded, stream) != cudaSuccess) return TKG_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmD, tmD, tmD, p, NoGroups{0}) != cudaSuccess) {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  }
  return TKG_OK;
}
