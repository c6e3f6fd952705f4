// tkg_api.cu -- the C ABI (include/tkg_gemm.h): argument checks, per-device
// state, options, tensor-map encoding, dispatch to the format launchers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "host_common.cuh"

namespace tkg {

// ------------------------------------------------------------------ options
static std::atomic<int> g_opts[16];

int option(tkg_option o) {
  const int i = int(o);
  return (i > 0 && i < 16) ? g_opts[i].load(std::memory_order_relaxed) : 0;
}

// ------------------------------------------------------------------ per-device state
static std::mutex g_dev_mu;
static unsigned int* g_status[64] = {};
static int g_sms[64] = {};
static int g_l2[64] = {};
static int g_clusters[64][4] = {};   // resident clusters of 2 and 3 one-per-SM CTAs

static int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return (dev >= 0 && dev < 64) ? dev : -1;
}

tkg_status device_status_word(unsigned int** out) {
  const int dev = current_device();
  if (dev < 0) return TKG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_status[dev]) {
    void* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return TKG_ERR_CUDA;
    if (cudaMemset(p, 0, 256) != cudaSuccess) return TKG_ERR_CUDA;
    g_status[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status[dev];
  return TKG_OK;
}

unsigned int* existing_status_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  return g_status[dev];
}

tkg_status device_sm_count(int* out) {
  const int dev = current_device();
  if (dev < 0) return TKG_ERR_CUDA;
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return TKG_ERR_CUDA;
    g_sms[dev] = n;
  }
  *out = g_sms[dev];
  return TKG_OK;
}

// Stands in for any kernel whose CTAs each take more than half of an SM's
// shared memory (one CTA per SM): how many clusters of such CTAs can be resident
// at once depends only on the cluster size and how the SMs group into GPCs.
static __global__ void __launch_bounds__(384, 1) cluster_capacity_probe() {}

tkg_status device_max_clusters(int size, int* out) {
  const int dev = current_device();
  if (dev < 0 || size < 2 || size > 3) return TKG_ERR_CUDA;
  if (g_clusters[dev][size] == 0) {
    int sms = 0;
    tkg_status st = device_sm_count(&sms);
    if (st != TKG_OK) return st;
    constexpr int kSmem = 160 * 1024;   // above half of an SM's 228 KB
    if (cudaFuncSetAttribute(cluster_capacity_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(size * (sms / size)), 1, 1);
    cfg.blockDim = dim3(384, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, cluster_capacity_probe, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    g_clusters[dev][size] = n;
  }
  *out = g_clusters[dev][size];
  return TKG_OK;
}

tkg_status device_l2_bytes(int* out) {
  const int dev = current_device();
  if (dev < 0) return TKG_ERR_CUDA;
  if (g_l2[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) return TKG_ERR_CUDA;
    g_l2[dev] = n;
  }
  *out = g_l2[dev];
  return TKG_OK;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Encoding a tensor map costs about a microsecond, and a GEMM needs up to
// five (a GEMM list five per GEMM); small GEMMs are bound by that host work.  Each thread keeps the maps it
// encoded in a small direct-mapped cache keyed by every encoding argument (a
// map holds only the address and geometry, never the data).
namespace {
struct MapKey {
  uint32_t dtype, rank, swizzle;
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  bool operator==(const MapKey& o) const {
    return dtype == o.dtype && rank == o.rank && swizzle == o.swizzle && base == o.base && dims[0] == o.dims[0] &&
           dims[1] == o.dims[1] && dims[2] == o.dims[2] && strides[0] == o.strides[0] &&
           strides[1] == o.strides[1] && box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2];
  }
};
struct MapEntry {
  bool valid = false;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapCacheSize = 256;   // 64 KB per thread
thread_local MapEntry t_map_cache[kMapCacheSize];

uint32_t key_hash(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
  for (int i = 0; i < 3; ++i) h ^= (k.dims[i] + 0x7F4A7C15ull * (i + 1)) * 0xBF58476D1CE4E5B9ull;
  h ^= (uint64_t(k.box[0]) << 32 | k.box[1]) * 0x94D049BB133111EBull;
  h ^= uint64_t(k.dtype) << 40 ^ uint64_t(k.swizzle) << 48 ^ k.strides[0];
  return uint32_t(h >> 32) % kMapCacheSize;
}

tkg_status encode_cached(CUtensorMap* map, const MapKey& key) {
  MapEntry& e = t_map_cache[key_hash(key)];
  if (e.valid && e.key == key) {
    *map = e.map;
    return TKG_OK;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return TKG_ERR_CUDA;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CUtensorMapDataType(key.dtype), key.rank, const_cast<void*>(key.base), key.dims, key.strides,
                  key.box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CUtensorMapSwizzle(key.swizzle),
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return TKG_ERR_INVALID_ARG;
  e.valid = true;
  e.key = key;
  e.map = *map;
  return TKG_OK;
}
}  // namespace

tkg_status encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                     uint64_t row_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz) {
  MapKey k{uint32_t(dtype), 2u, uint32_t(swz), base, {dim0, dim1, 0}, {row_bytes, 0}, {box0, box1, 0}};
  return encode_cached(map, k);
}

tkg_status encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                     uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                     uint32_t box2) {
  MapKey k{uint32_t(dtype), 3u, uint32_t(CU_TENSOR_MAP_SWIZZLE_NONE), base, {dim0, dim1, dim2},
           {stride1_bytes, stride2_bytes}, {box0, box1, box2}};
  return encode_cached(map, k);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks; returns TKG_OK and sets *empty when there is nothing to launch.
static tkg_status check_common(int m, int n, int k, const void* A, const void* B, void* D, int k_multiple,
                               bool* empty, cudaStream_t stream) {
  *empty = false;
  if (m < 0 || n < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (m == 0 || n == 0) {
    *empty = true;
    return TKG_OK;
  }
  if (!D) return TKG_ERR_INVALID_ARG;
  if (!aligned16(D) || (n % 8) != 0) return TKG_ERR_ALIGNMENT;
  if (k == 0) {   // empty sum: D = 0
    *empty = true;
    return cudaMemsetAsync(D, 0, size_t(m) * size_t(n) * 2, stream) == cudaSuccess ? TKG_OK : TKG_ERR_CUDA;
  }
  if (!A || !B) return TKG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || (k % k_multiple) != 0) return TKG_ERR_ALIGNMENT;
  return TKG_OK;
}

// Grouped GEMM: checks shared by the three formats.  Sets *rows to the sum of
// the group sizes and *empty when there is nothing to launch.
static tkg_status check_grouped(int groups, const int* m_sizes, int n, int k, const void* A, const void* B, void* D,
                                int k_multiple, int* rows, bool* empty, cudaStream_t stream) {
  *empty = false;
  *rows = 0;
  if (groups < 1 || !m_sizes || n < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (groups > kMaxGroups) return TKG_ERR_UNSUPPORTED;
  long long total = 0;
  for (int g = 0; g < groups; ++g) {
    if (m_sizes[g] < 0) return TKG_ERR_INVALID_ARG;
    total += m_sizes[g];
  }
  if (total > 0x7fffffffLL) return TKG_ERR_UNSUPPORTED;
  *rows = int(total);
  if (total == 0 || n == 0) {
    *empty = true;
    return TKG_OK;
  }
  return check_common(int(total), n, k, A, B, D, k_multiple, empty, stream);
}

}  // namespace tkg

using namespace tkg;

extern "C" {

tkg_status tkg_gemm_bf16(int m, int n, int k, const void* A, const void* B, void* D, float alpha,
                         cudaStream_t stream) {
  bool empty;
  tkg_status st = check_common(m, n, k, A, B, D, 8, &empty, stream);
  if (st != TKG_OK || empty) return st;
  Problem pr{m, n, k, A, B, nullptr, nullptr, nullptr, nullptr, D, alpha};
  return launch_bf16(pr, stream);
}

tkg_status tkg_gemm_mxfp8(int m, int n, int k, const void* A, const void* B, const void* sfa, const void* sfb,
                          void* D, float alpha, cudaStream_t stream) {
  bool empty;
  tkg_status st = check_common(m, n, k, A, B, D, 32, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  Problem pr{m, n, k, A, B, sfa, sfb, nullptr, nullptr, D, alpha};
  return launch_mxfp8(pr, stream);
}

tkg_status tkg_gemm_nvfp4(int m, int n, int k, const void* A, const void* B, const void* sfa, const void* sfb,
                          const float* tensor_scale_a, const float* tensor_scale_b, void* D, float alpha,
                          cudaStream_t stream) {
  bool empty;
  tkg_status st = check_common(m, n, k, A, B, D, 32, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  if ((tensor_scale_a && (reinterpret_cast<uintptr_t>(tensor_scale_a) & 3u)) ||
      (tensor_scale_b && (reinterpret_cast<uintptr_t>(tensor_scale_b) & 3u)))
    return TKG_ERR_ALIGNMENT;
  Problem pr{m, n, k, A, B, sfa, sfb, tensor_scale_a, tensor_scale_b, D, alpha};
  return launch_nvfp4(pr, stream);
}

// Row pitches of the strided entry points.  lda / ldb count the operands'
// storage units (BF16 elements; bytes of E4M3 or packed E2M1 codes), ldd BF16
// elements of D.  Checks as check_common, plus: a pitch shorter than a row is
// an invalid argument, a pitch that is not a multiple of 16 bytes a
// misalignment.  k == 0 zeroes the m x n block of D.
static tkg_status check_strided(int m, int n, int k, const void* A, int lda, const void* B, int ldb, void* D, int ldd,
                                int k_multiple, int unit_bytes, int units_per_row, bool* empty, cudaStream_t stream) {
  *empty = false;
  if (m < 0 || n < 0 || k < 0 || lda < 0 || ldb < 0 || ldd < 0) return TKG_ERR_INVALID_ARG;
  if (m == 0 || n == 0) {
    *empty = true;
    return TKG_OK;
  }
  if (!D || ldd < n) return TKG_ERR_INVALID_ARG;
  if (!aligned16(D) || (ldd % 8) != 0) return TKG_ERR_ALIGNMENT;
  if (k == 0) {
    *empty = true;
    return cudaMemset2DAsync(D, size_t(ldd) * 2, 0, size_t(n) * 2, size_t(m), stream) == cudaSuccess ? TKG_OK
                                                                                                     : TKG_ERR_CUDA;
  }
  if (!A || !B || lda < units_per_row || ldb < units_per_row) return TKG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || (k % k_multiple) != 0 || (size_t(lda) * unit_bytes) % 16 != 0 ||
      (size_t(ldb) * unit_bytes) % 16 != 0)
    return TKG_ERR_ALIGNMENT;
  return TKG_OK;
}

tkg_status tkg_gemm_bf16_strided(int m, int n, int k, const void* A, int lda, const void* B, int ldb, void* D, int ldd,
                                 float alpha, cudaStream_t stream) {
  bool empty;
  tkg_status st = check_strided(m, n, k, A, lda, B, ldb, D, ldd, 8, 2, k, &empty, stream);
  if (st != TKG_OK || empty) return st;
  Problem pr{m, n, k, A, B, nullptr, nullptr, nullptr, nullptr, D, alpha};
  pr.ldd = ldd;
  pr.lda_bytes = uint64_t(lda) * 2;
  pr.ldb_bytes = uint64_t(ldb) * 2;
  return launch_bf16(pr, stream);
}

tkg_status tkg_gemm_mxfp8_strided(int m, int n, int k, const void* A, int lda, const void* B, int ldb, const void* sfa,
                                  const void* sfb, void* D, int ldd, float alpha, cudaStream_t stream) {
  bool empty;
  tkg_status st = check_strided(m, n, k, A, lda, B, ldb, D, ldd, 32, 1, k, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  Problem pr{m, n, k, A, B, sfa, sfb, nullptr, nullptr, D, alpha};
  pr.ldd = ldd;
  pr.lda_bytes = uint64_t(lda);
  pr.ldb_bytes = uint64_t(ldb);
  return launch_mxfp8(pr, stream);
}

tkg_status tkg_gemm_nvfp4_strided(int m, int n, int k, const void* A, int lda, const void* B, int ldb, const void* sfa,
                                  const void* sfb, const float* tensor_scale_a, const float* tensor_scale_b, void* D,
                                  int ldd, float alpha, cudaStream_t stream) {
  bool empty;
  tkg_status st = check_strided(m, n, k, A, lda, B, ldb, D, ldd, 32, 1, k / 2, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  if ((tensor_scale_a && (reinterpret_cast<uintptr_t>(tensor_scale_a) & 3u)) ||
      (tensor_scale_b && (reinterpret_cast<uintptr_t>(tensor_scale_b) & 3u)))
    return TKG_ERR_ALIGNMENT;
  Problem pr{m, n, k, A, B, sfa, sfb, tensor_scale_a, tensor_scale_b, D, alpha};
  pr.ldd = ldd;
  pr.lda_bytes = uint64_t(lda);
  pr.ldb_bytes = uint64_t(ldb);
  return launch_nvfp4(pr, stream);
}

tkg_status tkg_gemm_grouped_bf16(int groups, const int* m_sizes, int n, int k, const void* A, const void* B, void* D,
                                 float alpha, cudaStream_t stream) {
  bool empty;
  int rows;
  tkg_status st = check_grouped(groups, m_sizes, n, k, A, B, D, 8, &rows, &empty, stream);
  if (st != TKG_OK || empty) return st;
  Problem pr{rows, n, k, A, B, nullptr, nullptr, nullptr, nullptr, D, alpha, groups, m_sizes};
  return launch_grouped_bf16(pr, stream);
}

tkg_status tkg_gemm_grouped_mxfp8(int groups, const int* m_sizes, int n, int k, const void* A, const void* B,
                                  const void* sfa, const void* sfb, void* D, float alpha, cudaStream_t stream) {
  bool empty;
  int rows;
  tkg_status st = check_grouped(groups, m_sizes, n, k, A, B, D, 32, &rows, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  Problem pr{rows, n, k, A, B, sfa, sfb, nullptr, nullptr, D, alpha, groups, m_sizes};
  return launch_grouped_mxfp8(pr, stream);
}

tkg_status tkg_gemm_grouped_nvfp4(int groups, const int* m_sizes, int n, int k, const void* A, const void* B,
                                  const void* sfa, const void* sfb, const float* tensor_scale_a,
                                  const float* tensor_scales_b, void* D, float alpha, cudaStream_t stream) {
  bool empty;
  int rows;
  tkg_status st = check_grouped(groups, m_sizes, n, k, A, B, D, 32, &rows, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  if ((tensor_scale_a && (reinterpret_cast<uintptr_t>(tensor_scale_a) & 3u)) ||
      (tensor_scales_b && (reinterpret_cast<uintptr_t>(tensor_scales_b) & 3u)))
    return TKG_ERR_ALIGNMENT;
  Problem pr{rows, n, k, A, B, sfa, sfb, tensor_scale_a, tensor_scales_b, D, alpha, groups, m_sizes};
  return launch_grouped_nvfp4(pr, stream);
}

// Device-resident group sizes: checks shared by the three formats.
static tkg_status check_grouped_dev(int groups, const int* m_sizes_dev, int m_capacity, int n, int k, const void* A,
                                    const void* B, void* D, int k_multiple, bool* empty, cudaStream_t stream) {
  *empty = false;
  if (groups < 1 || !m_sizes_dev || m_capacity < 0 || n < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (groups > kMaxGroups) return TKG_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(m_sizes_dev) & 3u) return TKG_ERR_ALIGNMENT;
  if (m_capacity == 0 || n == 0) {
    *empty = true;
    return TKG_OK;
  }
  if (k == 0) return TKG_ERR_UNSUPPORTED;   // the rows to zero are known only on the device
  return check_common(m_capacity, n, k, A, B, D, k_multiple, empty, stream);
}

tkg_status tkg_gemm_grouped_dev_bf16(int groups, const int* m_sizes_dev, int m_capacity, int n, int k, const void* A,
                                     const void* B, void* D, float alpha, cudaStream_t stream) {
  bool empty;
  tkg_status st = check_grouped_dev(groups, m_sizes_dev, m_capacity, n, k, A, B, D, 8, &empty, stream);
  if (st != TKG_OK || empty) return st;
  Problem pr{m_capacity, n, k, A, B, nullptr, nullptr, nullptr, nullptr, D, alpha, groups, m_sizes_dev};
  return launch_grouped_dev_bf16(pr, stream);
}

tkg_status tkg_gemm_grouped_dev_mxfp8(int groups, const int* m_sizes_dev, int m_capacity, int n, int k, const void* A,
                                      const void* B, const void* sfa, const void* sfb, void* D, float alpha,
                                      cudaStream_t stream) {
  bool empty;
  tkg_status st = check_grouped_dev(groups, m_sizes_dev, m_capacity, n, k, A, B, D, 32, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  Problem pr{m_capacity, n, k, A, B, sfa, sfb, nullptr, nullptr, D, alpha, groups, m_sizes_dev};
  return launch_grouped_dev_mxfp8(pr, stream);
}

tkg_status tkg_gemm_grouped_dev_nvfp4(int groups, const int* m_sizes_dev, int m_capacity, int n, int k, const void* A,
                                      const void* B, const void* sfa, const void* sfb, const float* tensor_scale_a,
                                      const float* tensor_scales_b, void* D, float alpha, cudaStream_t stream) {
  bool empty;
  tkg_status st = check_grouped_dev(groups, m_sizes_dev, m_capacity, n, k, A, B, D, 32, &empty, stream);
  if (st != TKG_OK || empty) return st;
  if (!sfa || !sfb) return TKG_ERR_INVALID_ARG;
  if (!aligned16(sfa) || !aligned16(sfb)) return TKG_ERR_ALIGNMENT;
  if ((tensor_scale_a && (reinterpret_cast<uintptr_t>(tensor_scale_a) & 3u)) ||
      (tensor_scales_b && (reinterpret_cast<uintptr_t>(tensor_scales_b) & 3u)))
    return TKG_ERR_ALIGNMENT;
  Problem pr{m_capacity, n, k, A, B, sfa, sfb, tensor_scale_a, tensor_scales_b, D, alpha, groups, m_sizes_dev};
  return launch_grouped_dev_nvfp4(pr, stream);
}

size_t tkg_grouped_dev_scale_bytes(int groups, int m_capacity, int k, int block) {
  if (groups < 1 || m_capacity < 0) return 0;
  return tkg_scale_bytes(m_capacity, k, block) + size_t(groups) * tkg_scale_bytes(128, k, block);
}

size_t tkg_grouped_scale_bytes(int groups, const int* m_sizes, int k, int block) {
  if (groups < 1 || !m_sizes) return 0;
  size_t total = 0;
  for (int g = 0; g < groups; ++g) {
    if (m_sizes[g] < 0) return 0;
    total += tkg_scale_bytes(m_sizes[g], k, block);
  }
  return total;
}

tkg_status tkg_get_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TKG_ERR_CUDA;
  unsigned int h = 0;
  // the library's word exists once an allocating entry point has run on this
  // device; before that no kernel can have set it, and nothing is allocated here
  if (unsigned int* w = existing_status_word()) {
    if (cudaMemcpyAsync(&h, w, sizeof h, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return TKG_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TKG_ERR_CUDA;
    if (h != 0) {
      if (cudaMemsetAsync(w, 0, sizeof h, stream) != cudaSuccess) return TKG_ERR_CUDA;
      if (cudaStreamSynchronize(stream) != cudaSuccess) return TKG_ERR_CUDA;
    }
  }
  // the allocation-free entry point's word, in its fixed array
  unsigned int h2 = 0;
  if (noalloc_take_status(stream, &h2) != TKG_OK) return TKG_ERR_CUDA;
  h |= h2;
  if (h == 0) return TKG_OK;
  if (h & DEV_ERR_TIMEOUT) return TKG_ERR_TIMEOUT;
  return (h & DEV_ERR_CHECK) ? TKG_ERR_CHECK : TKG_ERR_CUDA;
}

const char* tkg_status_string(tkg_status s) {
  switch (s) {
    case TKG_OK: return "ok";
    case TKG_ERR_INVALID_ARG: return "invalid argument";
    case TKG_ERR_ALIGNMENT: return "misaligned pointer or row pitch";
    case TKG_ERR_UNSUPPORTED: return "unsupported shape";
    case TKG_ERR_CUDA: return "CUDA error";
    case TKG_ERR_TIMEOUT: return "device wait timed out";
    case TKG_ERR_CHECK: return "internal check failed";
  }
  return "unknown status";
}

size_t tkg_scale_bytes(int rows, int k, int block) {
  if (rows < 0 || k < 0 || (block != 16 && block != 32)) return 0;
  const size_t rpad = size_t(ceil_div(rows, 128)) * 128;
  const size_t kbpad = size_t(ceil_div(ceil_div(k, block), 4)) * 4;
  return rpad * kbpad;
}

tkg_status tkg_set_option(tkg_option o, int value) {
  const int i = int(o);
  if (i <= 0 || i > int(TKG_OPT_EPILOGUE_STORE) || value < 0) return TKG_ERR_INVALID_ARG;
  if (o == TKG_OPT_CTA_GROUP && value > 2) return TKG_ERR_INVALID_ARG;
  g_opts[i].store(value, std::memory_order_relaxed);
  return TKG_OK;
}

int tkg_get_option(tkg_option o) { return option(o); }

}  // extern "C"
