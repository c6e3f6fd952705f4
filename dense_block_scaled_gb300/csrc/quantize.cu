// quantize.cu -- FP32 -> MXFP8 / NVFP4 quantisers and the row-major -> tiled
// scale-layout conversion.  All HBM-bound: 16-byte loads, several in flight per
// thread, one wave of resident blocks.
//
// Quantisation rules are those of the workload definition (MXFP8: E8M0 scale
// 2^ceil(log2(amax/448)) per 1x32 block, E4M3 RNE saturating; NVFP4: FP32
// tensor scale amax/(6*448), E4M3 block scale blockamax/(6*tensor scale) per
// 1x16 block, E2M1 RNE), for the MXFP8/NVFP4 formats of "ThunderKittens 2.0
// GPU Kernel优化" (table of updates).  Every FP32 step is one IEEE operation
// with round-to-nearest (explicit __f*_rn intrinsics, never contracted); the
// NVFP4 element quotients take a shortcut that provably gives the same codes
// (e2m1_quotients).
#include <cuda_runtime.h>

#include <cstdint>

#include "host_common.cuh"

namespace tkg {

// Byte offset of scale (r, kb) in the tiled layout (include/tkg_gemm.h).
__device__ __forceinline__ size_t sf_tiled_offset(int r, int kb, int ka) {
  return (size_t(r >> 7) * size_t(ka) + size_t(kb >> 2)) * 512u + size_t(r & 31) * 16u +
         size_t((r & 127) >> 5) * 4u + size_t(kb & 3);
}

// Two FP32 -> E4M3 (RNE, saturating); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two FP32 -> E2M1 (RNE, saturating); `lo` lands in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Value of a non-negative E4M3 code (bias 7, 3 mantissa bits, subnormals m * 2^-9).
__device__ __forceinline__ float e4m3_value(uint32_t s) {
  const uint32_t e = (s >> 3) & 0xFu, m = s & 7u;
  if (e == 0) return __fmul_rn(float(m), 1.0f / 512.0f);
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// MXFP8 scale exponent: smallest e with 448 * 2^e >= amax, clamped to [-127, 127].
// With amax = M * 2^E (M in [1, 2)), 448 = 1.75 * 2^8, that is
// e = E - 8 + (M > 1.75); subnormal or zero amax gives -127.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax);
  const int eb = int((u >> 23) & 0xFFu);
  if (eb == 0) return -127;
  int e = (eb - 127) - 8 + (((u & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Each warp walks its own contiguous range of passes, and every lane keeps the
// (row, K-block) of the block it works on up to date by addition, so the loop
// holds no integer division.  When k/bs is a multiple of 4, the four scale
// bytes of blocks kb..kb+3 (kb % 4 == 0) of a row are adjacent in the tiled
// layout and go out as one 32-bit store.
struct WarpRange {
  long long p0, p1;   // passes [p0, p1) of this warp
};
__device__ __forceinline__ WarpRange warp_range(long long passes, int unroll) {
  const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long per = ((passes + nwarps - 1) / nwarps + unroll - 1) / unroll * unroll;
  const long long p0 = warp * per;
  return {p0, p0 + per < passes ? p0 + per : passes};
}

// MXFP8: each lane takes 8 consecutive elements (two adjacent float4), so a
// 32-element block spans 4 lanes and a warp pass covers 8 blocks (1 KB of X);
// four passes per loop trip, all loads issued before any arithmetic.  Fewer
// shuffles and conversions per element than 4 elements a lane matter once the
// power cap lowers the clock (the kernel is then issue-bound).
constexpr int kMxUnroll = 4;

__global__ void __launch_bounds__(256) quant_mxfp8_kernel(long long nblk, int kblk, const float* __restrict__ X,
                                                          uint8_t* __restrict__ Q, uint8_t* __restrict__ SF,
                                                          int ka) {
  const int lane = threadIdx.x & 31;
  const WarpRange wr = warp_range((nblk + 7) / 8, kMxUnroll);
  if (wr.p0 >= wr.p1) return;
  const bool packed_sf = (kblk & 3) == 0;
  long long b = wr.p0 * 8 + (lane >> 2);   // this lane's block
  int r = int(b / kblk), kb = int(b - (long long)r * kblk);
  for (long long p = wr.p0; p < wr.p1; p += kMxUnroll) {
    float4 x[kMxUnroll][2];
#pragma unroll
    for (int u = 0; u < kMxUnroll; ++u) {
      const long long bu = b + 8 * u;
      const float4* src = reinterpret_cast<const float4*>(X + bu * 32 + 8 * (lane & 3));
      x[u][0] = bu < nblk ? __ldcs(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      x[u][1] = bu < nblk ? __ldcs(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kMxUnroll; ++u) {
      float a = fmaxf(fmaxf(fmaxf(fabsf(x[u][0].x), fabsf(x[u][0].y)), fmaxf(fabsf(x[u][0].z), fabsf(x[u][0].w))),
                      fmaxf(fmaxf(fabsf(x[u][1].x), fabsf(x[u][1].y)), fmaxf(fabsf(x[u][1].z), fabsf(x[u][1].w))));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
      const int e = mx_exponent(a);
      const float inv = __uint_as_float(uint32_t(127 - e) << 23);   // 2^-e, a normal float for e in [-127, 120]
      const uint32_t code = uint32_t(e + 127);
      // scale bytes of blocks kb..kb+3, gathered in lanes 0 and 16
      const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 4);
      const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 8);
      const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 12);
      if (b < nblk) {
        const uint32_t w0 = cvt_e4m3x2(__fmul_rn(x[u][0].x, inv), __fmul_rn(x[u][0].y, inv)) |
                            (cvt_e4m3x2(__fmul_rn(x[u][0].z, inv), __fmul_rn(x[u][0].w, inv)) << 16);
        const uint32_t w1 = cvt_e4m3x2(__fmul_rn(x[u][1].x, inv), __fmul_rn(x[u][1].y, inv)) |
                            (cvt_e4m3x2(__fmul_rn(x[u][1].z, inv), __fmul_rn(x[u][1].w, inv)) << 16);
        *reinterpret_cast<uint2*>(Q + b * 32 + 8 * (lane & 3)) = make_uint2(w0, w1);
        if (packed_sf) {
          if ((lane & 15) == 0)
            *reinterpret_cast<uint32_t*>(SF + sf_tiled_offset(r, kb, ka)) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
        } else if ((lane & 3) == 0) {
          SF[sf_tiled_offset(r, kb, ka)] = uint8_t(code);
        }
      }
      b += 8;
      kb += 8;
      while (kb >= kblk) {
        kb -= kblk;
        ++r;
      }
    }
  }
}

// amax over the whole tensor, as the bits of a non-negative float (monotone as unsigned).
constexpr int kAmaxUnroll = 4;
__global__ void __launch_bounds__(256) amax_kernel(long long n4, const float* __restrict__ X,
                                                   unsigned int* __restrict__ out) {
  float a = 0.f;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; i0 < n4; i0 += stride * kAmaxUnroll) {
    float4 x[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      const long long i = i0 + u * stride;
      x[u] = i < n4 ? __ldg(reinterpret_cast<const float4*>(X) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u)
      a = fmaxf(a, fmaxf(fmaxf(fabsf(x[u].x), fabsf(x[u].y)), fmaxf(fabsf(x[u].z), fabsf(x[u].w))));
  }
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x < 32) {
    float b = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 4; o > 0; o >>= 1) b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    if (threadIdx.x == 0) atomicMax(out, __float_as_uint(b));
  }
}

// t = amax / (6 * 448), in place.
__global__ void tensor_scale_kernel(unsigned int* __restrict__ word) {
  const float amax = __uint_as_float(*word);
  *reinterpret_cast<float*>(word) = __fdiv_rn(amax, 2688.0f);
}

// E2M1 codes of x0/den and x1/den (IEEE quotients), `x0` in the low nibble.
// The quotient is first taken as x * rcp.approx(den): rcp.approx is within 1
// ulp of 1/den for the normal den given here, so x * r lies within about 2^-22
// (relative) of the correctly rounded quotient.  Rounding to E2M1 is monotone,
// so if q * (1 - 2^-18) and q * (1 + 2^-18) round to the same code, so does the
// IEEE quotient, which lies between them; otherwise (a quotient within 2^-18 of
// a rounding boundary, where a tie may be at stake) the IEEE division decides.
__device__ __forceinline__ uint32_t e2m1_quotients(float x0, float x1, float den, float r) {
  const float q0 = x0 * r, q1 = x1 * r;
  constexpr float kLo = 1.0f - 1.0f / 262144.0f, kHi = 1.0f + 1.0f / 262144.0f;
  const uint32_t c_lo = cvt_e2m1x2(q0 * kLo, q1 * kLo);
  const uint32_t c_hi = cvt_e2m1x2(q0 * kHi, q1 * kHi);
  if (c_lo == c_hi) return c_lo;
  return cvt_e2m1x2(__fdiv_rn(x0, den), __fdiv_rn(x1, den));
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// NVFP4: one lane per 16-element block (its 64 bytes in four float4 loads), so
// the block amax, the block scale and the reciprocal are computed once per
// block; a warp pass covers 32 consecutive blocks (2 KB of X), two passes per
// loop trip.
constexpr int kNvUnroll = 2;

__global__ void __launch_bounds__(256) quant_nvfp4_kernel(long long nblk, int kblk, const float* __restrict__ X,
                                                          uint8_t* __restrict__ Q, uint8_t* __restrict__ SF, int ka,
                                                          const float* __restrict__ tptr) {
  const int lane = threadIdx.x & 31;
  const WarpRange wr = warp_range((nblk + 31) / 32, kNvUnroll);
  if (wr.p0 >= wr.p1) return;
  const bool packed_sf = (kblk & 3) == 0;
  const float t = __ldg(tptr);
  const float d = __fmul_rn(6.0f, t);
  long long b = wr.p0 * 32 + lane;   // this lane's block
  int r = int(b / kblk), kb = int(b - (long long)r * kblk);
  for (long long p = wr.p0; p < wr.p1; p += kNvUnroll) {
    float4 x[kNvUnroll][4];
#pragma unroll
    for (int u = 0; u < kNvUnroll; ++u) {
      const long long bu = b + 32 * u;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        x[u][j] = bu < nblk ? __ldcs(reinterpret_cast<const float4*>(X + bu * 16) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kNvUnroll; ++u) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        a = fmaxf(a, fmaxf(fmaxf(fabsf(x[u][j].x), fabsf(x[u][j].y)), fmaxf(fabsf(x[u][j].z), fabsf(x[u][j].w))));
      uint32_t s = 0;
      float den = 0.f;
      if (t > 0.f) {
        s = cvt_e4m3x2(__fdiv_rn(a, d), 0.f) & 0xFFu;
        den = __fmul_rn(e4m3_value(s), t);
      }
      // scale bytes of blocks kb..kb+3, gathered in lanes 0, 4, ...
      const uint32_t s1 = __shfl_down_sync(0xffffffffu, s, 1);
      const uint32_t s2 = __shfl_down_sync(0xffffffffu, s, 2);
      const uint32_t s3 = __shfl_down_sync(0xffffffffu, s, 3);
      if (b < nblk) {
        uint32_t w[2] = {0u, 0u};
        if (den > 0.f) {
          // 2^-124 <= den keeps 1/den a finite normal float
          const bool fast = den >= 4.7019774e-38f;
          const float rr = rcp_approx(den);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t lo = fast ? e2m1_quotients(x[u][j].x, x[u][j].y, den, rr)
                                     : cvt_e2m1x2(__fdiv_rn(x[u][j].x, den), __fdiv_rn(x[u][j].y, den));
            const uint32_t hi = fast ? e2m1_quotients(x[u][j].z, x[u][j].w, den, rr)
                                     : cvt_e2m1x2(__fdiv_rn(x[u][j].z, den), __fdiv_rn(x[u][j].w, den));
            w[j >> 1] |= (lo | (hi << 8)) << (16 * (j & 1));
          }
        }
        *reinterpret_cast<uint2*>(Q + b * 8) = make_uint2(w[0], w[1]);
        if (packed_sf) {
          if ((lane & 3) == 0)
            *reinterpret_cast<uint32_t*>(SF + sf_tiled_offset(r, kb, ka)) = s | (s1 << 8) | (s2 << 16) | (s3 << 24);
        } else {
          SF[sf_tiled_offset(r, kb, ka)] = uint8_t(s);
        }
      }
      b += 32;
      kb += 32;
      while (kb >= kblk) {
        kb -= kblk;
        ++r;
      }
    }
  }
}

__global__ void __launch_bounds__(256) scales_to_tiled_kernel(int rows, int kblocks, const uint8_t* __restrict__ src,
                                                              int ld, uint8_t* __restrict__ dst, int ka) {
  const long long n = (long long)rows * kblocks;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
    const int r = int(i / kblocks), kb = int(i % kblocks);
    dst[sf_tiled_offset(r, kb, ka)] = src[(size_t)r * ld + kb];
  }
}

// Blocks for `work_items` threads of `per_block`, capped at one full wave of
// resident blocks (the kernels loop over the rest).
template <typename Kern>
static int grid_for(Kern kern, long long work_items, int per_block) {
  int sms = 148;
  device_sm_count(&sms);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, per_block, 0) != cudaSuccess || per_sm <= 0) {
    cudaGetLastError();
    per_sm = 4;
  }
  long long want = (work_items + per_block - 1) / per_block;
  long long cap = (long long)sms * per_sm;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return int(want);
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace tkg

using namespace tkg;

extern "C" {

tkg_status tkg_quantize_mxfp8(int rows, int k, const float* X, void* Q, void* sf, cudaStream_t stream) {
  if (rows < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (rows == 0 || k == 0) return TKG_OK;
  if (!X || !Q || !sf) return TKG_ERR_INVALID_ARG;
  if (k % 32 != 0 || !aligned(X, 16) || !aligned(Q, 16) || !aligned(sf, 16)) return TKG_ERR_ALIGNMENT;
  const int kblk = k / 32, ka = (kblk + 3) / 4;
  if (cudaMemsetAsync(sf, 0, tkg_scale_bytes(rows, k, 32), stream) != cudaSuccess) return TKG_ERR_CUDA;
  const long long nblk = (long long)rows * kblk;
  const int grid = grid_for(quant_mxfp8_kernel, ((nblk + 7) / 8 + kMxUnroll - 1) / kMxUnroll * 32, 256);
  quant_mxfp8_kernel<<<grid, 256, 0, stream>>>(
      nblk, kblk, X, static_cast<uint8_t*>(Q), static_cast<uint8_t*>(sf), ka);
  return cudaGetLastError() == cudaSuccess ? TKG_OK : TKG_ERR_CUDA;
}

tkg_status tkg_quantize_nvfp4(int rows, int k, const float* X, void* Q, void* sf, float* tensor_scale,
                              cudaStream_t stream) {
  if (rows < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (!tensor_scale) return TKG_ERR_INVALID_ARG;
  if (!aligned(tensor_scale, 4)) return TKG_ERR_ALIGNMENT;
  if (cudaMemsetAsync(tensor_scale, 0, sizeof(float), stream) != cudaSuccess) return TKG_ERR_CUDA;
  if (rows == 0 || k == 0) return TKG_OK;
  if (!X || !Q || !sf) return TKG_ERR_INVALID_ARG;
  if (k % 32 != 0 || !aligned(X, 16) || !aligned(Q, 16) || !aligned(sf, 16)) return TKG_ERR_ALIGNMENT;
  const int kblk = k / 16, ka = (kblk + 3) / 4;
  if (cudaMemsetAsync(sf, 0, tkg_scale_bytes(rows, k, 16), stream) != cudaSuccess) return TKG_ERR_CUDA;
  unsigned int* word = reinterpret_cast<unsigned int*>(tensor_scale);
  const long long n4 = (long long)rows * k / 4;
  amax_kernel<<<grid_for(amax_kernel, (n4 + kAmaxUnroll - 1) / kAmaxUnroll, 256), 256, 0, stream>>>(n4, X, word);
  tensor_scale_kernel<<<1, 1, 0, stream>>>(word);
  const long long nblk = (long long)rows * kblk;
  const int grid = grid_for(quant_nvfp4_kernel, ((nblk + 31) / 32 + kNvUnroll - 1) / kNvUnroll * 32, 256);
  quant_nvfp4_kernel<<<grid, 256, 0, stream>>>(
      nblk, kblk, X, static_cast<uint8_t*>(Q), static_cast<uint8_t*>(sf), ka, tensor_scale);
  return cudaGetLastError() == cudaSuccess ? TKG_OK : TKG_ERR_CUDA;
}

tkg_status tkg_quantize_nvfp4_scaled(int rows, int k, const float* X, void* Q, void* sf, const float* tensor_scale,
                                     cudaStream_t stream) {
  if (rows < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (!tensor_scale) return TKG_ERR_INVALID_ARG;
  if (!aligned(tensor_scale, 4)) return TKG_ERR_ALIGNMENT;
  if (rows == 0 || k == 0) return TKG_OK;
  if (!X || !Q || !sf) return TKG_ERR_INVALID_ARG;
  if (k % 32 != 0 || !aligned(X, 16) || !aligned(Q, 16) || !aligned(sf, 16)) return TKG_ERR_ALIGNMENT;
  const int kblk = k / 16, ka = (kblk + 3) / 4;
  if (cudaMemsetAsync(sf, 0, tkg_scale_bytes(rows, k, 16), stream) != cudaSuccess) return TKG_ERR_CUDA;
  const long long nblk = (long long)rows * kblk;
  const int grid = grid_for(quant_nvfp4_kernel, ((nblk + 31) / 32 + kNvUnroll - 1) / kNvUnroll * 32, 256);
  quant_nvfp4_kernel<<<grid, 256, 0, stream>>>(
      nblk, kblk, X, static_cast<uint8_t*>(Q), static_cast<uint8_t*>(sf), ka, tensor_scale);
  return cudaGetLastError() == cudaSuccess ? TKG_OK : TKG_ERR_CUDA;
}

tkg_status tkg_scales_to_tiled(int rows, int kblocks, const void* src, int ld, void* dst, cudaStream_t stream) {
  if (rows < 0 || kblocks < 0 || ld < kblocks) return TKG_ERR_INVALID_ARG;
  if (rows == 0 || kblocks == 0) return TKG_OK;
  if (!src || !dst) return TKG_ERR_INVALID_ARG;
  const int ka = (kblocks + 3) / 4;
  const size_t bytes = size_t((rows + 127) / 128) * 128 * size_t(ka) * 4;
  if (cudaMemsetAsync(dst, 0, bytes, stream) != cudaSuccess) return TKG_ERR_CUDA;
  const long long n = (long long)rows * kblocks;
  scales_to_tiled_kernel<<<grid_for(scales_to_tiled_kernel, n, 256), 256, 0, stream>>>(
      rows, kblocks, static_cast<const uint8_t*>(src), ld, static_cast<uint8_t*>(dst), ka);
  return cudaGetLastError() == cudaSuccess ? TKG_OK : TKG_ERR_CUDA;
}

}  // extern "C"
