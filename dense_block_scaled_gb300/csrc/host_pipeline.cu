// host_pipeline.cu -- tkg_gemm_bf16_from_host: the BF16 GEMM on operands that
// live in host memory, with the copies overlapped with the GEMM.
//
// B goes to the device first (every output row needs all of it); A then
// follows in bands of rows on a copy stream while the GEMM of the previous
// band runs on the caller's stream, and each band of D goes back on a second
// copy stream as soon as its GEMM is done.  The two copy directions run at the
// same time, so a step costs about B's copy plus the GEMM plus one band of D,
// instead of the sum of all copies and the GEMM.
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.cuh"

namespace tkg {
namespace {

constexpr int kMaxBands = 8;
constexpr int kMinBandRows = 2048;

struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;   // host->device, device->host
  cudaEvent_t start, b_ready, out_done;
  cudaEvent_t a_ready[kMaxBands], c_done[kMaxBands];
};

std::mutex g_pipe_mu;   // guards the per-device pipes and serialises enqueueing
Pipe g_pipe[64];

// Streams and events of the current device, created on first use (held until
// the process exits).  Called with g_pipe_mu held.
tkg_status pipe_for_current_device(Pipe** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TKG_ERR_CUDA;
  Pipe& p = g_pipe[dev];
  if (!p.ready) {
    const unsigned flags = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, flags) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.b_ready, flags) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.out_done, flags) == cudaSuccess;
    for (int i = 0; ok && i < kMaxBands; ++i)
      ok = cudaEventCreateWithFlags(&p.a_ready[i], flags) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.c_done[i], flags) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return TKG_ERR_CUDA;
    }
    p.ready = true;
  }
  *out = &p;
  return TKG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tkg

using namespace tkg;

extern "C" tkg_status tkg_gemm_bf16_from_host(int m, int n, int k, const void* A_host, const void* B_host,
                                              void* D_host, void* A_dev, void* B_dev, void* D_dev, float alpha,
                                              cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0) return TKG_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return TKG_OK;
  if (!D_host || !D_dev) return TKG_ERR_INVALID_ARG;
  if (!aligned16(D_dev) || (n % 8) != 0) return TKG_ERR_ALIGNMENT;
  const size_t d_row = size_t(n) * 2;
  if (k == 0) {   // empty sum: D = 0
    if (cudaMemsetAsync(D_dev, 0, size_t(m) * d_row, stream) != cudaSuccess ||
        cudaMemcpyAsync(D_host, D_dev, size_t(m) * d_row, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return TKG_ERR_CUDA;
    return TKG_OK;
  }
  if (!A_host || !B_host || !A_dev || !B_dev) return TKG_ERR_INVALID_ARG;
  if (!aligned16(A_dev) || !aligned16(B_dev) || (k % 8) != 0) return TKG_ERR_ALIGNMENT;

  // bands of at least kMinBandRows rows (a multiple of 256), at most kMaxBands
  int bands = m / kMinBandRows;
  if (bands < 1) bands = 1;
  if (bands > kMaxBands) bands = kMaxBands;
  const int band_rows = ceil_div(ceil_div(m, bands), 256) * 256;
  bands = ceil_div(m, band_rows);
  const size_t a_row = size_t(k) * 2;

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  Pipe* pp = nullptr;
  tkg_status st = pipe_for_current_device(&pp);
  if (st != TKG_OK) return st;
  Pipe& p = *pp;
  auto fail = [] {
    cudaGetLastError();
    return TKG_ERR_CUDA;
  };
  // everything starts after the work already queued on the caller's stream
  if (cudaEventRecord(p.start, stream) != cudaSuccess || cudaStreamWaitEvent(p.in, p.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p.out, p.start, 0) != cudaSuccess)
    return fail();
  if (cudaMemcpyAsync(B_dev, B_host, size_t(n) * a_row, cudaMemcpyHostToDevice, p.in) != cudaSuccess ||
      cudaEventRecord(p.b_ready, p.in) != cudaSuccess)
    return fail();
  for (int i = 0; i < bands; ++i) {
    const int r0 = i * band_rows;
    const int rows = m - r0 < band_rows ? m - r0 : band_rows;
    if (cudaMemcpyAsync(static_cast<char*>(A_dev) + size_t(r0) * a_row,
                        static_cast<const char*>(A_host) + size_t(r0) * a_row, size_t(rows) * a_row,
                        cudaMemcpyHostToDevice, p.in) != cudaSuccess ||
        cudaEventRecord(p.a_ready[i], p.in) != cudaSuccess)
      return fail();
  }
  if (cudaStreamWaitEvent(stream, p.b_ready, 0) != cudaSuccess) return fail();
  for (int i = 0; i < bands; ++i) {
    const int r0 = i * band_rows;
    const int rows = m - r0 < band_rows ? m - r0 : band_rows;
    if (cudaStreamWaitEvent(stream, p.a_ready[i], 0) != cudaSuccess) return fail();
    Problem pr{rows, n, k, static_cast<const char*>(A_dev) + size_t(r0) * a_row, B_dev, nullptr, nullptr, nullptr,
               nullptr, static_cast<char*>(D_dev) + size_t(r0) * d_row, alpha};
    if ((st = launch_bf16(pr, stream)) != TKG_OK) return st;
    if (cudaEventRecord(p.c_done[i], stream) != cudaSuccess || cudaStreamWaitEvent(p.out, p.c_done[i], 0) != cudaSuccess)
      return fail();
    if (cudaMemcpyAsync(static_cast<char*>(D_host) + size_t(r0) * d_row,
                        static_cast<const char*>(D_dev) + size_t(r0) * d_row, size_t(rows) * d_row,
                        cudaMemcpyDeviceToHost, p.out) != cudaSuccess)
      return fail();
  }
  // the caller's stream resumes once D is back in host memory
  if (cudaEventRecord(p.out_done, p.out) != cudaSuccess || cudaStreamWaitEvent(stream, p.out_done, 0) != cudaSuccess)
    return fail();
  return TKG_OK;
}
