// host_pipeline.cu -- tkg_gemm_bf16_from_host: the BF16 GEMM on operands that
// live in host memory, with the copies overlapped with the GEMM.
//
// Both operands go to the device in bands of rows on one copy stream, A and B
// alternating so that the copied fractions of the two stay level.  Every
// copied band unlocks one rectangle of D: a band of A against the B bands
// already on the device, or a band of B against the A bands already there.
// Each rectangle is one GEMM launch on the caller's stream, queued behind its
// band's copy, and goes back to host memory on a second copy stream as soon
// as that launch is done.  The GEMM thus starts after one band of each
// operand instead of after all of B, and the step ends one rectangle (one
// band of B against all of A) after the last copy.
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.cuh"

namespace tkg {
namespace {

constexpr int kMaxBands = 8;          // per operand
constexpr int kMinBandRows = 2048;

struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;   // host->device, device->host
  cudaEvent_t start, out_done;
  cudaEvent_t landed[2 * kMaxBands];          // one per band copy, in copy order
  cudaEvent_t piece_done[2 * kMaxBands];      // one per rectangle of D
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
              cudaEventCreateWithFlags(&p.out_done, flags) == cudaSuccess;
    for (int i = 0; ok && i < 2 * kMaxBands; ++i)
      ok = cudaEventCreateWithFlags(&p.landed[i], flags) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.piece_done[i], flags) == cudaSuccess;
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

// `total` rows in `count` bands of `rows` rows (a multiple of `align`; the
// last band may be shorter): bands of at least kMinBandRows, at most kMaxBands.
struct Bands {
  int count, rows;
};
Bands split_rows(int total, int align) {
  int c = total / kMinBandRows;
  if (c < 1) c = 1;
  if (c > kMaxBands) c = kMaxBands;
  const int rows = ceil_div(ceil_div(total, c), align) * align;
  return Bands{ceil_div(total, rows), rows};
}

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

  // A bands whole pair tiles (256 rows), B bands whole dual-accumulate tiles
  // (512 rows), so only the last band of each leaves ragged tiles
  const Bands ba = split_rows(m, 256), bb = split_rows(n, 512);
  const size_t op_row = size_t(k) * 2;

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
  // (which, for an earlier call on the same staging buffers, ends when its D
  // is back in host memory)
  if (cudaEventRecord(p.start, stream) != cudaSuccess || cudaStreamWaitEvent(p.in, p.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p.out, p.start, 0) != cudaSuccess)
    return fail();

  int na = 0, nb = 0, copies = 0, pieces = 0;   // bands of A / B on the device
  while (na < ba.count || nb < bb.count) {
    // next: the operand whose copied fraction is smaller (B on a tie)
    const bool take_b =
        nb < bb.count && (na == ba.count || (long long)nb * ba.count <= (long long)na * bb.count);
    int r0, r1, c0, c1;   // the rectangle of D this copy unlocks
    const void* src;
    void* dst;
    size_t bytes;
    if (take_b) {
      c0 = nb * bb.rows;
      c1 = n - c0 < bb.rows ? n : c0 + bb.rows;
      r0 = 0;
      r1 = na * ba.rows < m ? na * ba.rows : m;
      src = static_cast<const char*>(B_host) + size_t(c0) * op_row;
      dst = static_cast<char*>(B_dev) + size_t(c0) * op_row;
      bytes = size_t(c1 - c0) * op_row;
      ++nb;
    } else {
      r0 = na * ba.rows;
      r1 = m - r0 < ba.rows ? m : r0 + ba.rows;
      c0 = 0;
      c1 = nb * bb.rows < n ? nb * bb.rows : n;
      src = static_cast<const char*>(A_host) + size_t(r0) * op_row;
      dst = static_cast<char*>(A_dev) + size_t(r0) * op_row;
      bytes = size_t(r1 - r0) * op_row;
      ++na;
    }
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, p.in) != cudaSuccess ||
        cudaEventRecord(p.landed[copies], p.in) != cudaSuccess)
      return fail();
    if (r1 > r0 && c1 > c0) {
      if (cudaStreamWaitEvent(stream, p.landed[copies], 0) != cudaSuccess) return fail();
      Problem pr{r1 - r0,
                 c1 - c0,
                 k,
                 static_cast<const char*>(A_dev) + size_t(r0) * op_row,
                 static_cast<const char*>(B_dev) + size_t(c0) * op_row,
                 nullptr,
                 nullptr,
                 nullptr,
                 nullptr,
                 static_cast<char*>(D_dev) + size_t(r0) * d_row + size_t(c0) * 2,
                 alpha};
      pr.ldd = n;
      if ((st = launch_bf16(pr, stream)) != TKG_OK) return st;
      if (cudaEventRecord(p.piece_done[pieces], stream) != cudaSuccess ||
          cudaStreamWaitEvent(p.out, p.piece_done[pieces], 0) != cudaSuccess)
        return fail();
      if (cudaMemcpy2DAsync(static_cast<char*>(D_host) + size_t(r0) * d_row + size_t(c0) * 2, d_row,
                            static_cast<const char*>(D_dev) + size_t(r0) * d_row + size_t(c0) * 2, d_row,
                            size_t(c1 - c0) * 2, size_t(r1 - r0), cudaMemcpyDeviceToHost, p.out) != cudaSuccess)
        return fail();
      ++pieces;
    }
    ++copies;
  }
  // the caller's stream resumes once D is back in host memory
  if (cudaEventRecord(p.out_done, p.out) != cudaSuccess || cudaStreamWaitEvent(stream, p.out_done, 0) != cudaSuccess)
    return fail();
  return TKG_OK;
}
