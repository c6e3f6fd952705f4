// gemm_grouped.cu -- grouped GEMM instantiations: groups of rows of A, each
// against its own N x K matrix of a stacked B (the expert layers of a
// mixture-of-experts model).  Same persistent kernel as the plain GEMM, with a
// per-call group table mapping output tiles to groups.
#include "host_common.cuh"

namespace tkg {

// Single-CTA tiles (128 x 256) or CTA pairs (256 x 256).  Automatic: single
// when no group has more than 128 rows (the decode regime of a mixture-of-
// experts layer), where the second CTA of every pair tile would hold no rows:
// 8 experts x 16 rows, N = 4096, K = 7168 measured 71 / 37 / 21 us single
// against 80 / 43 / 25 us in pairs (BF16 / MXFP8 / NVFP4), the 128 tiles
// filling one wave of SMs instead of two uneven waves of pairs.
static bool grouped_single_cta(const Problem& pr) {
  const int cg = option(TKG_OPT_CTA_GROUP);
  if (cg != 0) return cg == 1;
  for (int g = 0; g < pr.groups; ++g)
    if (pr.m_sizes[g] > 128) return false;
  return true;
}

tkg_status launch_grouped_bf16(const Problem& pr, cudaStream_t s) {
  if (grouped_single_cta(pr)) return launch_sched<FMT_BF16, 1, 256, 4, 2, 1>(pr, s);
  return launch_sched<FMT_BF16, 2, 256, 6, 2, 1>(pr, s);
}

tkg_status launch_grouped_mxfp8(const Problem& pr, cudaStream_t s) {
  if (grouped_single_cta(pr)) return launch_sched<FMT_MXFP8, 1, 256, 4, 1, 1>(pr, s);
  return launch_sched<FMT_MXFP8, 2, 256, 6, 1, 1>(pr, s);
}

tkg_status launch_grouped_nvfp4(const Problem& pr, cudaStream_t s) {
  if (grouped_single_cta(pr)) return launch_sched<FMT_NVFP4, 1, 256, 3, 1, 1>(pr, s);
  return launch_sched<FMT_NVFP4, 2, 256, 5, 1, 1>(pr, s);
}

// Device-resident group sizes: the shared-memory group table takes 2 KB, so
// these run one stage fewer than the host-table versions, or keep their stages
// with one epilogue staging buffer per warp (BF16 and MXFP8 single-CTA; BF16
// decode, 8 experts x 16 rows, N=4096, K=7168: 75.2 us at 4 stages against
// 76.6 us at 3 stages with two buffers).  Single-CTA tiles when the row
// capacity is at most 128 (no group can exceed one 128-row tile: the decode
// regime, as for the host-table launch above).
static bool grouped_dev_single_cta(const Problem& pr) {
  const int cg = option(TKG_OPT_CTA_GROUP);
  if (cg != 0) return cg == 1;
  return pr.m <= 128;
}

tkg_status launch_grouped_dev_bf16(const Problem& pr, cudaStream_t s) {
  if (grouped_dev_single_cta(pr)) return launch_sched<FMT_BF16, 1, 256, 4, 2, 2>(pr, s);
  return launch_sched<FMT_BF16, 2, 256, 5, 2, 2>(pr, s);
}

tkg_status launch_grouped_dev_mxfp8(const Problem& pr, cudaStream_t s) {
  if (grouped_dev_single_cta(pr)) return launch_sched<FMT_MXFP8, 1, 256, 4, 1, 2>(pr, s);
  return launch_sched<FMT_MXFP8, 2, 256, 5, 1, 2>(pr, s);
}

tkg_status launch_grouped_dev_nvfp4(const Problem& pr, cudaStream_t s) {
  if (grouped_dev_single_cta(pr)) return launch_sched<FMT_NVFP4, 1, 256, 3, 1, 2>(pr, s);
  return launch_sched<FMT_NVFP4, 2, 256, 4, 1, 2>(pr, s);
}

}  // namespace tkg
