// gemm_grouped.cu -- grouped GEMM instantiations: groups of rows of A, each
// against its own N x K matrix of a stacked B (the expert layers of a
// mixture-of-experts model).  Same persistent kernel as the plain GEMM, with a
// per-call group table mapping output tiles to groups.
#include "host_common.cuh"

namespace tkg {

tkg_status launch_grouped_bf16(const Problem& pr, cudaStream_t s) {
  if (option(TKG_OPT_CTA_GROUP) == 1) return launch_sched<FMT_BF16, 1, 256, 4, 2, 1>(pr, s);
  return launch_sched<FMT_BF16, 2, 256, 6, 2, 1>(pr, s);
}

tkg_status launch_grouped_mxfp8(const Problem& pr, cudaStream_t s) {
  if (option(TKG_OPT_CTA_GROUP) == 1) return launch_sched<FMT_MXFP8, 1, 256, 4, 1, 1>(pr, s);
  return launch_sched<FMT_MXFP8, 2, 256, 6, 1, 1>(pr, s);
}

tkg_status launch_grouped_nvfp4(const Problem& pr, cudaStream_t s) {
  if (option(TKG_OPT_CTA_GROUP) == 1) return launch_sched<FMT_NVFP4, 1, 256, 3, 1, 1>(pr, s);
  return launch_sched<FMT_NVFP4, 2, 256, 5, 1, 1>(pr, s);
}

// Device-resident group sizes: the shared-memory group table takes 2 KB, so
// these run one stage fewer than the host-table versions.
tkg_status launch_grouped_dev_bf16(const Problem& pr, cudaStream_t s) {
  return launch_sched<FMT_BF16, 2, 256, 5, 2, 2>(pr, s);
}

tkg_status launch_grouped_dev_mxfp8(const Problem& pr, cudaStream_t s) {
  return launch_sched<FMT_MXFP8, 2, 256, 5, 1, 2>(pr, s);
}

tkg_status launch_grouped_dev_nvfp4(const Problem& pr, cudaStream_t s) {
  return launch_sched<FMT_NVFP4, 2, 256, 4, 1, 2>(pr, s);
}

}  // namespace tkg
