// gemm_mxfp8.cu -- MXFP8 instantiations of the persistent tcgen05 GEMM and the choice
// between them.  Separate translation unit so the three formats compile in parallel.
#include "host_common.cuh"

namespace tkg {

tkg_status launch_mxfp8(const Problem& pr, cudaStream_t s) {
  // One 256-column accumulator: tensor memory (512 columns) cannot hold two
  // next to the scale regions.  The epilogue frees it as soon as it is in
  // registers, so the next tile's MMAs wait only for that drain.
  const int cg = option(TKG_OPT_CTA_GROUP);
  // few output tiles (skinny M): split K across a cluster
  const int split = choose_split(pr, FmtTraits<FMT_MXFP8>::kStageK);
  if (split >= 2 && pr.m <= 32) {
    // short A tiles leave room for a deeper B pipeline (the deepest that fits,
    // 10 stages, ran 0.5-1.6% slower at M = 1 and 16)
    if (split == 2) return launch_splitk<FMT_MXFP8, 2, 9, 32>(pr, s);
    return launch_splitk<FMT_MXFP8, 3, 9, 32>(pr, s);
  }
  if (split == 2) return launch_splitk<FMT_MXFP8, 2, 6>(pr, s);
  if (split == 3) return launch_splitk<FMT_MXFP8, 3, 6>(pr, s);
  if (option(TKG_OPT_SINGLE_STAGE)) return launch_sched<FMT_MXFP8, 2, 256, 1, 1>(pr, s);
  if (cg == 1) return launch_sched<FMT_MXFP8, 1, 256, 4, 1>(pr, s);
  return launch_sched<FMT_MXFP8, 2, 256, 6, 1>(pr, s);
}

}  // namespace tkg
