// gemm_bf16.cu -- BF16 instantiations of the persistent tcgen05 GEMM and the choice
// between them.  Separate translation unit so the three formats compile in parallel.
#include "host_common.cuh"

namespace tkg {

tkg_status launch_bf16(const Problem& pr, cudaStream_t s) {
  // All of N in one 256-column tile: single-CTA tiles (tall, narrow GEMMs ran
  // 1.6x faster on them than on CTA pairs, which gain nothing there)
  const int cg_opt = option(TKG_OPT_CTA_GROUP);
  const int cg = cg_opt != 0 ? cg_opt : (pr.n <= 256 ? 1 : 2);
  // few output tiles (skinny M): split K across a cluster
  const int split = choose_split(pr, FmtTraits<FMT_BF16>::kStageK);
  if (split >= 2 && pr.m <= 32) {
    // short A tiles leave room for a deeper B pipeline (the deepest that fits,
    // 11 stages, ran 0.5-1.6% slower at M = 1 and 16)
    if (split == 2) return launch_splitk<FMT_BF16, 2, 9, 32>(pr, s);
    return launch_splitk<FMT_BF16, 3, 9, 32>(pr, s);
  }
  if (split == 2) return launch_splitk<FMT_BF16, 2, 7>(pr, s);
  if (split == 3) return launch_splitk<FMT_BF16, 3, 7>(pr, s);
  if (option(TKG_OPT_SINGLE_STAGE)) return launch_sched<FMT_BF16, 2, 256, 1, 2>(pr, s);
  if (cg != 1 && option(TKG_OPT_ACC_STAGES) != 1 && use_dual_bf16(pr))
    return launch_sched<FMT_BF16, 2, 512, 4, 1>(pr, s);
  if (cg == 1) return launch_sched<FMT_BF16, 1, 256, 4, 2>(pr, s);
  if (option(TKG_OPT_ACC_STAGES) == 1) return launch_sched<FMT_BF16, 2, 256, 6, 1>(pr, s);
  return launch_sched<FMT_BF16, 2, 256, 6, 2>(pr, s);
}

}  // namespace tkg
