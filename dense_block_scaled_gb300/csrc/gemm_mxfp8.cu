// gemm_mxfp8.cu -- MXFP8 instantiations of the persistent tcgen05 GEMM and the choice
// between them.  Separate translation unit so the three formats compile in parallel.
#include "host_common.cuh"

namespace tkg {

tkg_status launch_mxfp8(const Problem& pr, cudaStream_t s) {
  const int cg = option(TKG_OPT_CTA_GROUP);
  if (option(TKG_OPT_SINGLE_STAGE)) return launch_gemm<FMT_MXFP8, 2, 256, 1, 1>(pr, s);
  if (cg == 1) return launch_gemm<FMT_MXFP8, 1, 256, 3, 1>(pr, s);
  return launch_gemm<FMT_MXFP8, 2, 256, 5, 1>(pr, s);
}

}  // namespace tkg
