// Block-scaled MXFP4 GEMM (kind::mxf4): not yet built.
#include "kernels.h"

namespace gp {
int mxf4_gemm_launch(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, TcParams, int, cudaStream_t) {
  return GP_ERR_UNSUPPORTED;
}
}  // namespace gp
