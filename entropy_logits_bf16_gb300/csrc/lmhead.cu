// rlk_lmhead_logprob: the fused LM-head path (tensor-core GEMM tiles folded
// into the online log-sum-exp / entropy state).  Not built yet: the entry
// point reports RLK_ERR_UNSUPPORTED.

#include "internal.h"

namespace rlk {

size_t lmhead_workspace_bytes(int64_t T, int64_t V, int64_t H) {
  (void)T;
  (void)V;
  (void)H;
  return 0;
}

cudaError_t launch_lmhead(const LmheadArgs& a, cudaStream_t stream) {
  (void)a;
  (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace rlk
