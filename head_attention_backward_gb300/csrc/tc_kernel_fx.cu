// The tensor-core backward kernel (tc_kernel.cuh) instantiated with the
// attention bias, dbias and dropout extras (TransformerEngine PR #446: the
// bias shapes and the philox seed / offset of ck_attn_bwd).  A translation
// unit of its own so that it compiles beside the plain instantiations.
#include "tc_kernel.cuh"

namespace attn {

int launch_bwd_tc_fx(const Problem& P, cudaStream_t st) {
  if (P.dtype == ATTN_FP16) return tc::launch_mode<__half, true>(P, st);
  return tc::launch_mode<__nv_bfloat16, true>(P, st);
}

}  // namespace attn
