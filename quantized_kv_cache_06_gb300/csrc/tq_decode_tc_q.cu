// Tensor-core paged decode over product-quantised key rows: the GQA-group-8 forms (D 128,
// 2- to 4-bit MSE indices, every V width).  The kernel is in tq_decode_tc.cuh.
#include "tq_decode_tc.cuh"

namespace tq {

cudaError_t launch_tc_prod_g8(const DecodeArgs& a, const DecodePlan& p, const float* p_all, cudaStream_t stream) {
  if (a.head_dim == 128 && a.num_q_heads / a.num_kv_heads == 8) {
    TQ_TCP_V(2, 8) TQ_TCP_V(3, 8) TQ_TCP_V(4, 8)
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
