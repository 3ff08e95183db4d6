// Tensor-core paged decode over product-quantised ("QJL residual") key rows: the host entry
// and the GQA-group-4 forms (D 128, 2- to 4-bit MSE indices, every V width); the group-8
// forms are in tq_decode_tc_q.cu.  The kernel is in tq_decode_tc.cuh; the projection
// p = S q~ comes from tq_qjl.cu.
#include "tq_decode_tc.cuh"

namespace tq {

bool tc_prod_decode_supported(const DecodeArgs& a) {
  const int G = a.num_kv_heads > 0 ? a.num_q_heads / a.num_kv_heads : 0;
  const int mb = a.k_bits - 1;  // a.k_bits: total key bits of the product rows
  return a.head_dim == 128 && a.block_size == kBS && a.num_kv_heads >= 1 && a.num_kv_heads <= 8 &&
         (G == 4 || G == 8) && mb >= 2 && mb <= 4 && a.v_bits >= 2 && a.v_bits <= 5;
}

cudaError_t launch_tc_prod(const DecodeArgs& a, const DecodePlan& p, const float* p_all, cudaStream_t stream) {
  if (a.head_dim == 128 && a.num_q_heads / a.num_kv_heads == 4) {
    TQ_TCP_V(2, 4) TQ_TCP_V(3, 4) TQ_TCP_V(4, 4)
  }
  return launch_tc_prod_g8(a, p, p_all, stream);
}

}  // namespace tq
