// Tensor-core paged decode (sm_103a): plain decode instantiations and the host entry points.
// The kernels and their description are in tq_decode_tc.cuh.
#include "tq_decode_tc.cuh"

namespace tq {

bool tc_decode_supported(const DecodeArgs& a) {
  const int G = a.num_kv_heads > 0 ? a.num_q_heads / a.num_kv_heads : 0;
  const bool b24 = (a.k_bits == 2 || a.k_bits == 4) && (a.v_bits == 2 || a.v_bits == 4);
  const bool b33 = a.k_bits == 3 && a.v_bits == 3;
  const bool b55 = a.k_bits == 5 && a.v_bits == 5;
  const bool bits_ok = b24 || b33 || b55;
  // exactly the instantiations in launch_decode_tc
  const bool dim_ok =
      a.head_dim == 128 || a.head_dim == 256 || (a.head_dim == 64 && a.k_bits == 4 && a.v_bits == 4);
  return a.block_size == kBS && a.num_kv_heads >= 1 && a.num_kv_heads <= 8 && (G == 4 || G == 8) && bits_ok && dim_ok;
}

int tc_partials_per_sequence_split() { return 1; }

cudaError_t launch_decode_tc(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  // Batches with a block-table row map (tq_paged_prefill) never come here: every shape this
  // kernel covers is also covered by the multi-query kernel, which takes them.
  if (a.bt_rows) return cudaErrorInvalidValue;
  return launch_decode_tc_dispatch(a, p, stream);
}

}  // namespace tq
