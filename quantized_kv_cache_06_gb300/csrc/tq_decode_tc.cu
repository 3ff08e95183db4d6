// Tensor-core paged decode (sm_103a): the host entry points.
// The kernels and their description are in tq_decode_tc.cuh.
#include "tq_decode_tc.cuh"

namespace tq {

bool tc_decode_supported(const DecodeArgs& a) {
  const int G = a.num_kv_heads > 0 ? a.num_q_heads / a.num_kv_heads : 0;
  const bool bits_ok = a.k_bits >= 2 && a.k_bits <= 5 && a.v_bits >= 2 && a.v_bits <= 5;
  // exactly the instantiations of launch_tc_part_a..f
  const bool dim_ok = a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256;
  return a.block_size == kBS && a.num_kv_heads >= 1 && a.num_kv_heads <= 8 && (G == 4 || G == 8) && bits_ok && dim_ok;
}

int tc_partials_per_sequence_split() { return 1; }

cudaError_t launch_decode_tc(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  // Batches with a block-table row map (tq_paged_prefill) never come here: plan_decode sends
  // the shapes the multi-query kernel does not take to the SIMT decode.
  if (a.bt_rows) return cudaErrorInvalidValue;
  cudaError_t (*const parts[])(const DecodeArgs&, const DecodePlan&, cudaStream_t) = {
      launch_tc_part_a, launch_tc_part_b, launch_tc_part_c, launch_tc_part_d, launch_tc_part_e, launch_tc_part_f};
  for (auto part : parts) {
    const cudaError_t err = part(a, p, stream);
    if (err != cudaErrorNotSupported) return err;
  }
  return cudaErrorInvalidValue;
}


}  // namespace tq
