// Tensor-core paged decode with a block-table row map (mixed prefill/decode: batch row i is
// one query token of sequence bt_rows[i]).  The kernels are in tq_decode_tc.cuh.
#include "tq_decode_tc.cuh"

namespace tq {

cudaError_t launch_decode_tc_rowmap(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  return launch_decode_tc_dispatch<true>(a, p, stream);
}

}  // namespace tq
