// Tensor-core paged decode: the instantiated forms at D 64, K widths 2 and 4, every V width, GQA
// groups 4 and 8 (the kernel is in tq_decode_tc.cuh).
#include "tq_decode_tc.cuh"

namespace tq {

cudaError_t launch_tc_part_e(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  TQ_TC_VBITS(64, 2, 2)
  TQ_TC_VBITS(64, 4, 2)
  return cudaErrorNotSupported;
}

}  // namespace tq
