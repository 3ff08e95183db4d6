// Tensor-core paged decode: the instantiated forms at D 128, K widths 2 and 4, every V width, GQA
// groups 4 and 8 (the kernel is in tq_decode_tc.cuh).
#include "tq_decode_tc.cuh"

namespace tq {

cudaError_t launch_tc_part_a(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  TQ_TC_VBITS(128, 2, 2)
  TQ_TC_VBITS(128, 4, 2)
  return cudaErrorNotSupported;
}

}  // namespace tq
