// Tensor-core paged decode: the instantiated forms at D 256, K widths 3 and 5, every V width, GQA
// groups 4 and 8 (the kernel is in tq_decode_tc.cuh).
#include "tq_decode_tc.cuh"

namespace tq {

cudaError_t launch_tc_part_d(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  TQ_TC_VBITS(256, 3, 1)
  TQ_TC_VBITS(256, 5, 1)
  return cudaErrorNotSupported;
}

}  // namespace tq
