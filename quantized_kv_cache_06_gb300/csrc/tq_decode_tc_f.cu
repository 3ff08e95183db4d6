// Tensor-core paged decode: the instantiated forms at D 64, K widths 3 and 5, every V width, GQA
// groups 4 and 8 (the kernel is in tq_decode_tc.cuh).
#include "tq_decode_tc.cuh"

namespace tq {

cudaError_t launch_tc_part_f(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  TQ_TC_VBITS(64, 3, 2)
  TQ_TC_VBITS(64, 5, 2)
  return cudaErrorNotSupported;
}

}  // namespace tq
