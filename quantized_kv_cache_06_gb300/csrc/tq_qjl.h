// Internal declarations of the product-quantised ("QJL residual") key path (tq_qjl.cu) and
// the slot check it shares with the MSE writer (tq_write.cu).  Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "tq_internal.h"

namespace tq {

// Enqueues the slot check alone: status <- kSlotOutOfRange if a slot is past the pages.
cudaError_t launch_validate_slots(const WriteArgs& a, cudaStream_t stream, int num_sms);

// WriteArgs.bits and DecodeArgs.k_bits are the total key bits b (MSE indices at b - 1 bits
// plus one sign bit); the centroids passed for the keys are the (b - 1)-bit MSE codebook;
// smat is S, fp32 [D][D] row-major.
bool prod_supported(int head_dim, int bits);
// The tensor-core form of the product-row writer (tq_write_tc.cu): fp16 / bf16 rows at
// head_dim 64 / 128 and fp32 rows at 64; launched after the slot check, on `grid` CTAs.
bool write_prod_tc_supported(const WriteArgs& a);
cudaError_t launch_write_prod_tc(const WriteArgs& a, const float* smat, cudaStream_t stream, int grid);
// Enqueues status reset, slot check and the product-row writer.
cudaError_t launch_write_prod(const WriteArgs& a, const float* smat, cudaStream_t stream, int num_sms);
// Workspace of the product-key decode for split plan p (a SIMT plan of plan_decode).
size_t prod_decode_workspace(const DecodeArgs& a, const DecodePlan& p);
// Enqueues status reset, the query projection S R q, the split decode and the combine.
cudaError_t launch_decode_prod(const DecodeArgs& a, const float* smat, const DecodePlan& p, cudaStream_t stream);

}  // namespace tq
