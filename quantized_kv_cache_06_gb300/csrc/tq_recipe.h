// Internal declarations of the recipe cache modes turboquant25 / turboquant35 (tq_recipe.cu):
// grouped product-quantised rows for K and V.  Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "tq_internal.h"
#include "tq_qjl.h"

namespace tq {

// The group codec of a recipe call.  head_dim D = 2 d; the high group is coded at bits_hi
// (MSE part bits_hi - 1 bits) and the low group at bits_lo.
struct RecipeArgs {
  const int32_t* order;  // device [H][D]: each kv head's high channels (sorted), then its low ones
  const float* mse_hi;   // device [2^(bits_hi - 1)], the MSE codebook of dimension d
  const float* mse_lo;   // device [2^(bits_lo - 1)]
  const float* smat;     // device [d][d] row-major, S_d
  int bits_hi;
  int bits_lo;
};

bool recipe_supported(int head_dim);
// Bytes of one recipe row: the high group's product row, then the low group's.
int recipe_row_bytes(int head_dim, int bits_hi, int bits_lo);
// WriteArgs.signs / DecodeArgs.signs are the d signs of R_d; head_dim is D.  Enqueues status
// reset, slot check and the writer.
cudaError_t launch_write_recipe(const WriteArgs& a, const RecipeArgs& rc, cudaStream_t stream, int num_sms);
// Workspace of the recipe decode for split plan p (a SIMT plan of plan_decode).
size_t recipe_decode_workspace(const DecodeArgs& a, const DecodePlan& p);
// Enqueues status reset, the query projections, the split decode and the combine.
cudaError_t launch_decode_recipe(const DecodeArgs& a, const RecipeArgs& rc, const DecodePlan& p, cudaStream_t stream);

}  // namespace tq
