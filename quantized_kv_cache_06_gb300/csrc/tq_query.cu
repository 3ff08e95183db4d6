// Int8 query quantiser for the INT8-query prefill ("vLLM Usage", Runtime Dispatch: cache
// plus INT8 prefill gate, the int8 query path; "vLLM Reference Audit", File Map: INT8-Q
// prefill, int8 query scale).
//
// One warp per (query row, q head): amax = max |q_j|, s = amax / 127 and code_j =
// round-half-even(q_j / s) clamped to [-127, 127], both divisions correctly rounded fp32
// (a zero row gives s = 0 and codes 0).  Lane l owns elements [l E, l E + E) of D = 32 E.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

template <int E>
__global__ void __launch_bounds__(256)
quantize_queries_kernel(const void* __restrict__ q, int q_dtype, int64_t rows, int8_t* __restrict__ codes,
                        float* __restrict__ scales) {
  constexpr int D = 32 * E;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    float v[E];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      v[i] = load_as_f32(q, r * D + lane * E + i, q_dtype);
      amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));
    const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      int c = 0;
      if (s > 0.f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(v[i], s))));
      codes[r * D + lane * E + i] = (int8_t)c;
    }
    if (lane == 0) scales[r] = s;
  }
}

}  // namespace

cudaError_t launch_quantize_queries(const void* q, int q_dtype, int64_t rows, int head_dim, int8_t* codes,
                                    float* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (head_dim == 16) return launch_quantize_d16(q, q_dtype, rows, codes, scales, stream);
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, (int64_t)sms * 8));
  switch (head_dim) {
    case 32: quantize_queries_kernel<1><<<grid, 256, 0, stream>>>(q, q_dtype, rows, codes, scales); break;
    case 64: quantize_queries_kernel<2><<<grid, 256, 0, stream>>>(q, q_dtype, rows, codes, scales); break;
    case 128: quantize_queries_kernel<4><<<grid, 256, 0, stream>>>(q, q_dtype, rows, codes, scales); break;
    case 256: quantize_queries_kernel<8><<<grid, 256, 0, stream>>>(q, q_dtype, rows, codes, scales); break;
    default: return cudaErrorInvalidValue;
  }
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

}  // namespace tq
