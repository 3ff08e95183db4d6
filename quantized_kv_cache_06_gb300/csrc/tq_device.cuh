// Device helpers shared by the writer and decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

constexpr unsigned kFullMask = 0xffffffffu;

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Loads E consecutive elements starting at p (aligned to E * sizeof(T) when that is
// 4, 8 or 16 bytes) into fp32 registers, using one vector load where possible.
template <typename T, int E>
__device__ __forceinline__ void load_chunk(const T* __restrict__ p, float (&v)[E]) {
  constexpr int bytes = E * (int)sizeof(T);
  if constexpr (bytes == 16 || bytes == 32) {
#pragma unroll
    for (int k = 0; k < bytes / 16; ++k) {
      uint4 w = __ldg(reinterpret_cast<const uint4*>(p) + k);
      const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
      for (int i = 0; i < 16 / (int)sizeof(T); ++i) v[k * (16 / (int)sizeof(T)) + i] = to_f32<T>(e[i]);
    }
  } else if constexpr (bytes == 8) {
    uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = to_f32<T>(e[i]);
  } else if constexpr (bytes == 4) {
    uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p));
    const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = to_f32<T>(e[i]);
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = to_f32<T>(p[i]);
  }
}

__device__ __forceinline__ float load_as_f32(const void* base, int64_t i, int dtype) {
  if (dtype == 0) return __ldg(reinterpret_cast<const float*>(base) + i);
  if (dtype == 1) return __half2float(reinterpret_cast<const __half*>(base)[i]);
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
}

// Element i of query (row, q head) r: q_dtype 0/1/2 as load_as_f32, 3 = int8 code times
// the (row, q head) scale q_scale[r].
__device__ __forceinline__ float load_query_f32(const void* q, const float* q_scale, int64_t r, int64_t i,
                                                int dtype) {
  if (dtype == 3) return (float)reinterpret_cast<const int8_t*>(q)[i] * __ldg(q_scale + r);
  return load_as_f32(q, i, dtype);
}

__device__ __forceinline__ void store_from_f32(void* base, int64_t i, int dtype, float v) {
  if (dtype == 0) reinterpret_cast<float*>(base)[i] = v;
  else if (dtype == 1) reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
  else reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFullMask, v, m);
  return v;
}
// 2^k for k in [-126, 127], from its bits.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }
// x * 2^k, exact while the result is representable, for |k| <= 252 (two normal factors).
__device__ __forceinline__ float scale_pow2(float x, int k) {
  const int a = k / 2;
  return x * pow2i(a) * pow2i(k - a);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, m));
  return v;
}

// Unnormalised natural-order Walsh-Hadamard transform of a D = 32 * E vector held by
// one warp, lane l owning elements [l*E, l*E + E).  Strides below E are butterflies
// inside a lane, strides E..16E are butterflies between lanes l and l ^ (stride/E).
template <int E>
__device__ __forceinline__ void fwht_warp(float (&v)[E]) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float p = __shfl_xor_sync(kFullMask, v[i], m);
      v[i] = upper ? (p - v[i]) : (v[i] + p);
    }
  }
}

}  // namespace tq
