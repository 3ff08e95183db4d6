// Dense readback of packed TurboQuant rows (sm_103a).
//
// TurboQuant docs: "vLLM Reference Audit" (file map: tq4_decompress, the TQ4 unpack
// kernel used for diagnostic readback of packed index bytes and norms) and
// "Architecture" (Diagnostic vs Serving Paths: dense reconstruction from packed bytes,
// for layout and distortion checks).  For every token t with slot s >= 0 and every kv
// head h the row pages[s / bs][s % bs][h] is reconstructed as nu * R^T c[idx]:
// unpack the b-bit indices (LSB-first stream), look the centroids up, apply the inverse
// rotation R^T = diag(s) H_D / sqrt(D), scale by the stored norm.  Negative slots give
// zero rows; a slot past the pages gives a zero row and TQ_ERR_SLOT_OUT_OF_RANGE.
//
// One warp per token (its H rows are contiguous in both the pages and the output); lane
// l owns coordinates [l E, l E + E), E = D / 32.  The lane's E indices sit in one 64-bit
// window of the row's index words; the centroid comes from a warp shuffle (lane k holds
// centroid k, b <= 5); the inverse WHT is the in-register + shuffle butterfly.  The work
// is a streaming read of RB bytes and a write of D output values per row (HBM bound).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kHeadChunk = 8;  // rows of one token whose loads are issued together

template <typename T, int E>
__device__ __forceinline__ void store_chunk(T* p, const float (&v)[E]) {
  constexpr int bytes = E * (int)sizeof(T);
  if constexpr (bytes == 8 || bytes == 16) {
    union {
      T e[E];
      uint2 u2;
      uint4 u4;
    } w;
#pragma unroll
    for (int i = 0; i < E; ++i) w.e[i] = from_f32<T>(v[i]);
    if constexpr (bytes == 8) *reinterpret_cast<uint2*>(p) = w.u2;
    else *reinterpret_cast<uint4*>(p) = w.u4;
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) p[i] = from_f32<T>(v[i]);
  }
}

template <typename T, int E, int BITS>
__global__ void __launch_bounds__(256) dequant_rows_kernel(DequantArgs a) {
  constexpr int D = 32 * E;
  constexpr int RB = D * BITS / 8 + 4;  // row bytes (D >= 32: a multiple of 4)
  constexpr int IB = D * BITS / 8;      // index bytes
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  const int lane = threadIdx.x & 31;
  const int H = a.num_kv_heads;
  const int64_t capacity = a.num_blocks * (int64_t)a.block_size;
  const float my_centroid = lane < (1 << BITS) ? __ldg(a.centroids + lane) : 0.f;
  float sgn[E];
#pragma unroll
  for (int i = 0; i < E; ++i) sgn[i] = __ldg(a.signs + lane * E + i) * (1.0f / sqrtf((float)D));
  // this lane's bits [o, o + E * BITS) of the index stream: words w0, w0 + 1 (both inside
  // the row: the window ends before the index bytes do, and the norm word follows them)
  const int o = lane * E * BITS;
  const int w0 = o >> 5, shift = o & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int64_t slot = t < a.num_tokens ? __ldg(a.slots + t) : -1;
  T* out = static_cast<T*>(a.out);
  for (; t < a.num_tokens; t += warps) {
    const int64_t next = t + warps < a.num_tokens ? __ldg(a.slots + t + warps) : -1;  // one token ahead
    const bool bad = slot >= capacity;
    if (bad && lane == 0 && a.status) atomicMax(a.status, (int32_t)kSlotOutOfRange);
    const bool live = slot >= 0 && !bad;
    const uint32_t* rows = reinterpret_cast<const uint32_t*>(a.pages + (live ? slot : 0) * (int64_t)H * RB);
    for (int h0 = 0; h0 < H; h0 += kHeadChunk) {
      // loads of up to kHeadChunk rows in flight before any of them is used
      uint32_t wlo[kHeadChunk], whi[kHeadChunk], wnu[kHeadChunk];
#pragma unroll
      for (int k = 0; k < kHeadChunk; ++k) {
        wlo[k] = whi[k] = wnu[k] = 0u;
        if (live && h0 + k < H) {
          const uint32_t* row = rows + (h0 + k) * (RB / 4);
          wlo[k] = __ldg(row + w0);
          whi[k] = __ldg(row + w0 + 1);
          wnu[k] = __ldg(row + IB / 4);
        }
      }
#pragma unroll
      for (int k = 0; k < kHeadChunk; ++k) {
        if (h0 + k >= H) break;
        float v[E];
        if (live) {
          const uint64_t win = ((uint64_t)whi[k] << 32 | wlo[k]) >> shift;
          const float nu = __uint_as_float(wnu[k]);
#pragma unroll
          for (int i = 0; i < E; ++i) {
            const int idx = (int)((uint32_t)(win >> (i * BITS)) & kMask);
            v[i] = __shfl_sync(kFullMask, my_centroid, idx);
          }
          fwht_warp<E>(v);
#pragma unroll
          for (int i = 0; i < E; ++i) v[i] *= sgn[i] * nu;
        } else {
#pragma unroll
          for (int i = 0; i < E; ++i) v[i] = 0.f;
        }
        store_chunk<T, E>(out + (t * H + h0 + k) * D + lane * E, v);
      }
    }
    slot = next;
  }
}

template <typename T, int E>
cudaError_t launch_bits(const DequantArgs& a, cudaStream_t stream, int grid) {
  switch (a.bits) {
    case 2: dequant_rows_kernel<T, E, 2><<<grid, 256, 0, stream>>>(a); break;
    case 3: dequant_rows_kernel<T, E, 3><<<grid, 256, 0, stream>>>(a); break;
    case 4: dequant_rows_kernel<T, E, 4><<<grid, 256, 0, stream>>>(a); break;
    case 5: dequant_rows_kernel<T, E, 5><<<grid, 256, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dim(const DequantArgs& a, cudaStream_t stream, int grid) {
  switch (a.head_dim) {
    case 32: return launch_bits<T, 1>(a, stream, grid);
    case 64: return launch_bits<T, 2>(a, stream, grid);
    case 128: return launch_bits<T, 4>(a, stream, grid);
    case 256: return launch_bits<T, 8>(a, stream, grid);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool dequant_supported(const DequantArgs& a) {
  const bool dim = a.head_dim == 32 || a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256;
  return dim && a.bits >= 2 && a.bits <= 5;
}

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t stream, int num_sms) {
  if (a.num_tokens <= 0) return cudaSuccess;
  const int64_t warps_wanted = a.num_tokens;
  const int64_t blocks = (warps_wanted + 7) / 8;
  const int grid = (int)(blocks < (int64_t)num_sms * 8 ? blocks : (int64_t)num_sms * 8);
  if (a.out_dtype == kF16) return launch_dim<__half>(a, stream, grid);
  if (a.out_dtype == kBF16) return launch_dim<__nv_bfloat16>(a, stream, grid);
  return launch_dim<float>(a, stream, grid);
}

}  // namespace tq
