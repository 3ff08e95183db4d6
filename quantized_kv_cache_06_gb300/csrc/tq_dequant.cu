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
// A lane owns 32 consecutive coordinates of one row (R = D / 32 lanes per row, 32 / R rows
// per warp step, rows taken in [token][head] order).  Its 32 b-bit indices are exactly b
// whole index words, so every field sits at a fixed bit position; the centroid comes from
// a warp shuffle (lane k holds centroid k, b <= 5); the inverse WHT is 5 in-register
// butterfly stages plus log2(R) shuffle stages, then x s_d nu / sqrt(D) and 16-byte stores.
// The work is a streaming read of RB bytes and a write of D values per row (HBM bound).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {


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

template <typename T, int D, int BITS>
__global__ void __launch_bounds__(256) dequant_rows_kernel(DequantArgs a) {
  constexpr int E = 32;                 // coordinates per lane
  constexpr int R = D / E;              // lanes per row
  constexpr int RPW = 32 / R;           // rows per warp step
  constexpr int RB = D * BITS / 8 + 4;  // row bytes (a multiple of 4)
  constexpr int IB = D * BITS / 8;      // index bytes
  const int lane = threadIdx.x & 31;
  const int part = lane % R, rl = lane / R;  // this lane: coordinates [32 part, 32 part + 32) of row rl
  const int H = a.num_kv_heads;
  const int64_t capacity = a.num_blocks * (int64_t)a.block_size;
  const int64_t num_rows = a.num_tokens * H;
  // centroid k sits in every lane l with l mod 2^b == k: a shuffle reads only the low 5 bits
  // of its source lane, so a field needs no mask
  const float my_centroid = __ldg(a.centroids + (lane & ((1 << BITS) - 1)));
  const float rsd = 1.0f / sqrtf((float)D);
  float sgn[E];
#pragma unroll
  for (int i = 0; i < E; ++i) sgn[i] = __ldg(a.signs + part * E + i) * rsd;
  T* out = static_cast<T*>(a.out);
  const int64_t step = (int64_t)gridDim.x * (blockDim.x >> 5) * RPW;
  // Loads run ahead of the math: the slot two steps ahead, the row words one step ahead.
  auto slot_of = [&](int64_t row) -> int64_t { return row < num_rows ? __ldg(a.slots + row / H) : -1; };
  struct RowLoad {
    uint32_t w[BITS];
    uint32_t nub;
    bool live;
  };
  auto load_row = [&](int64_t row, int64_t slot) {
    RowLoad L;
    const bool bad = slot >= capacity;
    if (bad && part == 0 && a.status) atomicMax(a.status, (int32_t)kSlotOutOfRange);
    L.live = slot >= 0 && !bad;
    L.nub = 0u;
#pragma unroll
    for (int k = 0; k < BITS; ++k) L.w[k] = 0u;
    if (L.live) {
      const int64_t t = row / H;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(a.pages + (slot * H + (row - t * H)) * RB);
#pragma unroll
      for (int k = 0; k < BITS; ++k) L.w[k] = __ldg(src + part * BITS + k);
      L.nub = __ldg(src + IB / 4);
    }
    return L;
  };
  int64_t row = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW + rl;
  int64_t slot_next = slot_of(row + step);
  RowLoad cur = load_row(row, slot_of(row));
  for (; row - rl < num_rows; row += step) {
    const RowLoad nxt = load_row(row + step, slot_next);
    slot_next = slot_of(row + 2 * step);
    const bool in = row < num_rows;
    const bool live = cur.live;
    const uint32_t* w = cur.w;
    const uint32_t nub = cur.nub;
    float v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {  // field i at bits [i b, i b + b) of the lane's words
      const int bit = i * BITS, k = bit >> 5, sh = bit & 31;
      uint32_t f = w[k] >> sh;
      if (sh + BITS > 32) f |= w[k + 1] << (32 - sh);
      v[i] = __shfl_sync(kFullMask, my_centroid, (int)f);
    }
    // unnormalised WHT of the D-vector spread over the row's R lanes: stride 1 in pairs,
    // strides 2..16 on packed pairs, then the strides between lanes
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float x = v[i], y = v[i + 1];
      v[i] = x + y;
      v[i + 1] = x - y;
    }
    const float2 minus1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int hs = 2; hs < E; hs <<= 1)
#pragma unroll
      for (int i = 0; i < E; i += 2)
        if ((i & hs) == 0) {
          const float2 x = make_float2(v[i], v[i + 1]), y = make_float2(v[i + hs], v[i + hs + 1]);
          const float2 sm = __fadd2_rn(x, y), df = __ffma2_rn(y, minus1, x);
          v[i] = sm.x;
          v[i + 1] = sm.y;
          v[i + hs] = df.x;
          v[i + hs + 1] = df.y;
        }
#pragma unroll
    for (int m = 1; m < R; m <<= 1) {
      const float f = (part & m) ? -1.f : 1.f;  // upper lane: p - v, lower lane: v + p
      const float2 f2 = make_float2(f, f);
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        const float2 p = make_float2(__shfl_xor_sync(kFullMask, v[i], m), __shfl_xor_sync(kFullMask, v[i + 1], m));
        const float2 r = __ffma2_rn(make_float2(v[i], v[i + 1]), f2, p);
        v[i] = r.x;
        v[i + 1] = r.y;
      }
    }
    const float nu = live ? __uint_as_float(nub) : 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] *= sgn[i] * nu;
    if (in) {
      T* dst = out + row * D + part * E;
#pragma unroll
      for (int k = 0; k < E * (int)sizeof(T) / 16; ++k) {
        constexpr int PER = 16 / (int)sizeof(T);
        float vk[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) vk[i] = v[k * PER + i];
        store_chunk<T, PER>(dst + k * PER, vk);
      }
    }
    cur = nxt;
  }
}

template <typename T, int D>
cudaError_t launch_bits(const DequantArgs& a, cudaStream_t stream, int grid) {
  switch (a.bits) {
    case 2: dequant_rows_kernel<T, D, 2><<<grid, 256, 0, stream>>>(a); break;
    case 3: dequant_rows_kernel<T, D, 3><<<grid, 256, 0, stream>>>(a); break;
    case 4: dequant_rows_kernel<T, D, 4><<<grid, 256, 0, stream>>>(a); break;
    case 5: dequant_rows_kernel<T, D, 5><<<grid, 256, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

template <typename T>
cudaError_t launch_dim(const DequantArgs& a, cudaStream_t stream, int grid) {
  switch (a.head_dim) {
    case 32: return launch_bits<T, 32>(a, stream, grid);
    case 64: return launch_bits<T, 64>(a, stream, grid);
    case 128: return launch_bits<T, 128>(a, stream, grid);
    case 256: return launch_bits<T, 256>(a, stream, grid);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool dequant_supported(const DequantArgs& a) {
  const bool dim = a.head_dim == 16 || a.head_dim == 32 || a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256;
  return dim && a.bits >= 2 && a.bits <= 5;
}

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t stream, int num_sms) {
  if (a.num_tokens <= 0) return cudaSuccess;
  if (a.head_dim == 16) return launch_dequant_d16(a, stream);
  const int64_t rows_per_warp = 32 / (a.head_dim / 32);
  const int64_t warps_wanted = (a.num_tokens * a.num_kv_heads + rows_per_warp - 1) / rows_per_warp;
  const int64_t blocks = (warps_wanted + 7) / 8;
  const int grid = (int)(blocks < (int64_t)num_sms * 8 ? blocks : (int64_t)num_sms * 8);
  if (a.out_dtype == kF16) return launch_dim<__half>(a, stream, grid);
  if (a.out_dtype == kBF16) return launch_dim<__nv_bfloat16>(a, stream, grid);
  return launch_dim<float>(a, stream, grid);
}

}  // namespace tq
