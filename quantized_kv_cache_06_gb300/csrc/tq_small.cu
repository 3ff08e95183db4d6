// head_dim 16: writer, paged decode / prefill, readback and int8 query quantiser (sm_103a,
// SIMT).
//
// TurboQuant docs: "vLLM Usage" (TQ Byte Layout: ceil(16 b / 8) + 4 bytes per row; Slot
// Mapping; TQ Packed Page Contract) and "Architecture" (Diagnostic vs Serving Paths).  The
// arithmetic is the one of the other head dims -- nu = ||x||, u = H_16 (s * x) / (4 nu),
// index = #{k : boundary_k < u}, LSB-first packing, fp32 norm appended; scores
// nu_k <R q, c[idx]> and values accumulated in rotated space, R^T applied once per output.
// At D = 16 a row is 8, 10, 12 or 14 bytes, not always a whole number of 32-bit words, so
// every kernel here reads and writes rows byte by byte; a row is short enough for one
// thread to hold it, so the 16-point Walsh-Hadamard transform runs in one thread's
// registers.  Decode: one CTA per (row of the batch, q head), its threads taking tokens in
// turn with a private online softmax, merged through shared memory at the end.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kD16 = 16;
constexpr int kSmallDecodeThreads = 128;
constexpr float kSmallLog2e = 1.4426950408889634f;

// Unnormalised natural-order Walsh-Hadamard transform of 16 values in registers.
__device__ __forceinline__ void fwht16(float (&v)[kD16]) {
#pragma unroll
  for (int h = 1; h < kD16; h <<= 1)
#pragma unroll
    for (int i = 0; i < kD16; ++i)
      if ((i & h) == 0) {
        const float x = v[i], y = v[i + h];
        v[i] = x + y;
        v[i + h] = x - y;
      }
}

// The 16 b-bit indices of a row from its first 2 b bytes (LSB-first stream).
__device__ __forceinline__ void unpack16(const uint8_t* __restrict__ row, int bits, int (&idx)[kD16]) {
  uint64_t lo = 0, hi = 0;  // stream bits [0, 64) and [64, 80)
  const int nbytes = 2 * bits;
  for (int k = 0; k < nbytes; ++k) {
    const uint64_t byte = __ldg(row + k);
    if (k < 8) lo |= byte << (8 * k);
    else hi |= byte << (8 * (k - 8));
  }
  const uint32_t mask = (1u << bits) - 1u;
#pragma unroll
  for (int j = 0; j < kD16; ++j) {
    const int bit = j * bits;
    uint32_t f;
    if (bit + bits <= 64) f = (uint32_t)(lo >> bit);
    else if (bit >= 64) f = (uint32_t)(hi >> (bit - 64));
    else f = (uint32_t)(lo >> bit) | (uint32_t)(hi << (64 - bit));
    idx[j] = (int)(f & mask);
  }
}

__device__ __forceinline__ float load_norm(const uint8_t* __restrict__ p) {
  const uint32_t w = (uint32_t)__ldg(p) | ((uint32_t)__ldg(p + 1) << 8) | ((uint32_t)__ldg(p + 2) << 16) |
                     ((uint32_t)__ldg(p + 3) << 24);
  return __uint_as_float(w);
}

template <typename T>
__global__ void __launch_bounds__(256)
write_d16_kernel(const T* __restrict__ raw, int64_t num_rows, int num_kv_heads, int bits,
                 const int64_t* __restrict__ slots, uint8_t* __restrict__ pages, const float* __restrict__ signs,
                 const float* __restrict__ centroids, const int32_t* __restrict__ status) {
  __shared__ float bnd[31];
  const int nc = 1 << bits;
  // decision points: correctly rounded midpoints of neighbouring fp32 centroids
  if (threadIdx.x < nc - 1) bnd[threadIdx.x] = 0.5f * (centroids[threadIdx.x] + centroids[threadIdx.x + 1]);
  __syncthreads();
  if (*status != kOk) return;  // a slot failed validation: write nothing
  float sg[kD16];
#pragma unroll
  for (int i = 0; i < kD16; ++i) sg[i] = __ldg(signs + i);
  const int rb = 2 * bits + 4;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < num_rows; r += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = r / num_kv_heads;
    const int h = (int)(r - t * num_kv_heads);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // "Slot Mapping": negative slots are ignored
    float v[kD16];
#pragma unroll
    for (int i = 0; i < kD16; ++i) v[i] = to_f32<T>(raw[r * kD16 + i]);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kD16; ++i) ss = fmaf(v[i], v[i], ss);
    const float nu = sqrtf(ss);
#pragma unroll
    for (int i = 0; i < kD16; ++i) v[i] *= sg[i];
    fwht16(v);
    const float inv = nu > 0.f ? 0.25f / nu : 0.f;  // y = H(s*x)/(sqrt(16) nu)
    uint32_t w[3] = {0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < kD16; ++j) {
      const float u = v[j] * inv;
      int idx = 0;  // #{k : boundary_k < u}
      for (int s = nc >> 1; s > 0; s >>= 1)
        if (u > bnd[idx + s - 1]) idx += s;
      const int bit = j * bits, wi = bit >> 5, o = bit & 31;
      w[wi] |= (uint32_t)idx << o;
      if (o + bits > 32) w[wi + 1] |= (uint32_t)idx >> (32 - o);
    }
    uint8_t* dst = pages + (slot * num_kv_heads + h) * (int64_t)rb;
    for (int k = 0; k < 2 * bits; ++k) dst[k] = (uint8_t)(w[k >> 2] >> (8 * (k & 3)));
    const uint32_t nb = __float_as_uint(nu);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[2 * bits + k] = (uint8_t)(nb >> (8 * k));
  }
}

// Merges (m, l, acc) of thread `other` into the running triple (base-2 online softmax).
__device__ __forceinline__ void merge_state(float& m, float& l, float (&acc)[kD16], float m2, float l2,
                                            const float* acc2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  const float w1 = m == -INFINITY ? 0.f : exp2f(m - mn), w2 = m2 == -INFINITY ? 0.f : exp2f(m2 - mn);
  l = l * w1 + l2 * w2;
#pragma unroll
  for (int i = 0; i < kD16; ++i) acc[i] = acc[i] * w1 + acc2[i] * w2;
  m = mn;
}

__global__ void __launch_bounds__(kSmallDecodeThreads) decode_d16_kernel(DecodeArgs a) {
  const int hq = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  const int G = a.num_q_heads / a.num_kv_heads, h = hq / G, H = a.num_kv_heads, bs = a.block_size;
  __shared__ float ck[32], cv[32];
  __shared__ float red[kSmallDecodeThreads][kD16 + 2];
  if (tid < (1 << a.k_bits)) ck[tid] = a.k_centroids[tid];
  if (tid < (1 << a.v_bits)) cv[tid] = a.v_centroids[tid];

  // q~ = R q times the softmax scale and log2(e) (every thread keeps it)
  const float scale = a.scale > 0.f ? a.scale : 0.25f;
  const float qmul = scale * kSmallLog2e * 0.25f;
  const int64_t qrow = (int64_t)b * a.num_q_heads + hq;
  float qr[kD16];
#pragma unroll
  for (int i = 0; i < kD16; ++i) qr[i] = load_query_f32(a.q, a.q_scale, qrow, qrow * kD16 + i, a.q_dtype) * __ldg(a.signs + i);
  fwht16(qr);
#pragma unroll
  for (int i = 0; i < kD16; ++i) qr[i] *= qmul;

  int len = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks_per_seq * bs;
  if (len < 0 || len > cap) {
    if (tid == 0 && hq == 0 && a.status) atomicMax(a.status, (int32_t)kInvalidArg);
    len = len < 0 ? 0 : cap;
  }
  const int bt_row = block_table_row(a, b);
  if (bt_row < 0) {  // a row map entry outside the table: nothing is read for this row
    if (tid == 0 && a.status) atomicMax(a.status, (int32_t)kInvalidArg);
    len = 0;
  }
  const int rbk = 2 * a.k_bits + 4, rbv = 2 * a.v_bits + 4;
  __syncthreads();

  float m = -INFINITY, l = 0.f, acc[kD16];
#pragma unroll
  for (int i = 0; i < kD16; ++i) acc[i] = 0.f;
  bool bad_block = false;
  for (int t = tid; t < len; t += kSmallDecodeThreads) {
    const int bid = __ldg(a.block_table + (int64_t)bt_row * a.max_blocks_per_seq + t / bs);
    if (bid < 0 || (int64_t)bid >= a.num_blocks) {
      bad_block = true;
      continue;
    }
    const int64_t row = ((int64_t)bid * bs + t % bs) * H + h;
    const uint8_t* kr = a.k_pages + row * rbk;
    const uint8_t* vr = a.v_pages + row * rbv;
    int ki[kD16], vi[kD16];
    unpack16(kr, a.k_bits, ki);
    unpack16(vr, a.v_bits, vi);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kD16; ++i) s = fmaf(qr[i], ck[ki[i]], s);
    s *= load_norm(kr + 2 * a.k_bits);
    const float vnorm = load_norm(vr + 2 * a.v_bits);
    const float mn = fmaxf(m, s);
    const float corr = m == -INFINITY ? 0.f : exp2f(m - mn);
    const float p = exp2f(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int i = 0; i < kD16; ++i) acc[i] = fmaf(p * vnorm, cv[vi[i]], acc[i] * corr);
    m = mn;
  }
  if (bad_block && a.status) atomicMax(a.status, (int32_t)kBlockOutOfRange);

  // merge the threads' states: shared memory, halving the active threads
  red[tid][0] = m;
  red[tid][1] = l;
#pragma unroll
  for (int i = 0; i < kD16; ++i) red[tid][2 + i] = acc[i];
  __syncthreads();
  for (int half = kSmallDecodeThreads / 2; half >= 1; half >>= 1) {
    if (tid < half) {
      merge_state(m, l, acc, red[tid + half][0], red[tid + half][1], &red[tid + half][2]);
      red[tid][0] = m;
      red[tid][1] = l;
#pragma unroll
      for (int i = 0; i < kD16; ++i) red[tid][2 + i] = acc[i];
    }
    __syncthreads();
  }
  if (tid == 0) {
    const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
    for (int i = 0; i < kD16; ++i) acc[i] *= inv;
    fwht16(acc);  // R^T o~ = diag(s) H o~ / 4
#pragma unroll
    for (int i = 0; i < kD16; ++i) store_from_f32(a.out, qrow * kD16 + i, a.out_dtype, acc[i] * __ldg(a.signs + i) * 0.25f);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) dequant_d16_kernel(DequantArgs a) {
  const int H = a.num_kv_heads;
  const int64_t capacity = a.num_blocks * (int64_t)a.block_size;
  const int64_t num_rows = a.num_tokens * H;
  const int rb = 2 * a.bits + 4;
  __shared__ float cen[32];
  if (threadIdx.x < (1 << a.bits)) cen[threadIdx.x] = a.centroids[threadIdx.x];
  __syncthreads();
  bool bad = false;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < num_rows; r += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = r / H;
    const int h = (int)(r - t * H);
    const int64_t slot = __ldg(a.slots + t);
    float v[kD16];
    if (slot >= 0 && slot < capacity) {
      const uint8_t* row = a.pages + (slot * H + h) * (int64_t)rb;
      int idx[kD16];
      unpack16(row, a.bits, idx);
      const float nu = load_norm(row + 2 * a.bits);
#pragma unroll
      for (int i = 0; i < kD16; ++i) v[i] = cen[idx[i]];
      fwht16(v);
#pragma unroll
      for (int i = 0; i < kD16; ++i) v[i] *= __ldg(a.signs + i) * 0.25f * nu;
    } else {
      bad |= slot >= capacity;
#pragma unroll
      for (int i = 0; i < kD16; ++i) v[i] = 0.f;
    }
    T* out = static_cast<T*>(a.out) + r * kD16;
#pragma unroll
    for (int i = 0; i < kD16; ++i) out[i] = from_f32<T>(v[i]);
  }
  if (bad && a.status) atomicMax(a.status, (int32_t)kSlotOutOfRange);
}

__global__ void __launch_bounds__(256)
quantize_d16_kernel(const void* __restrict__ q, int q_dtype, int64_t rows, int8_t* __restrict__ codes,
                    float* __restrict__ scales) {
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += (int64_t)gridDim.x * blockDim.x) {
    float v[kD16], amax = 0.f;
#pragma unroll
    for (int i = 0; i < kD16; ++i) {
      v[i] = load_as_f32(q, r * kD16 + i, q_dtype);
      amax = fmaxf(amax, fabsf(v[i]));
    }
    const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int i = 0; i < kD16; ++i)
      codes[r * kD16 + i] = (int8_t)(s > 0.f ? max(-127, min(127, __float2int_rn(__fdiv_rn(v[i], s)))) : 0);
    scales[r] = s;
  }
}

int small_grid(int64_t items, int threads) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return (int)std::max<int64_t>(1, std::min<int64_t>((items + threads - 1) / threads, (int64_t)sms * 8));
}

}  // namespace

cudaError_t launch_write_d16(const WriteArgs& a, cudaStream_t stream) {
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  const int grid = small_grid(rows, 256);
  switch (a.dtype) {
    case kF32: write_d16_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(a.raw), rows, a.num_kv_heads, a.bits, a.slots, a.pages, a.signs, a.centroids, a.status); break;
    case kF16: write_d16_kernel<__half><<<grid, 256, 0, stream>>>(static_cast<const __half*>(a.raw), rows, a.num_kv_heads, a.bits, a.slots, a.pages, a.signs, a.centroids, a.status); break;
    case kBF16: write_d16_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(a.raw), rows, a.num_kv_heads, a.bits, a.slots, a.pages, a.signs, a.centroids, a.status); break;
    default: return cudaErrorInvalidValue;
  }
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

cudaError_t launch_decode_d16(const DecodeArgs& a, cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  decode_d16_kernel<<<dim3(a.num_q_heads, a.batch), kSmallDecodeThreads, 0, stream>>>(a);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

cudaError_t launch_dequant_d16(const DequantArgs& a, cudaStream_t stream) {
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  if (rows <= 0) return cudaSuccess;
  const int grid = small_grid(rows, 256);
  switch (a.out_dtype) {
    case kF32: dequant_d16_kernel<float><<<grid, 256, 0, stream>>>(a); break;
    case kF16: dequant_d16_kernel<__half><<<grid, 256, 0, stream>>>(a); break;
    case kBF16: dequant_d16_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

cudaError_t launch_quantize_d16(const void* q, int q_dtype, int64_t rows, int8_t* codes, float* scales,
                                cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  quantize_d16_kernel<<<small_grid(rows, 256), 256, 0, stream>>>(q, q_dtype, rows, codes, scales);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

}  // namespace tq
