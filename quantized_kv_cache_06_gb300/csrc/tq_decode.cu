// Paged decode attention over packed TurboQuant pages.
//
// TurboQuant docs: "vLLM Usage" (TQ Packed Page Contract: decode_tq4_paged) and
// "Architecture" (Diagnostic vs Serving Paths: direct-QK keys, packed-V values; the
// paged path reads packed pages through the block table).
//
// Scores are taken in rotated space, s = scale * nu_k * <R q, c_k[idx]>, straight
// from the packed indices; values are accumulated in rotated space,
// acc = sum_t p_t nu_v,t c_v[idx_v,t], with an online softmax (base-2 exponent,
// log2(e) folded into the query); one inverse rotation R^T per output row is
// applied when the split-K partials are combined.
//
// Kernels:
//   decode_split_kernel  (SIMT) one CTA per (split, kv head, sequence); each warp
//                        walks tokens of the split; lane l owns coordinates
//                        [l*E, l*E+E) of the D = 32*E row.  Writes (m, l, acc[D])
//                        partials per (sequence, q head, split).
//   combine_kernel       one warp per (sequence, q head): merges the splits,
//                        divides by the softmax sum, applies R^T (in-register FWHT
//                        and sign flip) and casts to the output dtype.
// Kernel choice (plan_decode): the tensor-core decode (tq_decode_tc.cu) where it has an
// instantiation, else the multi-query kernel with one sequence per window
// (tq_prefill_mq.cu: D 64/128, 2/4-bit or equal 3/5-bit K/V), else the SIMT kernels.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kDecodeWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

struct SplitView {
  float* acc;  // [batch][num_q_heads][num_splits][D]
  float* ml;   // [batch][num_q_heads][num_splits][2]  (running max in log2 units, sum)
};

SplitView split_view(void* ws, int batch, int num_q_heads, int num_splits, int head_dim) {
  SplitView v;
  v.acc = static_cast<float*>(ws);
  v.ml = v.acc + (size_t)batch * num_q_heads * num_splits * head_dim;
  return v;
}

// b-bit index i (0-based within this lane's run) from a 64-bit little-endian window.
__device__ __forceinline__ int field(uint64_t win, int bitpos, int bits) {
  return (int)((win >> bitpos) & ((1u << bits) - 1u));
}

template <int E, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_split_kernel(DecodeArgs a, int num_splits, int blocks_per_split, SplitView part) {
  constexpr int D = 32 * E;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.num_kv_heads, bs = a.block_size;

  __shared__ float ck[32], cv[32];
  __shared__ float red_ml[kDecodeWarps][G][2];
  __shared__ float red_acc[kDecodeWarps][G][D];

  if (threadIdx.x < (1 << a.k_bits)) ck[threadIdx.x] = a.k_centroids[threadIdx.x];
  if (threadIdx.x < (1 << a.v_bits)) cv[threadIdx.x] = a.v_centroids[threadIdx.x];

  // q~ = R q = H(s*q)/sqrt(D), times the softmax scale and log2(e); every warp keeps
  // the G rotated heads of this kv head in registers.
  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kLog2e / sqrtf((float)D);
  float qr[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int64_t qrow = (int64_t)b * a.num_q_heads + (int64_t)h * G + g;  // (row, q head)
    const int64_t base = qrow * D + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i)
      qr[g][i] = load_query_f32(a.q, a.q_scale, qrow, base + i, a.q_dtype) * __ldg(a.signs + lane * E + i);
    fwht_warp<E>(qr[g]);
#pragma unroll
    for (int i = 0; i < E; ++i) qr[g][i] *= qmul;
  }

  int len = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks_per_seq * bs;
  if (len < 0 || len > cap) {
    if (threadIdx.x == 0 && split == 0 && h == 0 && a.status) atomicMax(a.status, (int32_t)kInvalidArg);
    len = len < 0 ? 0 : cap;
  }
  const int t_lo = split * blocks_per_split * bs;
  int t_hi = min(len, (split + 1) * blocks_per_split * bs);

  const int kib = D * a.k_bits / 8, vib = D * a.v_bits / 8;  // index bytes
  const int64_t krb = kib + 4, vrb = vib + 4;                 // row bytes
  const int kbit0 = lane * E * a.k_bits, vbit0 = lane * E * a.v_bits;

  float m[G], l[G], acc[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) acc[g][i] = 0.f;
  }
  __syncthreads();

  bool bad_block = false;
  const int bt_row = block_table_row(a, b);
  if (bt_row < 0) {  // a row map entry outside the table: nothing is read for this row
    if (threadIdx.x == 0 && a.status) atomicMax(a.status, (int32_t)kInvalidArg);
    t_hi = t_lo;
  }
  for (int t = t_lo + warp; t < t_hi; t += kDecodeWarps) {
    const int bid = __ldg(a.block_table + (int64_t)bt_row * a.max_blocks_per_seq + t / bs);
    if (bid < 0 || (int64_t)bid >= a.num_blocks) {
      bad_block = true;
      continue;
    }
    const int64_t row = ((int64_t)bid * bs + t % bs) * H + h;
    const uint32_t* kr = reinterpret_cast<const uint32_t*>(a.k_pages + row * krb);
    const uint32_t* vr = reinterpret_cast<const uint32_t*>(a.v_pages + row * vrb);

    const uint64_t kwin = (uint64_t)__ldg(kr + (kbit0 >> 5)) | ((uint64_t)__ldg(kr + (kbit0 >> 5) + 1) << 32);
    const uint64_t vwin = (uint64_t)__ldg(vr + (vbit0 >> 5)) | ((uint64_t)__ldg(vr + (vbit0 >> 5) + 1) << 32);
    const float knorm = __uint_as_float(__ldg(kr + kib / 4));
    const float vnorm = __uint_as_float(__ldg(vr + vib / 4));

    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float c = ck[field(kwin, (kbit0 & 31) + i * a.k_bits, a.k_bits)];
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = fmaf(qr[g][i], c, s[g]);
    }
    float vv[E];
#pragma unroll
    for (int i = 0; i < E; ++i) vv[i] = vnorm * cv[field(vwin, (vbit0 & 31) + i * a.v_bits, a.v_bits)];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sc = warp_sum(s[g]) * knorm;
      const float mn = fmaxf(m[g], sc);
      const float corr = exp2f(m[g] - mn);
      const float p = exp2f(sc - mn);
      l[g] = l[g] * corr + p;
#pragma unroll
      for (int i = 0; i < E; ++i) acc[g][i] = fmaf(p, vv[i], acc[g][i] * corr);
      m[g] = mn;
    }
  }
  if (__any_sync(kFullMask, bad_block) && lane == 0 && a.status) atomicMax(a.status, (int32_t)kBlockOutOfRange);

  // Merge the warps of this CTA, then write the split partial.
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_ml[warp][g][0] = m[g];
      red_ml[warp][g][1] = l[g];
    }
#pragma unroll
    for (int i = 0; i < E; ++i) red_acc[warp][g][lane * E + i] = acc[g][i];
  }
  __syncthreads();
  for (int g = warp; g < G; g += kDecodeWarps) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) mx = fmaxf(mx, red_ml[w][g][0]);
    float wt[kDecodeWarps], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      wt[w] = red_ml[w][g][0] == -INFINITY ? 0.f : exp2f(red_ml[w][g][0] - mx);
      lsum = fmaf(wt[w], red_ml[w][g][1], lsum);
    }
    const int64_t slot = ((int64_t)b * a.num_q_heads + (int64_t)h * G + g) * num_splits + split;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) s = fmaf(wt[w], red_acc[w][g][lane * E + i], s);
      part.acc[slot * D + lane * E + i] = s;
    }
    if (lane == 0) {
      part.ml[slot * 2 + 0] = mx;
      part.ml[slot * 2 + 1] = lsum;
    }
  }
}

template <int E>
__global__ void __launch_bounds__(256)
combine_kernel(int rows, int num_splits, SplitView part, const float* __restrict__ signs, void* out, int out_dtype) {
  constexpr int D = 32 * E;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* ml = part.ml + (int64_t)row * num_splits * 2;
  const float* acc = part.acc + (int64_t)row * num_splits * D;
  float mx = -INFINITY;
  for (int s = 0; s < num_splits; ++s) mx = fmaxf(mx, ml[2 * s]);
  float v[E];
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = 0.f;
  float lsum = 0.f;
  for (int s = 0; s < num_splits; ++s) {
    const float ms = ml[2 * s];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
    lsum = fmaf(w, ml[2 * s + 1], lsum);
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = fmaf(w, acc[(int64_t)s * D + lane * E + i], v[i]);
  }
  const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] *= inv;
  fwht_warp<E>(v);  // R^T o~ = diag(s) H o~ / sqrt(D)
  const float rs = 1.0f / sqrtf((float)D);
#pragma unroll
  for (int i = 0; i < E; ++i)
    store_from_f32(out, (int64_t)row * D + lane * E + i, out_dtype, v[i] * __ldg(signs + lane * E + i) * rs);
}

template <int E>
cudaError_t launch_split(const DecodeArgs& a, const DecodePlan& p, SplitView part, cudaStream_t stream) {
  const int G = a.num_q_heads / a.num_kv_heads;
  dim3 grid(p.num_splits, a.num_kv_heads, a.batch);
  switch (G) {
    case 1: decode_split_kernel<E, 1><<<grid, kDecodeWarps * 32, 0, stream>>>(a, p.num_splits, p.blocks_per_split, part); break;
    case 2: decode_split_kernel<E, 2><<<grid, kDecodeWarps * 32, 0, stream>>>(a, p.num_splits, p.blocks_per_split, part); break;
    case 4: decode_split_kernel<E, 4><<<grid, kDecodeWarps * 32, 0, stream>>>(a, p.num_splits, p.blocks_per_split, part); break;
    case 8: decode_split_kernel<E, 8><<<grid, kDecodeWarps * 32, 0, stream>>>(a, p.num_splits, p.blocks_per_split, part); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  count_launches(1);
  const int rows = a.batch * a.num_q_heads;
  combine_kernel<E><<<(rows + 7) / 8, 256, 0, stream>>>(rows, p.num_splits, part, a.signs, a.out, a.out_dtype);
  err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

}  // namespace

DecodePlan plan_decode(const DecodeArgs& a, int num_sms) {
  DecodePlan p{};
  if (a.k_bits > 0 && !a.bt_rows && tc_decode_supported(a)) {  // (row-mapped batches: no tensor-core form)
    // Tensor-core kernel: one CTA per SM over the flat block list; partial slots for
    // every (CTA, sequence) pair and warp slot, plus the block prefix sums.
    p.kernel = 2;
    p.num_splits = num_sms;
    p.blocks_per_split = 0;
    const size_t slots = (size_t)tc_partials_per_sequence_split() * (num_sms + a.batch);
    p.workspace_bytes = slots * a.num_q_heads * (a.head_dim + 2) * sizeof(float) + (a.batch + 1) * sizeof(int) + 16;
    return p;
  }
  if (a.k_bits > 0 && a.head_dim <= 128 && prefill_mq_supported(a)) {
    // shapes without a tensor-core decode instantiation (5-bit rows, 3-bit rows paired with
    // other widths, block sizes other than 16, GQA groups 1/2): the multi-query kernel with one sequence per window.  Its
    // D = 256 form (one 8-warp CTA per SM) is no faster than the SIMT kernel for one row
    // per window, so D = 256 decodes stay on the SIMT kernel.
    p.kernel = 3;
    p.mq = plan_prefill_mq(a, num_sms, true);
    p.num_splits = p.mq.nsplit;
    p.workspace_bytes = p.mq.workspace_bytes;
    return p;
  }
  p.kernel = 1;
  const int units = std::max(1, a.batch * a.num_kv_heads);
  const int target = num_sms * 8;
  int splits = (target + units - 1) / units;
  splits = std::max(1, std::min(splits, std::max(1, a.max_blocks_per_seq)));
  p.blocks_per_split = (std::max(1, a.max_blocks_per_seq) + splits - 1) / splits;
  p.num_splits = (std::max(1, a.max_blocks_per_seq) + p.blocks_per_split - 1) / p.blocks_per_split;
  p.workspace_bytes = (size_t)a.batch * a.num_q_heads * p.num_splits * (a.head_dim + 2) * sizeof(float);
  return p;
}

cudaError_t launch_combine_splits(const float* acc, const float* ml, int rows, int nsplit, int head_dim,
                                  const float* signs, void* out, int out_dtype, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  SplitView part;
  part.acc = const_cast<float*>(acc);
  part.ml = const_cast<float*>(ml);
  const int grid = (rows + 7) / 8;
  switch (head_dim) {
    case 32: combine_kernel<1><<<grid, 256, 0, stream>>>(rows, nsplit, part, signs, out, out_dtype); break;
    case 64: combine_kernel<2><<<grid, 256, 0, stream>>>(rows, nsplit, part, signs, out, out_dtype); break;
    case 128: combine_kernel<4><<<grid, 256, 0, stream>>>(rows, nsplit, part, signs, out, out_dtype); break;
    case 256: combine_kernel<8><<<grid, 256, 0, stream>>>(rows, nsplit, part, signs, out, out_dtype); break;
    default: return cudaErrorInvalidValue;
  }
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream) {
  if (a.status) {
    cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
  }
  if (a.batch == 0) return cudaSuccess;
  if (p.kernel == 2) return launch_decode_tc(a, p, stream);
  if (p.kernel == 3) return launch_prefill_mq(a, p.mq, stream);
  if (a.head_dim == 16) return launch_decode_d16(a, stream);
  SplitView part = split_view(a.workspace, a.batch, a.num_q_heads, p.num_splits, a.head_dim);
  switch (a.head_dim) {
    case 32: return launch_split<1>(a, p, part, stream);
    case 64: return launch_split<2>(a, p, part, stream);
    case 128: return launch_split<4>(a, p, part, stream);
    case 256: return launch_split<8>(a, p, part, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq

// ---------------------------------------------------------------------------------
// Fixed scratch for callers that cannot allocate device memory (tq_paged_decode_static).
// The array lives for the life of the process on every device that loads the library.
// Every call shares it, so calls whose work overlaps on the GPU race on it.  The
// decode writes every partial it later reads, so nothing in it needs clearing.
// ---------------------------------------------------------------------------------

namespace tq {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
__device__ __align__(256) unsigned char g_static_decode_scratch[kStaticScratchBytes];

std::mutex g_static_scratch_mutex;
void* g_static_scratch_ptr[128] = {};

}  // namespace

cudaError_t static_decode_scratch(void** ptr, size_t* capacity) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
  if (g_static_scratch_ptr[dev] == nullptr) {
    // The array's name in host code is only a host-side handle; the device address
    // must come from the runtime, with this device current.
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_decode_scratch);
    if (err != cudaSuccess) return err;
    g_static_scratch_ptr[dev] = p;
  }
  *ptr = g_static_scratch_ptr[dev];
  *capacity = kStaticScratchBytes;
  return cudaSuccess;
}

}  // namespace tq
