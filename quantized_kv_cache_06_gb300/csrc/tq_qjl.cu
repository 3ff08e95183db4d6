// Product-quantised ("QJL residual") key rows: writer and paged decode (sm_103a, SIMT forms;
// the tensor-core forms are in tq_write_tc.cu and tq_decode_tc_p.cu / _q.cu).
//
// TurboQuant docs: "vLLM Reference Audit" (File Map: "MSE and QJL codecs" with indices,
// norms and signs, TurboQuantMSE / TurboQuantProd; Feature Checklist: "QJL residual").
// A key row at b bits holds the (b - 1)-bit MSE indices of y = R x / ||x|| (LSB-first),
// then one sign bit per coordinate of S r, r = y - c[idx] the rotated residual and S a
// D x D standard-normal matrix, then nu = ||x|| and gamma = ||r|| as fp32:
// RB = D (b - 1) / 8 + D / 8 + 8.  A query q scores the row as
//   nu (<R q, c[idx]> + gamma sqrt(pi / 2) / D <S R q, 2 z - 1>),
// an estimate of <q, x> that is unbiased over the draw of S.  Values stay MSE rows.
//
// Kernels:
//   write_prod_kernel       (shapes without the tensor-core writer of tq_write_tc.cu: fp32
//                           rows at D = 128) one warp per (token, head) row: norm, rotation (warp FWHT),
//                           indices, residual; the D projections S r come from S^T staged
//                           in shared memory, output i = lane + 32 e, so a warp ballot per
//                           e is directly sign word e of the row.
//   qjl_project_kernel      S^T staged once per CTA; a warp per (sequence, q head): q_rot = R q times the softmax
//                           scale and log2(e) (as the decode uses it) and p = S q_rot,
//                           written to the workspace.
//   decode_prod_split_kernel  the SIMT split decode with the sketch term added to the MSE
//                           score before the warp reduction; the split combine is shared.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "tq_device.cuh"
#include "tq_qjl.h"

namespace tq {
namespace {

constexpr int kProdWarps = 8;
constexpr int kProdDecodeWarps = 4;
constexpr float kProdLog2e = 1.4426950408889634f;
constexpr float kSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi / 2)

template <typename T, int E>
__global__ void __launch_bounds__(kProdWarps * 32)
write_prod_kernel(const T* __restrict__ raw, int64_t num_rows, int num_kv_heads, int bits,
                  const int64_t* __restrict__ slots, uint8_t* __restrict__ pages,
                  const float* __restrict__ signs, const float* __restrict__ centroids,
                  const float* __restrict__ smat, const int32_t* __restrict__ status) {
  constexpr int D = 32 * E;
  extern __shared__ float s_t[];  // S^T, padded: s_t[j * (D + 1) + i] = S[i][j]
  __shared__ float boundary[16], cent[16];
  __shared__ float rbuf[kProdWarps][D];
  __shared__ uint32_t rowbuf[kProdWarps][D * 4 / 32 + D / 32 + 2];

  const int mb = bits - 1;  // MSE bits, 2..4
  const int nc = 1 << mb;
  if (threadIdx.x < nc - 1) boundary[threadIdx.x] = 0.5f * (centroids[threadIdx.x] + centroids[threadIdx.x + 1]);
  if (threadIdx.x < nc) cent[threadIdx.x] = centroids[threadIdx.x];
  for (int k = threadIdx.x; k < D * D; k += blockDim.x) {  // coalesced reads, conflict-free stores
    const int i = k / D, j = k - i * D;
    s_t[j * (D + 1) + i] = __ldg(smat + k);
  }
  __syncthreads();
  if (*status != kOk) return;  // a slot failed validation: write nothing

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int index_words = D * mb / 32;
  const int row_words = index_words + E + 2;
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  float sg[E];
#pragma unroll
  for (int i = 0; i < E; ++i) sg[i] = __ldg(signs + lane * E + i);
  uint32_t* buf = rowbuf[warp];
  float* res = rbuf[warp];

  for (int64_t r = (int64_t)blockIdx.x * kProdWarps + warp; r < num_rows; r += (int64_t)gridDim.x * kProdWarps) {
    const int64_t t = r / num_kv_heads;
    const int h = (int)(r - t * num_kv_heads);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // "Slot Mapping": negative slots are ignored

    float v[E];
    load_chunk<T, E>(raw + r * D + lane * E, v);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(v[i], v[i], ss);
    const float nu = sqrtf(warp_sum(ss));
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] *= sg[i];
    fwht_warp<E>(v);
    const float inv = nu > 0.f ? inv_sqrt_d / nu : 0.f;  // y = H(s*x)/(sqrt(D) nu)

    for (int w = lane; w < row_words; w += 32) buf[w] = 0u;
    __syncwarp();
    float rs = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float u = v[i] * inv;
      int idx = 0;  // #{k : boundary_k < u}
      for (int s = nc >> 1; s > 0; s >>= 1)
        if (u > boundary[idx + s - 1]) idx += s;
      const int bit = (lane * E + i) * mb;
      const int w = bit >> 5, o = bit & 31;
      atomicOr(&buf[w], (uint32_t)idx << o);
      if (o + mb > 32) atomicOr(&buf[w + 1], (uint32_t)idx >> (32 - o));
      const float d = u - cent[idx];
      res[lane * E + i] = d;
      rs = fmaf(d, d, rs);
    }
    const float gamma = sqrtf(warp_sum(rs));
    __syncwarp();
    // sign word e: bit `lane` is [(S r)_(lane + 32 e) >= 0]
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = lane + 32 * e;
      float acc = 0.f;
      for (int j = 0; j < D; ++j) acc = fmaf(s_t[j * (D + 1) + i], res[j], acc);
      const uint32_t mask = __ballot_sync(kFullMask, acc >= 0.f);
      if (lane == 0) buf[index_words + e] = mask;
    }
    if (lane == 0) {
      buf[index_words + E] = __float_as_uint(nu);
      buf[index_words + E + 1] = __float_as_uint(gamma);
    }
    __syncwarp();
    uint32_t* dst = reinterpret_cast<uint32_t*>(pages + (slot * num_kv_heads + h) * (int64_t)(row_words * 4));
    for (int w = lane; w < row_words; w += 32) dst[w] = buf[w];
    __syncwarp();
  }
}

// p[row][i] = sum_j S[i][j] q_rot[j] for row = (sequence, q head), q_rot = R q times the
// softmax scale and log2(e) -- the decode's own rotated query.  A CTA of 8 warps takes
// kProjRows rows per warp: S^T is staged in shared memory once (padded to D + 1 columns, so
// the staging stores and the reads of column i by lane i are conflict free), each query row
// goes through the warp FWHT, and lane l accumulates outputs l + 32 e of the warp's rows
// together over j (one shared load of S^T serves every row; the sum over j runs in order).
// The product-key split kernel is launched as a programmatic dependent of this grid and
// reads p only after waiting for it.
constexpr int kProjRows = 2;
template <int E>
__global__ void __launch_bounds__(256)
qjl_project_kernel(DecodeArgs a, const float* __restrict__ smat, float* __restrict__ p_out) {
  constexpr int D = 32 * E;
  extern __shared__ float s_t[];  // S^T, padded: s_t[j * (D + 1) + i] = S[i][j]
  __shared__ __align__(16) float qs[8][kProjRows][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 16
  for (int k = threadIdx.x; k < D * D; k += blockDim.x) {  // 16 loads in flight per thread
    const int i = k / D, j = k - i * D;
    s_t[j * (D + 1) + i] = __ldg(smat + k);
  }
  __syncthreads();
  // the dependent split grid may be scheduled now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int64_t rows = (int64_t)a.batch * a.num_q_heads;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + warp) * kProjRows;
  if (row0 >= rows) return;
  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kProdLog2e / sqrtf((float)D);
#pragma unroll
  for (int r = 0; r < kProjRows; ++r) {
    float qr[E];
    if (row0 + r < rows) {
#pragma unroll
      for (int i = 0; i < E; ++i)
        qr[i] = load_as_f32(a.q, (row0 + r) * D + lane * E + i, a.q_dtype) * __ldg(a.signs + lane * E + i);
      fwht_warp<E>(qr);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) qr[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < E; ++i) qs[warp][r][lane * E + i] = qr[i] * qmul;
  }
  __syncwarp();
  float acc[kProjRows][E];
#pragma unroll
  for (int r = 0; r < kProjRows; ++r)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
#pragma unroll 2
  for (int j = 0; j < D; j += 4) {
    float4 q4[kProjRows];
#pragma unroll
    for (int r = 0; r < kProjRows; ++r) q4[r] = *reinterpret_cast<const float4*>(&qs[warp][r][j]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float sv = s_t[(j + u) * (D + 1) + lane + 32 * e];
#pragma unroll
        for (int r = 0; r < kProjRows; ++r) {
          const float qj = u == 0 ? q4[r].x : u == 1 ? q4[r].y : u == 2 ? q4[r].z : q4[r].w;
          acc[r][e] = fmaf(sv, qj, acc[r][e]);
        }
      }
  }
#pragma unroll
  for (int r = 0; r < kProjRows; ++r)
    if (row0 + r < rows)
#pragma unroll
      for (int e = 0; e < E; ++e) p_out[(row0 + r) * D + lane + 32 * e] = acc[r][e];
}

// Enqueues the projection of every (sequence, q head) of `a` into p_out [rows][D].
template <int E>
cudaError_t launch_qjl_project(const DecodeArgs& a, const float* smat, float* p_out, cudaStream_t stream) {
  constexpr int D = 32 * E;
  const int64_t rows = (int64_t)a.batch * a.num_q_heads;
  const size_t smem = (size_t)D * (D + 1) * sizeof(float);
  cudaError_t err = cudaFuncSetAttribute(qjl_project_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t per_cta = 8 * kProjRows;
  qjl_project_kernel<E><<<(unsigned)((rows + per_cta - 1) / per_cta), 256, smem, stream>>>(a, smat, p_out);
  err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

struct ProdSplitView {
  float* acc;  // [batch][num_q_heads][num_splits][D]
  float* ml;   // [batch][num_q_heads][num_splits][2]
};

__device__ __forceinline__ int field_of(uint64_t win, int bitpos, int bits) {
  return (int)((win >> bitpos) & ((1u << bits) - 1u));
}

// SIMT split decode over product-quantised key rows and MSE value rows (k_bits is the
// total key width: k_bits - 1 index bits plus the sign bit; k_centroids are the MSE ones).
template <int E, int G>
__global__ void __launch_bounds__(kProdDecodeWarps * 32)
decode_prod_split_kernel(DecodeArgs a, const float* __restrict__ p_all, int num_splits, int blocks_per_split,
                         ProdSplitView part) {
  constexpr int D = 32 * E;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.num_kv_heads, bs = a.block_size;
  const int kmb = a.k_bits - 1;  // key index bits

  __shared__ float ck[32], cv[32];
  __shared__ float red_ml[kProdDecodeWarps][G][2];
  __shared__ float red_acc[kProdDecodeWarps][G][D];

  if (threadIdx.x < (1 << kmb)) ck[threadIdx.x] = a.k_centroids[threadIdx.x];
  if (threadIdx.x < (1 << a.v_bits)) cv[threadIdx.x] = a.v_centroids[threadIdx.x];

  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kProdLog2e / sqrtf((float)D);
  float qr[G][E], pp[G][E];  // rotated query (coordinates lane E + i), projection (lane + 32 e)
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int64_t qrow = (int64_t)b * a.num_q_heads + (int64_t)h * G + g;
#pragma unroll
    for (int i = 0; i < E; ++i) qr[g][i] = load_as_f32(a.q, qrow * D + lane * E + i, a.q_dtype) * __ldg(a.signs + lane * E + i);
    fwht_warp<E>(qr[g]);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      qr[g][i] *= qmul;
      pp[g][i] = __ldg(p_all + qrow * D + lane + 32 * i);
    }
  }

  int len = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks_per_seq * bs;
  if (len < 0 || len > cap) {
    if (threadIdx.x == 0 && split == 0 && h == 0 && a.status) atomicMax(a.status, (int32_t)kInvalidArg);
    len = len < 0 ? 0 : cap;
  }
  const int t_lo = split * blocks_per_split * bs;
  const int t_hi = min(len, (split + 1) * blocks_per_split * bs);

  const int kib = D * kmb / 8, vib = D * a.v_bits / 8;  // index bytes
  const int64_t krb = kib + D / 8 + 8, vrb = vib + 4;     // row bytes
  const int kbit0 = lane * E * kmb, vbit0 = lane * E * a.v_bits;
  const float sketch = kSqrtHalfPi / (float)D;

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
  for (int t = t_lo + warp; t < t_hi; t += kProdDecodeWarps) {
    const int bid = __ldg(a.block_table + (int64_t)b * a.max_blocks_per_seq + t / bs);
    if (bid < 0 || (int64_t)bid >= a.num_blocks) {
      bad_block = true;
      continue;
    }
    const int64_t row = ((int64_t)bid * bs + t % bs) * H + h;
    const uint32_t* kr = reinterpret_cast<const uint32_t*>(a.k_pages + row * krb);
    const uint32_t* vr = reinterpret_cast<const uint32_t*>(a.v_pages + row * vrb);

    const uint64_t kwin = (uint64_t)__ldg(kr + (kbit0 >> 5)) | ((uint64_t)__ldg(kr + (kbit0 >> 5) + 1) << 32);
    const uint64_t vwin = (uint64_t)__ldg(vr + (vbit0 >> 5)) | ((uint64_t)__ldg(vr + (vbit0 >> 5) + 1) << 32);
    uint32_t zw[E];
#pragma unroll
    for (int e = 0; e < E; ++e) zw[e] = __ldg(kr + kib / 4 + e);
    const float knorm = __uint_as_float(__ldg(kr + kib / 4 + E));
    const float kgamma = __uint_as_float(__ldg(kr + kib / 4 + E + 1));
    const float vnorm = __uint_as_float(__ldg(vr + vib / 4));

    float s[G], zs[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = zs[g] = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float c = ck[field_of(kwin, (kbit0 & 31) + i * kmb, kmb)];
      const float zsign = ((zw[i] >> lane) & 1u) ? 1.f : -1.f;  // coordinate lane + 32 i
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s[g] = fmaf(qr[g][i], c, s[g]);
        zs[g] = fmaf(pp[g][i], zsign, zs[g]);
      }
    }
    float vv[E];
#pragma unroll
    for (int i = 0; i < E; ++i) vv[i] = vnorm * cv[field_of(vwin, (vbit0 & 31) + i * a.v_bits, a.v_bits)];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sc = warp_sum(fmaf(kgamma * sketch, zs[g], s[g])) * knorm;
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

  // merge the warps of this CTA, then write the split partial
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
  for (int g = warp; g < G; g += kProdDecodeWarps) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kProdDecodeWarps; ++w) mx = fmaxf(mx, red_ml[w][g][0]);
    float wt[kProdDecodeWarps], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kProdDecodeWarps; ++w) {
      wt[w] = red_ml[w][g][0] == -INFINITY ? 0.f : exp2f(red_ml[w][g][0] - mx);
      lsum = fmaf(wt[w], red_ml[w][g][1], lsum);
    }
    const int64_t slot = ((int64_t)b * a.num_q_heads + (int64_t)h * G + g) * num_splits + split;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kProdDecodeWarps; ++w) sum = fmaf(wt[w], red_acc[w][g][lane * E + i], sum);
      part.acc[slot * D + lane * E + i] = sum;
    }
    if (lane == 0) {
      part.ml[slot * 2 + 0] = mx;
      part.ml[slot * 2 + 1] = lsum;
    }
  }
}

template <int E>
cudaError_t launch_prod_decode_e(const DecodeArgs& a, const float* smat, const DecodePlan& p, cudaStream_t stream) {
  constexpr int D = 32 * E;
  const int64_t qrows = (int64_t)a.batch * a.num_q_heads;
  ProdSplitView part;
  part.acc = static_cast<float*>(a.workspace);
  part.ml = part.acc + (size_t)qrows * p.num_splits * D;
  float* p_all = part.ml + (size_t)qrows * p.num_splits * 2;
  cudaError_t err = launch_qjl_project<E>(a, smat, p_all, stream);
  if (err != cudaSuccess) return err;
  const int G = a.num_q_heads / a.num_kv_heads;
  dim3 grid(p.num_splits, a.num_kv_heads, a.batch);
  switch (G) {
    case 1: decode_prod_split_kernel<E, 1><<<grid, kProdDecodeWarps * 32, 0, stream>>>(a, p_all, p.num_splits, p.blocks_per_split, part); break;
    case 2: decode_prod_split_kernel<E, 2><<<grid, kProdDecodeWarps * 32, 0, stream>>>(a, p_all, p.num_splits, p.blocks_per_split, part); break;
    case 4: decode_prod_split_kernel<E, 4><<<grid, kProdDecodeWarps * 32, 0, stream>>>(a, p_all, p.num_splits, p.blocks_per_split, part); break;
    case 8: decode_prod_split_kernel<E, 8><<<grid, kProdDecodeWarps * 32, 0, stream>>>(a, p_all, p.num_splits, p.blocks_per_split, part); break;
    default: return cudaErrorInvalidValue;
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  count_launches(1);
  return launch_combine_splits(part.acc, part.ml, (int)qrows, p.num_splits, D, a.signs, a.out, a.out_dtype, stream);
}

}  // namespace

bool prod_supported(int head_dim, int bits) { return (head_dim == 64 || head_dim == 128) && bits >= 3 && bits <= 5; }

namespace {
// The tensor-core form: one CTA per SM, the split partials and prefix sums of the
// tensor-core decode, then p (16-byte aligned).
DecodePlan prod_tc_plan(const DecodeArgs& a) {
  DecodePlan p{};
  p.kernel = 2;
  p.num_splits = device_sms();
  const size_t slots = (size_t)tc_partials_per_sequence_split() * (p.num_splits + std::max(0, a.batch));
  p.workspace_bytes =
      (slots * a.num_q_heads * (a.head_dim + 2) * sizeof(float) + (std::max(0, a.batch) + 1) * sizeof(int) + 15) / 16 * 16;
  return p;
}
}  // namespace

size_t prod_decode_workspace(const DecodeArgs& a, const DecodePlan& p) {
  const size_t qrows = (size_t)std::max(0, a.batch) * a.num_q_heads;
  const size_t simt = qrows * p.num_splits * (a.head_dim + 2) * sizeof(float) + qrows * a.head_dim * sizeof(float) + 16;
  const size_t tc = prod_tc_plan(a).workspace_bytes + qrows * a.head_dim * sizeof(float) + 16;
  return std::max(simt, tc);  // either form fits, whatever the widths
}

cudaError_t launch_write_prod(const WriteArgs& a, const float* smat, cudaStream_t stream, int num_sms) {
  cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  if (a.num_tokens == 0) return cudaSuccess;
  err = launch_validate_slots(a, stream, num_sms);
  if (err != cudaSuccess) return err;
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  if (write_prod_tc_supported(a)) {
    const int64_t tiles = (rows + 15) / 16;
    return launch_write_prod_tc(a, smat, stream,
                                (int)std::max<int64_t>(1, std::min<int64_t>((tiles + 7) / 8, (int64_t)num_sms * 2)));
  }
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + kProdWarps - 1) / kProdWarps, (int64_t)num_sms * 3));
  const size_t smem = (size_t)a.head_dim * (a.head_dim + 1) * sizeof(float);
#define TQ_PROD_W(T, E)                                                                                       \
  {                                                                                                           \
    auto kern = write_prod_kernel<T, E>;                                                                      \
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);                 \
    if (err != cudaSuccess) return err;                                                                       \
    kern<<<grid, kProdWarps * 32, smem, stream>>>(static_cast<const T*>(a.raw), rows, a.num_kv_heads, a.bits, \
                                                  a.slots, a.pages, a.signs, a.centroids, smat, a.status);    \
    err = cudaGetLastError();                                                                                 \
    if (err == cudaSuccess) count_launches(1);                                                                \
    return err;                                                                                               \
  }
  const int E = a.head_dim / 32;
  if (a.dtype == kF16) {
    if (E == 2) TQ_PROD_W(__half, 2)
    if (E == 4) TQ_PROD_W(__half, 4)
  } else if (a.dtype == kBF16) {
    if (E == 2) TQ_PROD_W(__nv_bfloat16, 2)
    if (E == 4) TQ_PROD_W(__nv_bfloat16, 4)
  } else {
    if (E == 2) TQ_PROD_W(float, 2)
    if (E == 4) TQ_PROD_W(float, 4)
  }
#undef TQ_PROD_W
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_prod(const DecodeArgs& a, const float* smat, const DecodePlan& p, cudaStream_t stream) {
  if (a.status) {
    cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
  }
  if (a.batch == 0) return cudaSuccess;
  if (tc_prod_decode_supported(a)) {
    // p = S q~ after the tensor-core partials, then the tensor-core split kernel and combine
    const DecodePlan tp = prod_tc_plan(a);
    float* p_all = reinterpret_cast<float*>(static_cast<unsigned char*>(a.workspace) + tp.workspace_bytes);
    const cudaError_t err = launch_qjl_project<4>(a, smat, p_all, stream);
    if (err != cudaSuccess) return err;
    return launch_tc_prod(a, tp, p_all, stream);
  }
  if (a.head_dim == 64) return launch_prod_decode_e<2>(a, smat, p, stream);
  if (a.head_dim == 128) return launch_prod_decode_e<4>(a, smat, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace tq
