// Recipe cache modes turboquant25 / turboquant35: grouped product-quantised rows, writer
// and paged decode (sm_103a, SIMT).
//
// TurboQuant docs: "vLLM Usage" (Cache Dtypes: turboquant25 and turboquant35, recipe
// modes require metadata; Metadata Validation Rules; Page Geometry: recipe row bytes) and
// "Architecture" (vLLM Runtime Mapping: channels selected by energy, recipe vector rows
// pack and unpack grouped MSE+QJL rows); "vLLM Reference Audit" lists the recipe update
// and decode kernels as missing.
//
// Row (a reading: the pages name the parts, not the numbers).  A row's D channels form a
// high group and a low group of d = D / 2 channels; order[h][0, D) lists kv head h's high
// group (sorted), then its low group (the complement, ascending).  Group g is one
// product-quantised vector of dimension d at bits_g (turboquant25: 3 and 2, turboquant35:
// 4 and 3 -- the recipe name is the mean bits per channel): the (bits_g - 1)-bit MSE
// indices of y = R_d x_g / ||x_g|| (LSB first), one sign bit per coordinate of S_d r
// (r = y - c[idx], bit = 1 for a non-negative projection), then nu_g = ||x_g|| and
// gamma_g = ||r|| as fp32.  The row holds the high group's bytes, then the low group's.
// R_d (RHT of dimension d) and S_d (d x d standard normal) are shared by both groups and
// by K and V, which both use recipe rows.
//
// Kernels:
//   write_recipe_kernel        a warp per sixteen (token, head, group) units: channel gather,
//                              norm, rotation (warp FWHT), indices and residual of each, then
//                              the sketch of the sixteen as m16n8k16 MMAs (fp16 hi / lo
//                              splits of r and S_d) and the sign words from ballots.
//   recipe_project_kernel      one warp per (sequence, q head): per group the rotated
//                              gathered query q_g = R_d q[order_g] (times the softmax scale
//                              and log2 e) and its projection p_g = S_d q_g.
//   decode_recipe_split_kernel the SIMT split decode, 32-token tiles per warp: scores with
//                              a lane per token (every q head at once), one softmax step
//                              per tile, values with lanes over coordinates.  Score of key
//                              row k:
//                                sum_g nu_g (<q_g, c_g[idx]> + gamma_g kappa <p_g, 2z - 1>),
//                              kappa = sqrt(pi / 2) / d.  The value reconstruction
//                              nu R_d^T (c[idx] + gamma kappa S_d^T (2z - 1)) is linear, so
//                              the kernel keeps two accumulators per group,
//                              sum p nu c[idx] and sum p nu gamma kappa (2z - 1), and no
//                              per-token S_d^T product is needed.
//   combine_recipe_kernel      one warp per (sequence, q head): merges the splits, then per
//                              group w = acc_c + S_d^T acc_z, R_d^T w / l, scattered back to
//                              the group's channels.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "tq_device.cuh"
#include "tq_recipe.h"

namespace tq {
namespace {

constexpr int kRecWarps = 8;
constexpr int kRecDecodeWarps = 4;
constexpr float kRecLog2e = 1.4426950408889634f;
constexpr float kRecSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi / 2)

// 32-bit words of group g's part of a row: d (b - 1) / 32 index words, d / 32 sign words,
// nu, gamma.
__host__ __device__ constexpr int group_words(int d, int bits) { return d * (bits - 1) / 32 + d / 32 + 2; }

// Units (row, group) are taken sixteen at a time per warp (eight rows, both groups), in
// batches of four: each unit's gather, norm, rotation, indices and residual (the four units'
// loads issued together, their reductions interleaved), the residual r stored into the warp's
// A tile as fp16 hi = r 2^10 and lo = (r 2^10 - hi) 2^12.  Then the sketch S_d r of the
// sixteen on the tensor cores (m16n8k16): r_hi S_hi into one accumulator, r_lo S_hi +
// r_hi S_lo into another (~22 significant bits, as in an fp32 sum), and each sign word from
// ballots of the accumulators, assembled by one lane.
constexpr int kRecUnits = 16;
constexpr int kRecBatch = 4;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void rec_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void rec_ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
// bit c of a nibble to bit 2 c
__device__ __forceinline__ uint32_t spread_nibble(uint32_t x) {
  x = (x | (x << 2)) & 0x33u;
  return (x | (x << 1)) & 0x55u;
}

// Shared memory of the writer: S hi and lo, then per warp its A tile hi and lo; rows of
// d + 8 halves (16 bytes of padding put the 8 rows of an ldmatrix in different banks).
__host__ __device__ constexpr int recipe_write_smem(int d) { return (2 * d + kRecWarps * 2 * kRecUnits) * (d + 8) * 2; }

// idx = #{k : b_k < y} over the 2^MB - 1 decision points held in registers (ties and NaN: the
// lower index)
template <int MB>
__device__ __forceinline__ int rec_index(float y, const float (&b)[7]) {
  int idx = 0;
#pragma unroll
  for (int k = 0; k < (1 << MB) - 1; ++k) idx += y > b[k] ? 1 : 0;
  return idx;
}

// MB0 / MB1: MSE index bits of the high / low group.
template <typename T, int E, int MB0, int MB1>
__global__ void __launch_bounds__(kRecWarps * 32, 3)
write_recipe_kernel(const T* __restrict__ raw, int64_t num_rows, int num_kv_heads, const int64_t* __restrict__ slots,
                    uint8_t* __restrict__ pages, RecipeArgs rc, const float* __restrict__ signs,
                    const int32_t* __restrict__ status) {
  constexpr int d = 32 * E, D = 2 * d;
  constexpr int kUnitWords = 3 * E + E + 2;  // largest group: 3-bit indices, signs, nu, gamma
  constexpr int kRow = d + 8;
  extern __shared__ __align__(16) unsigned char rec_smem[];
  __half* s_hi = reinterpret_cast<__half*>(rec_smem);  // S[i][j] (i: projection, j: coordinate)
  __half* s_lo = s_hi + d * kRow;                       // (S - hi) 2^12
  __shared__ float cen[2][8];
  __shared__ uint32_t rowbuf[kRecWarps][kRecUnits][kUnitWords];
  __shared__ int64_t slot_s[kRecWarps][kRecUnits];
  __shared__ int head_s[kRecWarps][kRecUnits];

  const int tid = threadIdx.x;
  constexpr int mb0 = MB0, mb1 = MB1;
  constexpr int nc0 = 1 << MB0, nc1 = 1 << MB1;
  // the decision points of both groups, in registers
  float bhi[7], blo[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    bhi[k] = k < nc0 - 1 ? 0.5f * (__ldg(rc.mse_hi + k) + __ldg(rc.mse_hi + k + 1)) : INFINITY;
    blo[k] = k < nc1 - 1 ? 0.5f * (__ldg(rc.mse_lo + k) + __ldg(rc.mse_lo + k + 1)) : INFINITY;
  }
  if (tid < nc0) cen[0][tid] = rc.mse_hi[tid];
  if (tid < nc1) cen[1][tid] = rc.mse_lo[tid];
  for (int k = tid; k < d * d; k += blockDim.x) {
    const int i = k / d, j = k - i * d;
    const float sv = __ldg(rc.smat + k);
    const __half hi = __float2half_rn(sv);
    s_hi[i * kRow + j] = hi;
    s_lo[i * kRow + j] = __float2half_rn((sv - __half2float(hi)) * 4096.0f);
  }
  __syncthreads();
  if (*status != kOk) return;  // a slot failed validation: write nothing

  const int warp = tid >> 5, lane = tid & 31;
  const int row_words = group_words(d, rc.bits_hi) + group_words(d, rc.bits_lo);
  const float inv_sqrt_d = 1.0f / sqrtf((float)d);
  float sg[E];
#pragma unroll
  for (int i = 0; i < E; ++i) sg[i] = __ldg(signs + lane * E + i);
  __half* a_hi = s_lo + d * kRow + warp * (2 * kRecUnits * kRow);  // this warp's A tile: unit k, coordinate j
  __half* a_lo = a_hi + kRecUnits * kRow;
  // ldmatrix lane addresses: A rows (units) lane & 15, k half lane >> 4; B rows (projections)
  // (lane & 7) + 8 (lane >> 4), k half (lane >> 3) & 1
  const uint32_t a_lane = smem_u32(a_hi) + (uint32_t)(((lane & 15) * kRow + (lane >> 4) * 8) * 2);
  const uint32_t a_lo_off = (uint32_t)(kRecUnits * kRow * 2);
  const uint32_t b_lane = smem_u32(s_hi) + (uint32_t)((((lane & 7) + 8 * (lane >> 4)) * kRow + ((lane >> 3) & 1) * 8) * 2);
  const uint32_t b_lo_off = (uint32_t)(d * kRow * 2);

  const int64_t units = 2 * num_rows;
  const int64_t ustride = (int64_t)gridDim.x * kRecWarps * kRecUnits;
  for (int64_t u0 = ((int64_t)blockIdx.x * kRecWarps + warp) * kRecUnits; u0 < units; u0 += ustride) {
#pragma unroll 1
    for (int q = 0; q < kRecUnits / kRecBatch; ++q) {
      const int64_t ub = u0 + kRecBatch * q;  // units ub .. ub + 3: rows r0, r0 + 1, both groups
      int64_t slot_k[kRecBatch];
      float nu_k[kRecBatch], gamma_k[kRecBatch];
      float v[kRecBatch][E];
      const int64_t r0 = ub >> 1;
      const int64_t t0 = r0 / num_kv_heads;
      const int h0 = (int)(r0 - t0 * num_kv_heads);
      const bool wrap = h0 + 1 == num_kv_heads;
      const int64_t t1 = wrap ? t0 + 1 : t0;
      const int h1 = wrap ? 0 : h0 + 1;
#pragma unroll
      for (int k = 0; k < kRecBatch; ++k) {
        const int64_t u = ub + k;
        const int64_t r = r0 + (k >> 1);
        const int g = k & 1;
        const int64_t t = (k >> 1) ? t1 : t0;
        const int h = (k >> 1) ? h1 : h0;
        slot_k[k] = u < units ? __ldg(slots + t) : -1;
        const int32_t* ord = rc.order + (int64_t)h * D + g * d + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) v[k][i] = u < units ? to_f32<T>(raw[r * D + __ldg(ord + i)]) : 0.f;
        if (lane == 0) {
          slot_s[warp][kRecBatch * q + k] = slot_k[k];
          head_s[warp][kRecBatch * q + k] = h;
        }
      }
#pragma unroll
      for (int k = 0; k < kRecBatch; ++k) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) ss = fmaf(v[k][i], v[k][i], ss);
        nu_k[k] = ss;
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
        for (int k = 0; k < kRecBatch; ++k) nu_k[k] += __shfl_xor_sync(kFullMask, nu_k[k], m);
#pragma unroll
      for (int k = 0; k < kRecBatch; ++k) {
        nu_k[k] = sqrtf(nu_k[k]);
#pragma unroll
        for (int i = 0; i < E; ++i) v[k][i] *= sg[i];
        fwht_warp<E>(v[k]);
      }
#pragma unroll
      for (int k = 0; k < kRecBatch; ++k) {
        const int g = k & 1;
        const int uk = kRecBatch * q + k;
        uint32_t* buf = rowbuf[warp][uk];
        __half* arow_hi = a_hi + uk * kRow + lane * E;
        __half* arow_lo = a_lo + uk * kRow + lane * E;
        gamma_k[k] = 0.f;
        if (slot_k[k] < 0) {  // "Slot Mapping": negative slots are ignored (zero residual)
#pragma unroll
          for (int i = 0; i < E; ++i) arow_hi[i] = arow_lo[i] = __float2half_rn(0.f);
          continue;
        }
        const int mb = g ? mb1 : mb0;
        const float nu = nu_k[k];
        const float inv = nu > 0.f ? inv_sqrt_d / nu : 0.f;  // y = H(s*x)/(sqrt(d) nu)

        const int index_words = d * mb / 32;
        for (int w = lane; w < index_words; w += 32) buf[w] = 0u;
        __syncwarp();
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const float y = v[k][i] * inv;
          const int idx = g ? rec_index<MB1>(y, blo) : rec_index<MB0>(y, bhi);
          const int bit = (lane * E + i) * mb;
          const int w = bit >> 5, o = bit & 31;
          atomicOr(&buf[w], (uint32_t)idx << o);
          if (o + mb > 32) atomicOr(&buf[w + 1], (uint32_t)idx >> (32 - o));
          const float dr = y - cen[g][idx];
          rs = fmaf(dr, dr, rs);
          const float x = dr * 1024.0f;
          const __half xh = __float2half_rn(x);
          arow_hi[i] = xh;
          arow_lo[i] = __float2half_rn((x - __half2float(xh)) * 4096.0f);
        }
        gamma_k[k] = rs;
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
        for (int k = 0; k < kRecBatch; ++k) gamma_k[k] += __shfl_xor_sync(kFullMask, gamma_k[k], m);
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kRecBatch; ++k) {
          if (slot_k[k] < 0) continue;
          const int iw = d * ((k & 1) ? mb1 : mb0) / 32;
          rowbuf[warp][kRecBatch * q + k][iw + E] = __float_as_uint(nu_k[k]);
          rowbuf[warp][kRecBatch * q + k][iw + E + 1] = __float_as_uint(sqrtf(gamma_k[k]));
        }
      }
    }
    __syncwarp();
    // ---- sketch of the sixteen residuals: sign word e holds projections 32 e .. 32 e + 31
    // (n-tiles 4 e .. 4 e + 3); lane u < 16 assembles unit u's word
    const int u = lane & 15, ur = u & 7, uh = u >> 3;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      uint32_t word = 0u;
#pragma unroll
      for (int np = 0; np < 2; ++np) {  // n-tiles 4 e + 2 np and 4 e + 2 np + 1
        float am[2][4], al[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) am[n][x] = al[n][x] = 0.f;
#pragma unroll
        for (int ks = 0; ks < d / 16; ++ks) {
          uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
          rec_ldsm_x4(a_lane + ks * 32, h0, h1, h2, h3);
          rec_ldsm_x4(a_lane + a_lo_off + ks * 32, l0, l1, l2, l3);
          const uint32_t boff = (uint32_t)((32 * e + 16 * np) * kRow * 2 + ks * 32);
          uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
          rec_ldsm_x4(b_lane + boff, b0, b1, b2, b3);
          rec_ldsm_x4(b_lane + b_lo_off + boff, c0, c1, c2, c3);
          rec_mma(am[0], h0, h1, h2, h3, b0, b1);
          rec_mma(am[1], h0, h1, h2, h3, b2, b3);
          rec_mma(al[0], l0, l1, l2, l3, b0, b1);
          rec_mma(al[1], l0, l1, l2, l3, b2, b3);
          rec_mma(al[0], h0, h1, h2, h3, c0, c1);
          rec_mma(al[1], h0, h1, h2, h3, c2, c3);
        }
        // accumulator x of n-tile 4 e + 2 np + n on lane (g, c): unit g + 8 (x >> 1),
        // projection 32 e + 8 (2 np + n) + 2 c + (x & 1); its ballot bit 4 g + c
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const uint32_t bal = __ballot_sync(kFullMask, fmaf(al[n][x], 1.0f / 4096, am[n][x]) >= 0.f);
            if ((x >> 1) == uh) word |= spread_nibble((bal >> (4 * ur)) & 15u) << (8 * (2 * np + n) + (x & 1));
          }
      }
      if (lane < 16 && slot_s[warp][u] >= 0) rowbuf[warp][u][d * ((u & 1) ? mb1 : mb0) / 32 + e] = word;
    }
    __syncwarp();
    for (int k = 0; k < kRecUnits; ++k) {
      const int64_t slot = slot_s[warp][k];
      if (slot < 0) continue;  // (the same on every lane)
      const int g = k & 1;
      const int gw = d * (g ? mb1 : mb0) / 32 + E + 2;
      uint32_t* dst = reinterpret_cast<uint32_t*>(pages + (slot * num_kv_heads + head_s[warp][k]) * (int64_t)(row_words * 4)) +
                      (g ? group_words(d, rc.bits_hi) : 0);
      for (int w = lane; w < gw; w += 32) dst[w] = rowbuf[warp][k][w];
    }
    __syncwarp();
  }
}

// p[row][g][i] = sum_j S[i][j] q_g[j], q_g = R_d q[row][order_g] times the softmax scale
// and log2(e) (the decode's own rotated query), row = (sequence, q head).
template <int E>
__global__ void __launch_bounds__(256)
recipe_project_kernel(DecodeArgs a, RecipeArgs rc, float* __restrict__ p_out) {
  constexpr int d = 32 * E, D = 2 * d;
  __shared__ float qs[8][2][d];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= (int64_t)a.batch * a.num_q_heads) return;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int h = (int)(row % a.num_q_heads) / G;
  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kRecLog2e / sqrtf((float)d);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    float qr[E];
    const int32_t* ord = rc.order + (int64_t)h * D + g * d + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i) qr[i] = load_as_f32(a.q, row * D + __ldg(ord + i), a.q_dtype) * __ldg(a.signs + lane * E + i);
    fwht_warp<E>(qr);
#pragma unroll
    for (int i = 0; i < E; ++i) qs[warp][g][lane * E + i] = qr[i] * qmul;
  }
  __syncwarp();
#pragma unroll
  for (int g = 0; g < 2; ++g)
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = lane + 32 * e;
      float acc = 0.f;
      for (int j = 0; j < d; ++j) acc = fmaf(__ldg(rc.smat + (int64_t)i * d + j), qs[warp][g][j], acc);
      p_out[(row * 2 + g) * d + i] = acc;
    }
}

struct RecipeSplitView {
  float* acc;  // [rows][nsplit][2 D]: acc_c (group-major, coordinate j), then acc_z (coordinate i)
  float* ml;   // [rows][nsplit][2]  (running max in log2 units, sum)
};

__device__ __forceinline__ int rfield(uint64_t win, int bitpos, int bits) {
  return (int)((win >> bitpos) & ((1u << bits) - 1u));
}

// One group of one packed row, as this lane needs it: the MSE indices of coordinates
// lane E + i, the sign words (bit `lane` of word e: coordinate lane + 32 e), nu, gamma.
template <int E>
struct GroupView {
  int idx[E];
  uint32_t zw[E];
  float nu, gamma;
};

template <int E>
__device__ __forceinline__ GroupView<E> read_group(const uint32_t* __restrict__ gw, int mb, int lane) {
  constexpr int d = 32 * E;
  GroupView<E> v;
  const int bit0 = lane * E * mb;
  const uint64_t win = (uint64_t)__ldg(gw + (bit0 >> 5)) | ((uint64_t)__ldg(gw + (bit0 >> 5) + 1) << 32);
#pragma unroll
  for (int i = 0; i < E; ++i) v.idx[i] = rfield(win, (bit0 & 31) + i * mb, mb);
  const int iw = d * mb / 32;
#pragma unroll
  for (int e = 0; e < E; ++e) v.zw[e] = __ldg(gw + iw + e);
  v.nu = __uint_as_float(__ldg(gw + iw + E));
  v.gamma = __uint_as_float(__ldg(gw + iw + E + 1));
  return v;
}

// Score of one key group for every q head of the kv head, by one lane for its own token:
// sc[g] += nu (sum_j q_g[j] c[idx_j] + gamma kappa sum_j p_g[j] (2 z_j - 1)), with
// sum_j p_g[j] (2 z_j - 1) = 2 sum_j z_j p_g[j] - sum_j p_g[j].  q and p come from shared
// memory ([coordinate][head], the same address on every lane).
// read_group from a row staged in shared memory
template <int E>
__device__ __forceinline__ GroupView<E> read_group_s(const uint32_t* gw, int mb, int lane) {
  constexpr int d = 32 * E;
  GroupView<E> v;
  const int bit0 = lane * E * mb;
  const uint64_t win = (uint64_t)gw[bit0 >> 5] | ((uint64_t)gw[(bit0 >> 5) + 1] << 32);
#pragma unroll
  for (int i = 0; i < E; ++i) v.idx[i] = rfield(win, (bit0 & 31) + i * mb, mb);
  const int iw = d * mb / 32;
#pragma unroll
  for (int e = 0; e < E; ++e) v.zw[e] = gw[iw + e];
  v.nu = __uint_as_float(gw[iw + E]);
  v.gamma = __uint_as_float(gw[iw + E + 1]);
  return v;
}

// PAIRS: the group's words start 8-byte aligned and are even in number (64-bit loads).
template <int E, int G, int MB, bool PAIRS>
__device__ __forceinline__ void recipe_group_score(const uint32_t* __restrict__ gw, const float (*qs)[G],
                                                   const float (*ps)[G], const float* cent, const float* psum,
                                                   float kappa, float (&sc)[G]) {
  constexpr int d = 32 * E, IW = d * MB / 32;
  uint32_t w[IW + E + 2];
  if constexpr (PAIRS) {
#pragma unroll
    for (int k = 0; k < (IW + E + 2) / 2; ++k) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(gw) + k);
      w[2 * k] = x.x;
      w[2 * k + 1] = x.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < IW + E + 2; ++k) w[k] = __ldg(gw + k);
  }
  float sm[G], sz[G];
#pragma unroll
  for (int g = 0; g < G; ++g) sm[g] = sz[g] = 0.f;
#pragma unroll
  for (int j = 0; j < d; ++j) {
    const int bit = j * MB, wi = bit >> 5, o = bit & 31;
    uint32_t f = w[wi] >> o;
    if (o + MB > 32) f |= w[wi + 1] << (32 - o);
    const float c = cent[f & ((1u << MB) - 1u)];
    const float z = (float)((w[IW + (j >> 5)] >> (j & 31)) & 1u);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      sm[g] = fmaf(qs[j][g], c, sm[g]);
      sz[g] = fmaf(ps[j][g], z, sz[g]);
    }
  }
  const float nu = __uint_as_float(w[IW + E]), gk = __uint_as_float(w[IW + E + 1]) * kappa;
#pragma unroll
  for (int g = 0; g < G; ++g) sc[g] = fmaf(nu, fmaf(gk, fmaf(2.f, sz[g], -psum[g]), sm[g]), sc[g]);
}

// Tiles of 32 tokens per warp.  Scores: lane = token, every q head of the kv head at once
// (no per-token reductions); the tile's softmax step (running max, correction, weights) once
// per tile; values: lanes over coordinates, the tile's tokens accumulated with their weights
// from shared memory.  MB0 / MB1: MSE index bits of the high / low group.
template <int E, int G, int MB0, int MB1>
__global__ void __launch_bounds__(kRecDecodeWarps * 32)
decode_recipe_split_kernel(DecodeArgs a, RecipeArgs rc, const float* __restrict__ p_all, int num_splits,
                           int blocks_per_split, RecipeSplitView part) {
  constexpr int d = 32 * E, D = 2 * d;
  constexpr int kWh = d * MB0 / 32 + E + 2;  // words of the high group
  constexpr int rbw = kWh + d * MB1 / 32 + E + 2;  // words of a row
  // rows and both groups 8-byte aligned (pages are 16-byte aligned): 64-bit row loads
  constexpr bool kPairs = rbw % 2 == 0 && kWh % 2 == 0 && (d * MB1 / 32 + E + 2) % 2 == 0;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.num_kv_heads, bs = a.block_size;

  __shared__ float cent[2][8];
  __shared__ __align__(16) float qs[2][d][G];  // rotated query, coordinate j of group grp, head g
  __shared__ __align__(16) float ps[2][d][G];  // its projection p = S_d q, coordinate j
  __shared__ float psum[2][G];                 // sum_j p[j]
  __shared__ __align__(16) float pt[kRecDecodeWarps][32][G];  // the tile's weights (0: no token)
  __shared__ int64_t trow[kRecDecodeWarps][32];               // the tile's page rows (-1: none)
  __shared__ float red_ml[kRecDecodeWarps][G][2];
  // The tile's value rows (fetched by the lane of each token while it scores it; an odd row
  // stride keeps those stores conflict free), sharing memory with the final merge's buffer.
  constexpr int kVStride = (rbw % 2 == 0) ? rbw + 1 : rbw;
  constexpr int kRedBytes = kRecDecodeWarps * G * 2 * D * 4, kVBytes = kRecDecodeWarps * 32 * kVStride * 4;
  __shared__ __align__(16) unsigned char merge_u[kRedBytes > kVBytes ? kRedBytes : kVBytes];
  float(*red_acc)[G][2 * D] = reinterpret_cast<float(*)[G][2 * D]>(merge_u);
  uint32_t(*vbuf)[32][kVStride] = reinterpret_cast<uint32_t(*)[32][kVStride]>(merge_u);
  if (threadIdx.x < (1 << MB0)) cent[0][threadIdx.x] = rc.mse_hi[threadIdx.x];
  if (threadIdx.x < (1 << MB1)) cent[1][threadIdx.x] = rc.mse_lo[threadIdx.x];

  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kRecLog2e / sqrtf((float)d);
  const float kappa = kRecSqrtHalfPi / (float)d;
  for (int g = warp; g < G; g += kRecDecodeWarps) {
    const int64_t qrow = (int64_t)b * a.num_q_heads + (int64_t)h * G + g;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      float qr[E];
      const int32_t* ord = rc.order + (int64_t)h * D + grp * d + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        qr[i] = load_as_f32(a.q, qrow * D + __ldg(ord + i), a.q_dtype) * __ldg(a.signs + lane * E + i);
      fwht_warp<E>(qr);
      float ssum = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        qs[grp][lane * E + i][g] = qr[i] * qmul;
        const float pv = __ldg(p_all + (qrow * 2 + grp) * d + lane + 32 * i);
        ps[grp][lane + 32 * i][g] = pv;
        ssum += pv;
      }
      ssum = warp_sum(ssum);
      if (lane == 0) psum[grp][g] = ssum;
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

  float m[G], l[G], acc_c[G][2][E], acc_z[G][2][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int i = 0; i < E; ++i) acc_c[g][grp][i] = acc_z[g][grp][i] = 0.f;
  }
  __syncthreads();

  bool bad_block = false;
  for (int tb = t_lo + 32 * warp; tb < t_hi; tb += 32 * kRecDecodeWarps) {
    // ---- scores: this lane's token ---------------------------------------------------
    const int t = tb + lane;
    int64_t row = -1;
    if (t < t_hi) {
      const int bid = __ldg(a.block_table + (int64_t)b * a.max_blocks_per_seq + t / bs);
      if (bid < 0 || (int64_t)bid >= a.num_blocks) bad_block = true;
      else row = ((int64_t)bid * bs + t % bs) * H + h;
    }
    float sc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) sc[g] = row >= 0 ? 0.f : -INFINITY;
    if (row >= 0) {
      const uint32_t* vr = reinterpret_cast<const uint32_t*>(a.v_pages) + row * rbw;
      uint32_t vw[rbw];  // this token's value row, in flight while the key row is scored
      if constexpr (kPairs) {
#pragma unroll
        for (int k = 0; k < rbw / 2; ++k) {
          const uint2 x = __ldg(reinterpret_cast<const uint2*>(vr) + k);
          vw[2 * k] = x.x;
          vw[2 * k + 1] = x.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < rbw; ++k) vw[k] = __ldg(vr + k);
      }
      const uint32_t* kr = reinterpret_cast<const uint32_t*>(a.k_pages) + row * rbw;
      recipe_group_score<E, G, MB0, kPairs>(kr, qs[0], ps[0], cent[0], psum[0], kappa, sc);
      recipe_group_score<E, G, MB1, kPairs>(kr + kWh, qs[1], ps[1], cent[1], psum[1], kappa, sc);
#pragma unroll
      for (int k = 0; k < rbw; ++k) vbuf[warp][lane][k] = vw[k];
    }
    trow[warp][lane] = row;
    // ---- the tile's softmax step (m, l, the correction: the same on every lane) -----
    float corr[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float tmax = warp_max(sc[g]);
      const float mn = fmaxf(m[g], tmax);
      corr[g] = 1.f;
      float p = 0.f;
      if (mn != -INFINITY) {  // some token of this or an earlier tile
        corr[g] = exp2f(m[g] - mn);  // 0 while m is -inf
        p = exp2f(sc[g] - mn);       // 0 for a masked token
      }
      l[g] = fmaf(l[g], corr[g], warp_sum(p));
      m[g] = mn;
      pt[warp][lane][g] = p;
    }
    __syncwarp();
    // ---- values: lanes over coordinates, the tile's tokens in order -----------------
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int grp = 0; grp < 2; ++grp)
#pragma unroll
        for (int i = 0; i < E; ++i) {
          acc_c[g][grp][i] *= corr[g];
          acc_z[g][grp][i] *= corr[g];
        }
    const int nt = min(32, t_hi - tb);
    for (int k = 0; k < nt; ++k) {
      if (trow[warp][k] < 0) continue;  // (the same on every lane)
      const uint32_t* vr = vbuf[warp][k];
      float pk[G];
#pragma unroll
      for (int g = 0; g < G; ++g) pk[g] = pt[warp][k][g];
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        const GroupView<E> v = read_group_s<E>(vr + (grp ? kWh : 0), grp ? MB1 : MB0, lane);
        const float vzs = v.nu * v.gamma * kappa;
        float vc[E], vz[E];  // nu c[idx] and nu gamma kappa (2z - 1)
#pragma unroll
        for (int i = 0; i < E; ++i) {
          vc[i] = v.nu * cent[grp][v.idx[i]];
          vz[i] = ((v.zw[i] >> lane) & 1u) ? vzs : -vzs;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int i = 0; i < E; ++i) {
            acc_c[g][grp][i] = fmaf(pk[g], vc[i], acc_c[g][grp][i]);
            acc_z[g][grp][i] = fmaf(pk[g], vz[i], acc_z[g][grp][i]);
          }
      }
    }
    __syncwarp();  // the next tile rewrites pt / trow
  }
  if (__any_sync(kFullMask, bad_block) && lane == 0 && a.status) atomicMax(a.status, (int32_t)kBlockOutOfRange);
  __syncthreads();  // every warp is done with its value rows: the merge buffer may be written

  // merge the warps of this CTA, then write the split partial
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_ml[warp][g][0] = m[g];
      red_ml[warp][g][1] = l[g];
    }
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int i = 0; i < E; ++i) {
        red_acc[warp][g][grp * d + lane * E + i] = acc_c[g][grp][i];
        red_acc[warp][g][D + grp * d + lane + 32 * i] = acc_z[g][grp][i];
      }
  }
  __syncthreads();
  for (int g = warp; g < G; g += kRecDecodeWarps) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kRecDecodeWarps; ++w) mx = fmaxf(mx, red_ml[w][g][0]);
    float wt[kRecDecodeWarps], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kRecDecodeWarps; ++w) {
      wt[w] = red_ml[w][g][0] == -INFINITY ? 0.f : exp2f(red_ml[w][g][0] - mx);
      lsum = fmaf(wt[w], red_ml[w][g][1], lsum);
    }
    const int64_t slot = ((int64_t)b * a.num_q_heads + (int64_t)h * G + g) * num_splits + split;
    for (int k = lane; k < 2 * D; k += 32) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kRecDecodeWarps; ++w) sum = fmaf(wt[w], red_acc[w][g][k], sum);
      part.acc[slot * 2 * D + k] = sum;
    }
    if (lane == 0) {
      part.ml[slot * 2 + 0] = mx;
      part.ml[slot * 2 + 1] = lsum;
    }
  }
}

template <int E>
__global__ void __launch_bounds__(256)
combine_recipe_kernel(DecodeArgs a, RecipeArgs rc, int num_splits, RecipeSplitView part) {
  constexpr int d = 32 * E, D = 2 * d;
  __shared__ float zs[8][d];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= (int64_t)a.batch * a.num_q_heads) return;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int h = (int)(row % a.num_q_heads) / G;
  const float* ml = part.ml + row * num_splits * 2;
  const float* acc = part.acc + row * num_splits * 2 * D;
  float mx = -INFINITY;
  for (int s = 0; s < num_splits; ++s) mx = fmaxf(mx, ml[2 * s]);
  float vc[2][E], vz[2][E], lsum = 0.f;
#pragma unroll
  for (int grp = 0; grp < 2; ++grp)
#pragma unroll
    for (int i = 0; i < E; ++i) vc[grp][i] = vz[grp][i] = 0.f;
  for (int s = 0; s < num_splits; ++s) {
    const float ms = ml[2 * s];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
    lsum = fmaf(w, ml[2 * s + 1], lsum);
    const float* as = acc + (int64_t)s * 2 * D;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int i = 0; i < E; ++i) {
        vc[grp][i] = fmaf(w, as[grp * d + lane * E + i], vc[grp][i]);
        vz[grp][i] = fmaf(w, as[D + grp * d + lane + 32 * i], vz[grp][i]);
      }
  }
  const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
  const float rs = 1.0f / sqrtf((float)d);
#pragma unroll
  for (int grp = 0; grp < 2; ++grp) {
#pragma unroll
    for (int i = 0; i < E; ++i) zs[warp][lane + 32 * i] = vz[grp][i];
    __syncwarp();
    float w[E];  // acc_c + S^T acc_z at coordinates lane E + i
#pragma unroll
    for (int i = 0; i < E; ++i) w[i] = vc[grp][i];
    for (int k = 0; k < d; ++k) {
      const float z = zs[warp][k];
#pragma unroll
      for (int i = 0; i < E; ++i) w[i] = fmaf(__ldg(rc.smat + (int64_t)k * d + lane * E + i), z, w[i]);
    }
    __syncwarp();  // zs is rewritten for the next group
#pragma unroll
    for (int i = 0; i < E; ++i) w[i] *= inv;
    fwht_warp<E>(w);  // R_d^T w = diag(s) H w / sqrt(d)
    const int32_t* ord = rc.order + (int64_t)h * D + grp * d + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i)
      store_from_f32(a.out, row * D + __ldg(ord + i), a.out_dtype, w[i] * __ldg(a.signs + lane * E + i) * rs);
  }
}

template <typename T, int E, int MB0, int MB1>
cudaError_t launch_write_recipe_mb(const WriteArgs& a, const RecipeArgs& rc, cudaStream_t stream, int num_sms) {
  constexpr int d = 32 * E;
  const int64_t units = 2 * a.num_tokens * a.num_kv_heads;
  const int64_t per_cta = (int64_t)kRecWarps * kRecUnits;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((units + per_cta - 1) / per_cta, (int64_t)num_sms * 3));
  const size_t smem = (size_t)recipe_write_smem(d);
  auto kern = write_recipe_kernel<T, E, MB0, MB1>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kRecWarps * 32, smem, stream>>>(static_cast<const T*>(a.raw), a.num_tokens * a.num_kv_heads,
                                               a.num_kv_heads, a.slots, a.pages, rc, a.signs, a.status);
  err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

template <typename T, int E>
cudaError_t launch_write_recipe_typed(const WriteArgs& a, const RecipeArgs& rc, cudaStream_t stream, int num_sms) {
  if (rc.bits_hi == 3 && rc.bits_lo == 2) return launch_write_recipe_mb<T, E, 2, 1>(a, rc, stream, num_sms);  // turboquant25
  if (rc.bits_hi == 4 && rc.bits_lo == 3) return launch_write_recipe_mb<T, E, 3, 2>(a, rc, stream, num_sms);  // turboquant35
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_write_recipe_dim(const WriteArgs& a, const RecipeArgs& rc, cudaStream_t stream, int num_sms) {
  if (a.head_dim == 64) return launch_write_recipe_typed<T, 1>(a, rc, stream, num_sms);
  if (a.head_dim == 128) return launch_write_recipe_typed<T, 2>(a, rc, stream, num_sms);
  return cudaErrorInvalidValue;
}

template <int E, int MB0, int MB1>
cudaError_t launch_recipe_split_g(int G, dim3 grid, cudaStream_t stream, const DecodeArgs& a, const RecipeArgs& rc,
                                  const float* p_all, const DecodePlan& p, RecipeSplitView part) {
  switch (G) {
    case 1: decode_recipe_split_kernel<E, 1, MB0, MB1><<<grid, kRecDecodeWarps * 32, 0, stream>>>(a, rc, p_all, p.num_splits, p.blocks_per_split, part); break;
    case 2: decode_recipe_split_kernel<E, 2, MB0, MB1><<<grid, kRecDecodeWarps * 32, 0, stream>>>(a, rc, p_all, p.num_splits, p.blocks_per_split, part); break;
    case 4: decode_recipe_split_kernel<E, 4, MB0, MB1><<<grid, kRecDecodeWarps * 32, 0, stream>>>(a, rc, p_all, p.num_splits, p.blocks_per_split, part); break;
    case 8: decode_recipe_split_kernel<E, 8, MB0, MB1><<<grid, kRecDecodeWarps * 32, 0, stream>>>(a, rc, p_all, p.num_splits, p.blocks_per_split, part); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int E>
cudaError_t launch_decode_recipe_e(const DecodeArgs& a, const RecipeArgs& rc, const DecodePlan& p,
                                   cudaStream_t stream) {
  constexpr int D = 64 * E;
  const int64_t qrows = (int64_t)a.batch * a.num_q_heads;
  RecipeSplitView part;
  part.acc = static_cast<float*>(a.workspace);
  part.ml = part.acc + (size_t)qrows * p.num_splits * 2 * D;
  float* p_all = part.ml + (size_t)qrows * p.num_splits * 2;
  const unsigned rgrid = (unsigned)((qrows + 7) / 8);
  recipe_project_kernel<E><<<rgrid, 256, 0, stream>>>(a, rc, p_all);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  count_launches(1);
  const int G = a.num_q_heads / a.num_kv_heads;
  dim3 grid(p.num_splits, a.num_kv_heads, a.batch);
  const int mb0 = rc.bits_hi - 1, mb1 = rc.bits_lo - 1;
  if (mb0 == 2 && mb1 == 1) {  // turboquant25
    err = launch_recipe_split_g<E, 2, 1>(G, grid, stream, a, rc, p_all, p, part);
  } else if (mb0 == 3 && mb1 == 2) {  // turboquant35
    err = launch_recipe_split_g<E, 3, 2>(G, grid, stream, a, rc, p_all, p, part);
  } else {
    return cudaErrorInvalidValue;
  }
  if (err != cudaSuccess) return err;
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  count_launches(1);
  combine_recipe_kernel<E><<<rgrid, 256, 0, stream>>>(a, rc, p.num_splits, part);
  err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

}  // namespace

bool recipe_supported(int head_dim) { return head_dim == 64 || head_dim == 128; }

int recipe_row_bytes(int head_dim, int bits_hi, int bits_lo) {
  const int d = head_dim / 2;
  return 4 * (group_words(d, bits_hi) + group_words(d, bits_lo));
}

size_t recipe_decode_workspace(const DecodeArgs& a, const DecodePlan& p) {
  const size_t qrows = (size_t)std::max(0, a.batch) * a.num_q_heads;
  return qrows * p.num_splits * (2 * a.head_dim + 2) * sizeof(float) + qrows * a.head_dim * sizeof(float) + 16;
}

cudaError_t launch_write_recipe(const WriteArgs& a, const RecipeArgs& rc, cudaStream_t stream, int num_sms) {
  cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  if (a.num_tokens == 0) return cudaSuccess;
  err = launch_validate_slots(a, stream, num_sms);
  if (err != cudaSuccess) return err;
  switch (a.dtype) {
    case kF32: return launch_write_recipe_dim<float>(a, rc, stream, num_sms);
    case kF16: return launch_write_recipe_dim<__half>(a, rc, stream, num_sms);
    case kBF16: return launch_write_recipe_dim<__nv_bfloat16>(a, rc, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_recipe(const DecodeArgs& a, const RecipeArgs& rc, const DecodePlan& p, cudaStream_t stream) {
  if (a.status) {
    cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
  }
  if (a.batch == 0) return cudaSuccess;
  if (a.head_dim == 64) return launch_decode_recipe_e<1>(a, rc, p, stream);
  if (a.head_dim == 128) return launch_decode_recipe_e<2>(a, rc, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace tq
