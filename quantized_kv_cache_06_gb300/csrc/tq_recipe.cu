// Recipe cache modes turboquant25 / turboquant35: grouped product-quantised rows, writer
// and paged decode (sm_103a: m16n8k16 MMAs for the sketch, the scores and the values).
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
//   write_recipe_kernel        32 staged rows of one kv head per warp, a lane per (row, group)
//                              unit: channel gather, norm, rotation (FWHT in registers),
//                              indices and residual; then the sketch of sixteen units at a
//                              time as m16n8k16 MMAs (fp16 hi / lo splits of r and S_d) and
//                              the sign words from per-lane partial words.
//   recipe_project_kernel      one warp per (sequence, q head): per group the rotated
//                              gathered query q_g = R_d q[order_g] (times the softmax scale
//                              and log2 e) and its projection p_g = S_d q_g.
//   decode_recipe_tc_kernel    the split decode: 16-token tiles staged by cp.async, scores
//                              and values as m16n8k16 MMAs (pair tables of centroids, +-1
//                              sign operands).  Score of key row k:
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

constexpr int kRecWarps = 4;
constexpr float kRecLog2e = 1.4426950408889634f;
constexpr float kRecSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi / 2)

// 32-bit words of group g's part of a row: d (b - 1) / 32 index words, d / 32 sign words,
// nu, gamma.
__host__ __device__ constexpr int group_words(int d, int bits) { return d * (bits - 1) / 32 + d / 32 + 2; }

// Rows (token, kv head) are taken 32 at a time per warp, all of one kv head.  The warp stages
// the 32 raw rows in shared memory (4-byte cp.async copies; rows an odd number of words apart,
// so that a lane per row reads any column without bank conflicts), then encodes group 0 and
// group 1 in turn with a lane per row: the gather of the group's d channels through the
// channel order (the head's order bytes broadcast from shared memory), the sign flip as a
// sign-bit XOR, the d-point FWHT in registers (the stage order of the warp transform), the
// norm, the indices (a count of the decision points below the coordinate, held in registers),
// their packing, and the residual r, stored as fp16 hi = r 2^10 and lo = (r 2^10 - hi) 2^12.
// The residuals go to the warp's A tile sixteen at a time, and the sketch S_d r of the sixteen
// runs as m16n8k16 MMAs: r_hi S_hi into one accumulator, r_lo S_hi + r_hi S_lo into another
// (~22 significant bits, as in an fp32 sum); each lane sets the sign bits of its own
// accumulators into partial words, ORed across the four lanes of a unit pair.  The tile's
// finished rows are staged in the A tile and written with lanes over consecutive words.
constexpr int kRecRows = 32;   // rows per warp tile
constexpr int kRecUnits = 16;  // units per sketch pass

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

// Shared memory of the writer: S hi and lo, then per warp its A tile hi and lo (rows of d + 8
// halves: 16 bytes of padding put the 8 rows of an ldmatrix in different banks), then per warp
// its staged raw rows (stride raw_words + 1 words) and its head's D order bytes.
__host__ __device__ constexpr int recipe_write_smem(int d, int raw_words) {
  return (2 * d + kRecWarps * 2 * kRecUnits) * (d + 8) * 2 + kRecWarps * (kRecRows * (raw_words + 1) * 4 + 2 * d);
}

// idx = #{k : b_k < y} over the 2^MB - 1 decision points held in registers (ties and NaN: the
// lower index)
template <int MB>
__device__ __forceinline__ int rec_index(float y, const float (&b)[7]) {
  int idx = 0;
#pragma unroll
  for (int k = 0; k < (1 << MB) - 1; ++k) idx += y > b[k] ? 1 : 0;
  return idx;
}

__device__ __forceinline__ void rec_cp4w(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
template <typename T>
__device__ __forceinline__ float rec_raw_at(const uint32_t* row, int ch) {
  return to_f32<T>(reinterpret_cast<const T*>(row)[ch]);
}

// MB0 / MB1: MSE index bits of the high / low group.
template <typename T, int E, int MB0, int MB1>
__global__ void __launch_bounds__(kRecWarps * 32, 3)
write_recipe_kernel(const T* __restrict__ raw, int64_t num_tokens, int num_kv_heads, const int64_t* __restrict__ slots,
                    uint8_t* __restrict__ pages, RecipeArgs rc, const float* __restrict__ signs,
                    const int32_t* __restrict__ status) {
  constexpr int d = 32 * E, D = 2 * d;
  constexpr int kRow = d + 8;
  constexpr int kRawWords = D * (int)sizeof(T) / 4;  // words of one raw row
  constexpr int kRS = kRawWords + 1;
  constexpr int kWh = group_words(d, MB0 + 1);
  constexpr int kRowWords = kWh + group_words(d, MB1 + 1);
  extern __shared__ __align__(16) unsigned char rec_smem[];
  __half* s_hi = reinterpret_cast<__half*>(rec_smem);  // S[i][j] (i: projection, j: coordinate)
  __half* s_lo = s_hi + d * kRow;                       // (S - hi) 2^12
  __shared__ float cen[2][8];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  // the signs of R_d as bits (bit j of word w: coordinate 32 w + j negative)
  uint32_t sgm[E];
#pragma unroll
  for (int w = 0; w < E; ++w) sgm[w] = __ballot_sync(kFullMask, __ldg(signs + 32 * w + lane) < 0.f);
  __syncthreads();
  if (*status != kOk) return;  // a slot failed validation: write nothing

  const float inv_sqrt_d = 1.0f / sqrtf((float)d);
  __half* a_hi = s_lo + d * kRow + warp * (2 * kRecUnits * kRow);  // this warp's A tile: unit k, coordinate j
  __half* a_lo = a_hi + kRecUnits * kRow;
  uint32_t* raw_s = reinterpret_cast<uint32_t*>(rec_smem + (size_t)(2 * d + kRecWarps * 2 * kRecUnits) * kRow * 2) +
                    warp * (kRecRows * kRS + D / 4);
  uint32_t* ord_s = raw_s + kRecRows * kRS;  // the tile's head: its D channel-order bytes
  // ldmatrix lane addresses: A rows (units) lane & 15, k half lane >> 4; B rows (projections)
  // (lane & 7) + 8 (lane >> 4), k half (lane >> 3) & 1
  const uint32_t a_lane = smem_u32(a_hi) + (uint32_t)(((lane & 15) * kRow + (lane >> 4) * 8) * 2);
  const uint32_t a_lo_off = (uint32_t)(kRecUnits * kRow * 2);
  const uint32_t b_lane = smem_u32(s_hi) + (uint32_t)((((lane & 7) + 8 * (lane >> 4)) * kRow + ((lane >> 3) & 1) * 8) * 2);
  const uint32_t b_lo_off = (uint32_t)(d * kRow * 2);

  // finished rows of a tile, staged in the A tile (free once the second group's sketch is done)
  constexpr int kOutStride = kRowWords | 1;
  static_assert(kRecRows * kOutStride * 4 <= 2 * kRecUnits * kRow * 2, "the tile's rows fit in the A tile");
  uint32_t* out_s = reinterpret_cast<uint32_t*>(a_hi);

  const int64_t ntb = (num_tokens + kRecRows - 1) / kRecRows;
  const int64_t tiles = ntb * num_kv_heads;
  const int64_t tstride = (int64_t)gridDim.x * kRecWarps;
  // Stages tile tl (its head's order bytes, its raw rows) and commits the copies as one group.
  auto stage = [&](int64_t tl) {
    const int64_t tb = tl / num_kv_heads;
    const int h = (int)(tl - tb * num_kv_heads);
    const int64_t t0 = tb * kRecRows;
    const int nrows = (int)min((int64_t)kRecRows, num_tokens - t0);
    for (int i = lane; i < D; i += 32) reinterpret_cast<uint8_t*>(ord_s)[i] = (uint8_t)__ldg(rc.order + (int64_t)h * D + i);
    const uint32_t dst0 = smem_u32(raw_s);
    for (int r = 0; r < nrows; ++r) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(raw + ((t0 + r) * num_kv_heads + h) * D);
#pragma unroll
      for (int w = lane; w < kRawWords; w += 32) rec_cp4w(dst0 + (uint32_t)(r * kRS + w) * 4u, src + w);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  // The sketch of the sixteen units of pass p held in the A tile: sign word e of unit 16 p + u
  // is kept by lane 16 p + u.
  auto sketch = [&](int p, uint32_t (&sw)[E]) {
    const int u = lane & 15;
    const uint32_t cbit = 1u << (2 * (lane & 3));  // this lane's column pair in a byte
#pragma unroll
    for (int e = 0; e < E; ++e) {
      uint32_t pw[2] = {0u, 0u};  // partial sign words of units lane / 4 and lane / 4 + 8
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
        // projection 32 e + 8 (2 np + n) + 2 c + (x & 1)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x)
            if (fmaf(al[n][x], 1.0f / 4096, am[n][x]) >= 0.f) pw[x >> 1] |= cbit << (8 * (2 * np + n) + (x & 1));
      }
      // the four lanes of a unit pair hold disjoint bits: OR them, then unit u's word from
      // lane 4 (u mod 8)
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        pw[0] |= __shfl_xor_sync(kFullMask, pw[0], m);
        pw[1] |= __shfl_xor_sync(kFullMask, pw[1], m);
      }
      const uint32_t wa = __shfl_sync(kFullMask, pw[0], 4 * (u & 7));
      const uint32_t wb = __shfl_sync(kFullMask, pw[1], 4 * (u & 7));
      if ((lane >> 4) == p) sw[e] = (u >> 3) ? wb : wa;
    }
  };

  int64_t tl = (int64_t)blockIdx.x * kRecWarps + warp;
  if (tl < tiles) stage(tl);
  for (; tl < tiles; tl += tstride) {
    const int64_t tb = tl / num_kv_heads;
    const int h = (int)(tl - tb * num_kv_heads);
    const int64_t t0 = tb * kRecRows;
    const bool valid = t0 + lane < num_tokens;
    const int64_t slot = valid ? __ldg(slots + t0 + lane) : -1;
    const bool live = slot >= 0;  // "Slot Mapping": negative slots are ignored
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    __syncwarp();
    const uint32_t* rrow = raw_s + lane * kRS;
    uint32_t gw0[E * MB0 + E + 2];  // the first group's words, held until the row is written
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int mb = g ? MB1 : MB0;
      float y[d];
      // gather of the group's channels (this lane's row), sign flip, norm (eight partial sums
      // of squares, added as a tree)
      float ssp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j4 = 0; j4 < d / 4; ++j4) {
        const uint32_t o4 = ord_s[g * (d / 4) + j4];  // (the same word on every lane)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = 4 * j4 + q;
          const float x = live ? rec_raw_at<T>(rrow, (int)__byte_perm(o4, 0u, 0x4440u + q)) : 0.f;
          ssp[j & 7] = fmaf(x, x, ssp[j & 7]);
          y[j] = __uint_as_float(__float_as_uint(x) ^ ((sgm[j >> 5] << (31 - (j & 31))) & 0x80000000u));
        }
      }
      if (g == 1) {  // the raw tile is consumed: stage the next tile behind this group's encode
        __syncwarp();
        if (tl + tstride < tiles) stage(tl + tstride);
      }
      // y = H (s * x) / (sqrt(d) nu): the d-point FWHT in registers
#pragma unroll
      for (int hs = 1; hs < d; hs <<= 1)
#pragma unroll
        for (int i = 0; i < d; ++i)
          if ((i & hs) == 0) {
            const float p0 = y[i], p1 = y[i + hs];
            y[i] = p0 + p1;
            y[i + hs] = p0 - p1;
          }
      const float nu = sqrtf(((ssp[0] + ssp[1]) + (ssp[2] + ssp[3])) + ((ssp[4] + ssp[5]) + (ssp[6] + ssp[7])));
      const float inv = nu > 0.f ? inv_sqrt_d / nu : 0.f;
      // indices (packed LSB first), residual (fp16 hi / lo pairs), gamma^2
      constexpr int kIW = E * (MB0 > MB1 ? MB0 : MB1);
      uint32_t iw[kIW];
#pragma unroll
      for (int w = 0; w < kIW; ++w) iw[w] = 0u;
      uint32_t rh[d / 2], rl[d / 2];
      float rsp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < d; j += 2) {  // a pair of coordinates: one packed fp16 conversion each
        float x2[2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int jj = j + e2;
          const float yv = y[jj] * inv;
          const int idx = g ? rec_index<MB1>(yv, blo) : rec_index<MB0>(yv, bhi);
          const int bit = jj * mb, w = bit >> 5, o = bit & 31;
          iw[w] |= (uint32_t)idx << o;
          if (o + mb > 32) iw[w + 1] |= (uint32_t)idx >> (32 - o);
          const float dr = yv - cen[g][idx];
          rsp[jj & 3] = fmaf(dr, dr, rsp[jj & 3]);
          x2[e2] = dr * 1024.0f;
        }
        // (rows of dead lanes gathered zeros: their residual is finite and never written)
        const __half2 h2 = __floats2half2_rn(x2[0], x2[1]);
        const float2 hf = __half22float2(h2);
        const __half2 l2 = __floats2half2_rn((x2[0] - hf.x) * 4096.0f, (x2[1] - hf.y) * 4096.0f);
        rh[j >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
        rl[j >> 1] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      // the sketch, sixteen units per pass
      uint32_t sw[E];
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        if ((lane >> 4) == pass) {
          uint4* dh = reinterpret_cast<uint4*>(a_hi + (lane & 15) * kRow);
          uint4* dl = reinterpret_cast<uint4*>(a_lo + (lane & 15) * kRow);
#pragma unroll
          for (int k = 0; k < d / 8; ++k) {
            dh[k] = make_uint4(rh[4 * k], rh[4 * k + 1], rh[4 * k + 2], rh[4 * k + 3]);
            dl[k] = make_uint4(rl[4 * k], rl[4 * k + 1], rl[4 * k + 2], rl[4 * k + 3]);
          }
        }
        __syncwarp();
        sketch(pass, sw);
        __syncwarp();  // the A tile is rewritten by the next pass
      }
      const int iwn = E * mb;
      if (g == 0) {
#pragma unroll
        for (int w = 0; w < E * MB0; ++w) gw0[w] = iw[w];
#pragma unroll
        for (int e = 0; e < E; ++e) gw0[E * MB0 + e] = sw[e];
        gw0[E * MB0 + E] = __float_as_uint(nu);
        gw0[E * MB0 + E + 1] = __float_as_uint(sqrtf((rsp[0] + rsp[1]) + (rsp[2] + rsp[3])));
      } else {
        // this lane's row into the staging rows, then the tile's rows written with lanes over
        // consecutive words
        uint32_t* orow = out_s + lane * kOutStride;
#pragma unroll
        for (int w = 0; w < kWh; ++w) orow[w] = gw0[w];
#pragma unroll
        for (int w = 0; w < E * MB1; ++w) orow[kWh + w] = iw[w];
#pragma unroll
        for (int e = 0; e < E; ++e) orow[kWh + iwn + e] = sw[e];
        orow[kWh + iwn + E] = __float_as_uint(nu);
        orow[kWh + iwn + E + 1] = __float_as_uint(sqrtf((rsp[0] + rsp[1]) + (rsp[2] + rsp[3])));
        __syncwarp();
#pragma unroll 2
        for (int q = lane; q < kRecRows * kRowWords; q += 32) {
          const int r = q / kRowWords, w = q - r * kRowWords;
          const int64_t sr = __shfl_sync(kFullMask, slot, r);
          if (sr >= 0) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(pages + (sr * num_kv_heads + h) * (int64_t)(kRowWords * 4));
            dst[w] = out_s[r * kOutStride + w];
          }
        }
        __syncwarp();  // the A tile is the next tile's again
      }
    }
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
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

// Merges the NW warps' partials of one CTA (running max in log2 units and sum per q head;
// value accumulators as in RecipeSplitView) and writes the CTA's split partial for q rows
// row0 + g.  Called after a barrier that makes every warp's partial visible.
template <int NW, int G, int D>
__device__ __forceinline__ void recipe_merge_write(const float (*red_ml)[G][2], const float (*red_acc)[G][2 * D],
                                                   int64_t row0, int num_splits, int split, RecipeSplitView part,
                                                   int warp, int lane) {
  for (int g = warp; g < G; g += NW) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, red_ml[w][g][0]);
    float wt[NW], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      wt[w] = red_ml[w][g][0] == -INFINITY ? 0.f : exp2f(red_ml[w][g][0] - mx);
      lsum = fmaf(wt[w], red_ml[w][g][1], lsum);
    }
    const int64_t slot = (row0 + g) * num_splits + split;
    for (int k = lane; k < 2 * D; k += 32) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) sum = fmaf(wt[w], red_acc[w][g][k], sum);
      part.acc[slot * 2 * D + k] = sum;
    }
    if (lane == 0) {
      part.ml[slot * 2 + 0] = mx;
      part.ml[slot * 2 + 1] = lsum;
    }
  }
}

// ---- tensor-core split decode ------------------------------------------------------------
// Each warp takes 16-token tiles of its split in turn.  The tile's K and V rows are staged in
// shared memory by cp.async, three tiles per warp (the next two tiles' copies in flight while
// this one is computed, their block ids loaded an iteration earlier; four lanes copy a row;
// rows of tokens past the sequence end or in a block with a bad id are zero-filled).  Every
// contraction is an m16n8k16 MMA with fp32 accumulation whose n = 8 columns hold q heads 0-3
// twice: columns 0-3 take the fp16 hi part of the B operand, columns 4-7 its remainder, so one
// MMA gives both products and every product keeps ~22 significant bits.
//
// Scores of a group: A = the K tile (tokens x coordinates); the lane of column c takes the
// coordinates [8E c, 8E c + 8E) in pairs, each A register one entry of a pair table (the
// centroids of two adjacent coordinates: fp16 hi in .x, remainder in .y; sixteen copies, so a
// 64-bit lookup by a half warp never conflicts) addressed by the pair's 2 MB-bit field;
// B = the rotated query.  The sign term takes A = +-1 built from two sign bits 16 apart (one
// shift, one LOP3 per register) against B = p = S_d q.  score = sum_g nu_g (m_g + gamma_g
// kappa s_g).
//
// Values of a group: A = the V tile transposed (coordinates x tokens); the lane of row gr
// takes the coordinates [4E gr, 4E gr + 4E) of four tokens, two table entries merged by PRMT
// per register, and the sign term from bytes of two tokens' sign words.  B = the weights
// p nu 2^(12 - e) (values) and p nu gamma kappa 2^(12 - e) (signs), where 2^e bounds every
// value norm the warp has seen (when e grows the accumulators are scaled by the same power of
// two, exactly, with the softmax correction) and p <= 2^3 (the running max lags a score by
// at most three log2 units), so no weight leaves fp16 range.
constexpr int kRecTcWarps = 4;
constexpr int kRecTcStages = 3;  // tiles staged per warp: the current one and two in flight
constexpr float kRecSlack = 3.0f;  // log2 units the running max may lag behind a score

__device__ __forceinline__ void rec_cp8(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void rec_cp4(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void rec_cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void rec_cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// (x0, x1) as an fp16 pair (x0 in the low half): the rounded values, or with `rem` the
// remainders x - fp16(x)
__device__ __forceinline__ uint32_t rec_split_pack(float x0, float x1, bool rem) {
  const __half2 hi = __floats2half2_rn(x0, x1);
  const __half2 lo = __floats2half2_rn(x0 - __low2float(hi), x1 - __high2float(hi));
  const __half2 r = rem ? lo : hi;
  return *reinterpret_cast<const uint32_t*>(&r);
}
// fp16 pair of +-1 from bits 15 and 31 of x (bit set: +1)
__device__ __forceinline__ uint32_t rec_sign2(uint32_t x) { return (~x & 0x80008000u) | 0x3C003C00u; }
// Byte offset, within a pair table, of the entry whose fbits-bit field sits at bit sh of x,
// in the copy of this lane (lane8 = 8 (lane mod 16); entries are 128 bytes apart).
__device__ __forceinline__ uint32_t rec_tab_off(uint32_t x, int sh, int fbits, uint32_t lane8) {
  const uint32_t y = sh >= 7 ? (x >> (sh - 7)) : (x << (7 - sh));
  return (y & (((1u << fbits) - 1u) << 7)) | lane8;
}
// Pair-table entry f of a codebook of 2^mb centroids: (c[f mod 2^mb], c[f / 2^mb]).
__device__ __forceinline__ uint2 rec_pair_entry(const float* __restrict__ cent, int f, int mb) {
  const float c0 = __ldg(cent + (f & ((1 << mb) - 1))), c1 = __ldg(cent + (f >> mb));
  uint2 e;
  e.x = rec_split_pack(c0, c1, false);
  e.y = rec_split_pack(c0, c1, true);
  return e;
}

// CTAs per SM: four for turboquant25 (128 registers, a few bytes of spills, measured faster
// than three), three for turboquant35 (its three staged tiles per warp take 43 KB of shared
// memory, and four CTAs at 128 registers measured slower).
template <int E, int G, int MB0, int MB1>
__global__ void __launch_bounds__(kRecTcWarps * 32, (MB0 == 2 && G <= 4) ? 4 : 3)
decode_recipe_tc_kernel(DecodeArgs a, RecipeArgs rc, const float* __restrict__ p_all, int num_splits,
                        int blocks_per_split, RecipeSplitView part) {
  // G <= 4: the eight MMA columns hold four q heads' hi parts (columns 0-3) and remainders
  // (4-7) of one B operand.  G = 8: they hold the eight heads, and the hi parts and the
  // remainders are two B operands, each with its own MMA into the same accumulators.
  static_assert(G <= 4 || G == 8, "up to four q heads, or eight");
  constexpr bool kG8 = G == 8;
  constexpr int GC = kG8 ? 8 : 4;      // q heads held (the ones past G are zero)
  constexpr int kSets = kG8 ? 2 : 1;   // B operands per product
  constexpr int d = 32 * E, D = 2 * d;
  constexpr int kWh = E * MB0 + E + 2;        // words of the high group
  constexpr int rbw = kWh + E * MB1 + E + 2;  // words of a row
  constexpr bool kPairs = rbw % 2 == 0;       // rows, groups and (nu, gamma) 8-byte aligned
  static_assert(!kPairs || (kWh % 2 == 0 && (E * MB0 + E) % 2 == 0 && (E * MB1 + E) % 2 == 0), "alignment");
  constexpr int kBuf = 32 * rbw;  // one staged tile: the 16 K rows, then the 16 V rows
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, c = lane & 3;
  const int H = a.num_kv_heads, bs = a.block_size;

  __shared__ __align__(16) uint2 tab0[1 << (2 * MB0)][16];
  __shared__ __align__(16) uint2 tab1[1 << (2 * MB1)][16];
  __shared__ __align__(16) float qv[2][2][GC][d];          // [q | p][group][q head][coordinate]
  __shared__ __align__(16) float pt[kRecTcWarps][GC][16];  // the tile's weights [q head][token]
  __shared__ float red_ml[kRecTcWarps][G][2];
  // the warps' staged tiles, then (after the last tile) the merge buffer: dynamic shared
  // memory of recipe_tc_dyn_words words
  extern __shared__ __align__(16) uint32_t stage_u[];
  float(*red_acc)[G][2 * D] = reinterpret_cast<float(*)[G][2 * D]>(stage_u);

  for (int i = threadIdx.x; i < (1 << (2 * MB0)) * 16; i += blockDim.x) tab0[i >> 4][i & 15] = rec_pair_entry(rc.mse_hi, i >> 4, MB0);
  for (int i = threadIdx.x; i < (1 << (2 * MB1)) * 16; i += blockDim.x) tab1[i >> 4][i & 15] = rec_pair_entry(rc.mse_lo, i >> 4, MB1);
  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kRecLog2e / sqrtf((float)d);
  const float kappa = kRecSqrtHalfPi / (float)d;
  for (int g = warp; g < GC; g += kRecTcWarps) {  // heads past G: zero query, never written
    const int64_t qrow = (int64_t)b * a.num_q_heads + (int64_t)h * G + g;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      float qr[E];
      const int32_t* ord = rc.order + (int64_t)h * D + grp * d + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        qr[i] = g < G ? load_as_f32(a.q, qrow * D + __ldg(ord + i), a.q_dtype) * __ldg(a.signs + lane * E + i) : 0.f;
      fwht_warp<E>(qr);
#pragma unroll
      for (int i = 0; i < E; ++i) {
        qv[0][grp][g][lane * E + i] = qr[i] * qmul;
        qv[1][grp][g][lane + 32 * i] = g < G ? __ldg(p_all + (qrow * 2 + grp) * d + lane + 32 * i) : 0.f;
      }
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
  __syncthreads();

  // B operands of the scores: column n = gr is q head gr mod 4, its fp16 hi part for gr < 4
  // and its remainder for gr >= 4 (G <= 4), or q head gr, hi parts in set 0 and remainders in
  // set 1 (G = 8).  Pair kp = 2 s + slot of k-step s: coordinates 8E c + 2 kp (+1) for the
  // centroid term; for the sign term the pair P = 4E c + kp, coordinates 32 (P / 16) + P mod 16
  // and 16 above.
  const bool rem_col = !kG8 && gr >= 4;
  const int hq = kG8 ? gr : (gr & 3);
  // The fragments are the same for every warp of the CTA: warp 0 stores them once in shared
  // memory, over the query they were built from, and each k-step loads its pair (64 bits).
  uint2 bqr[kSets][2][2 * E], bpr[kSets][2][2 * E];
#pragma unroll
  for (int st = 0; st < kSets; ++st)
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int s = 0; s < 2 * E; ++s) {
        uint32_t fq[2], fp[2];
        const bool rem = kG8 ? st == 1 : rem_col;
#pragma unroll
        for (int slot = 0; slot < 2; ++slot) {
          const int kp = 2 * s + slot;
          const int j = 8 * E * c + 2 * kp;
          fq[slot] = rec_split_pack(qv[0][grp][hq][j], qv[0][grp][hq][j + 1], rem);
          const int pp = 4 * E * c + kp;
          const int js = 32 * (pp >> 4) + (pp & 15);
          fp[slot] = rec_split_pack(qv[1][grp][hq][js], qv[1][grp][hq][js + 16], rem);
        }
        bqr[st][grp][s] = make_uint2(fq[0], fq[1]);
        bpr[st][grp][s] = make_uint2(fp[0], fp[1]);
      }
  static_assert(kSets * 2 * 2 * 2 * E * 32 * 8 <= (int)sizeof(qv), "the fragments fit over the query");
  // [set][q | p][group][s][lane]
  uint2(*bfr)[2][2][2 * E][32] = reinterpret_cast<uint2(*)[2][2][2 * E][32]>(&qv[0][0][0][0]);
  __syncthreads();  // every warp has read the query
  if (warp == 0) {
#pragma unroll
    for (int st = 0; st < kSets; ++st)
#pragma unroll
      for (int grp = 0; grp < 2; ++grp)
#pragma unroll
        for (int s = 0; s < 2 * E; ++s) {
          bfr[st][0][grp][s][lane] = bqr[st][grp][s];
          bfr[st][1][grp][s][lane] = bpr[st][grp][s];
        }
  }
  __syncthreads();
  const int sw_k = (4 * E * c) >> 4, sh_k = (4 * E * c) & 15;  // this lane's sign word, first bit
  const uint32_t lane8 = (uint32_t)(lane & 15) << 3;
  const unsigned char* tabs[2] = {reinterpret_cast<const unsigned char*>(&tab0[0][0]),
                                  reinterpret_cast<const unsigned char*>(&tab1[0][0])};

  // staging: the lane (gr, c) copies chunks c, c + 4, ... of the K and V rows of its tokens
  // gr and gr + 8 (the tokens it scores), so one copy instruction touches eight rows
  const uint32_t* stage_w = stage_u + warp * kRecTcStages * kBuf;
  const uint32_t stage_base = smem_u32(stage_w);
  const bool bs_pow2 = (bs & (bs - 1)) == 0;
  const int bs_shift = __ffs(bs) - 1;
  bool bad_block = false;
  // Block id of this lane's token gr + 8 r of the tile at t0 (loaded an iteration before its
  // copies; -1 past the end).
  auto load_bid = [&](int t0, int r) -> int {
    const int t = t0 + gr + 8 * r;
    if (t >= t_hi) return -1;
    return __ldg(a.block_table + (int64_t)b * a.max_blocks_per_seq + (bs_pow2 ? (t >> bs_shift) : t / bs));
  };
  // Issues the copies of the tile at token t0 into buffer buf and commits them as one group;
  // returns bit r set when token gr + 8 r is valid (rows of other tokens are zero-filled).
  auto issue = [&](int t0, int bid0, int bid1, int buf) -> uint32_t {
    uint32_t okm = 0u;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = t0 + gr + 8 * r;
      const int bid = r ? bid1 : bid0;
      bool ok = false;
      int64_t row = 0;
      if (t < t_hi) {
        const int blk = bs_pow2 ? (t >> bs_shift) : t / bs;
        if (bid < 0 || (int64_t)bid >= a.num_blocks) {
          bad_block = true;
        } else {
          ok = true;
          row = ((int64_t)bid * bs + (t - blk * bs)) * H + h;
        }
      }
      okm |= ok ? (1u << r) : 0u;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const unsigned char* src = (kv ? a.v_pages : a.k_pages) + row * (int64_t)(4 * rbw);
        const uint32_t dst = stage_base + (uint32_t)((buf * 32 + kv * 16 + gr + 8 * r) * rbw) * 4u;
        if constexpr (kPairs) {
          const uint32_t nb = ok ? 8u : 0u;
#pragma unroll
          for (int k = 0; k < (rbw / 2 + 3) / 4; ++k)
            if (c + 4 * k < rbw / 2) rec_cp8(dst + 8 * (c + 4 * k), src + 8 * (c + 4 * k), nb);
        } else {
          const uint32_t nb = ok ? 4u : 0u;
#pragma unroll
          for (int k = 0; k < (rbw + 3) / 4; ++k)
            if (c + 4 * k < rbw) rec_cp4(dst + 4 * (c + 4 * k), src + 4 * (c + 4 * k), nb);
        }
      }
    }
    rec_cp_commit();
    return okm;
  };

  float ov[2][2 * E][4], oz[2][2 * E][4];  // value accumulators: rows coordinates, columns heads
#pragma unroll
  for (int grp = 0; grp < 2; ++grp)
#pragma unroll
    for (int u = 0; u < 2 * E; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i) ov[grp][u][i] = oz[grp][u][i] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // q heads 2 (c mod 2) + e
  int e_run = -115;  // every value norm seen so far is below 2^e_run

  static_assert(kRecTcStages == 3, "the flags of the tiles in flight are held in vm0, vm1");
  constexpr int kStep = 16 * kRecTcWarps;
  int t0 = t_lo + 16 * warp;
  // prologue: tiles 0 and 1 (a group is committed for each, empty past the end)
  uint32_t vm0 = 0u, vm1 = 0u;
  if (t0 < t_hi) vm0 = issue(t0, load_bid(t0, 0), load_bid(t0, 1), 0); else rec_cp_commit();
  if (t0 + kStep < t_hi) vm1 = issue(t0 + kStep, load_bid(t0 + kStep, 0), load_bid(t0 + kStep, 1), 1); else rec_cp_commit();
  int bid_n0 = load_bid(t0 + 2 * kStep, 0), bid_n1 = load_bid(t0 + 2 * kStep, 1);
  int buf = 0;
  for (; t0 < t_hi; t0 += kStep) {
    const int tn = t0 + 2 * kStep;
    const int bufn = buf == 0 ? 2 : buf - 1;  // (buf + 2) mod 3
    uint32_t vmn = 0u;
    if (tn < t_hi) vmn = issue(tn, bid_n0, bid_n1, bufn); else rec_cp_commit();
    bid_n0 = load_bid(tn + kStep, 0);  // used by the next iteration's copies
    bid_n1 = load_bid(tn + kStep, 1);
    rec_cp_wait<kRecTcStages - 1>();  // this tile's group is complete
    __syncwarp();
    const uint32_t* tile = stage_w + buf * kBuf;
    const uint32_t vm = vm0;

    // ---- scores of tokens gr + 8 r, q heads 2 (c mod 2) + e (G <= 4: this lane's column
    // part) or 2 c + e (G = 8) ----
    float sc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const int MB = grp ? MB1 : MB0, goff = grp ? kWh : 0, IW = E * MB;
      const unsigned char* tabp = tabs[grp];
      uint32_t ch[2][E], sg[2];
      float nk[2], gk[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t* kr = tile + (gr + 8 * r) * rbw + goff;
#pragma unroll
        for (int q = 0; q < E; ++q) {  // coordinates [8E c + 8 q, + 8)
          const int bit = (8 * E * c + 8 * q) * MB;
          ch[r][q] = __funnelshift_r(kr[bit >> 5], kr[(bit >> 5) + 1], bit & 31);
        }
        sg[r] = kr[IW + sw_k] >> sh_k;
        nk[r] = __uint_as_float(kr[IW + E]);
        gk[r] = __uint_as_float(kr[IW + E + 1]) * kappa;
      }
      float am[4] = {0.f, 0.f, 0.f, 0.f}, as[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 2 * E; ++s) {
        uint2 tv[2][2];
        uint32_t sv[2][2];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int slot = 0; slot < 2; ++slot) {
            const int kp = 2 * s + slot;
            tv[r][slot] = *reinterpret_cast<const uint2*>(tabp + rec_tab_off(ch[r][kp >> 2], 2 * MB * (kp & 3), 2 * MB, lane8));
            sv[r][slot] = rec_sign2(sg[r] << (15 - kp));
          }
        const uint2 bq = bfr[0][0][grp][s][lane], bp = bfr[0][1][grp][s][lane];
        rec_mma(am, tv[0][0].x, tv[1][0].x, tv[0][1].x, tv[1][1].x, bq.x, bq.y);
        rec_mma(am, tv[0][0].y, tv[1][0].y, tv[0][1].y, tv[1][1].y, bq.x, bq.y);
        rec_mma(as, sv[0][0], sv[1][0], sv[0][1], sv[1][1], bp.x, bp.y);
        if constexpr (kG8) {  // the remainders of q and p (centroid remainder x q remainder: dropped)
          const uint2 bq1 = bfr[kSets - 1][0][grp][s][lane], bp1 = bfr[kSets - 1][1][grp][s][lane];
          rec_mma(am, tv[0][0].x, tv[1][0].x, tv[0][1].x, tv[1][1].x, bq1.x, bq1.y);
          rec_mma(as, sv[0][0], sv[1][0], sv[0][1], sv[1][1], bp1.x, bp1.y);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int e = 0; e < 2; ++e) sc[r][e] = fmaf(nk[r], fmaf(gk[r], as[2 * r + e], am[2 * r + e]), sc[r][e]);
    }
    // hi + lo column parts; masked tokens
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if constexpr (!kG8) sc[r][e] += __shfl_xor_sync(kFullMask, sc[r][e], 2);
        if (!((vm >> r) & 1u)) sc[r][e] = -INFINITY;
      }

    // ---- the tile's softmax step: the running max moves only when a score passes it by
    // more than kRecSlack (so p <= 2^kRecSlack and, with the value scale, every weight stays
    // below 2^15), and the accumulators are rescaled only then ----
    float corr[2], p[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float tm = fmaxf(sc[0][e], sc[1][e]);
      tm = fmaxf(tm, __shfl_xor_sync(kFullMask, tm, 4));
      tm = fmaxf(tm, __shfl_xor_sync(kFullMask, tm, 8));
      tm = fmaxf(tm, __shfl_xor_sync(kFullMask, tm, 16));
      corr[e] = 1.f;
      if (tm > m_run[e] + kRecSlack) {  // (never for a tile without tokens: tm = -inf)
        corr[e] = exp2f(m_run[e] - tm);  // 0 while m is -inf
        m_run[e] = tm;
      }
      p[0][e] = p[1][e] = 0.f;
      if (m_run[e] != -INFINITY) {  // some token of this or an earlier tile
        p[0][e] = exp2f(sc[0][e] - m_run[e]);
        p[1][e] = exp2f(sc[1][e] - m_run[e]);
      }
      l_run[e] = fmaf(l_run[e], corr[e], p[0][e] + p[1][e]);
    }
    if (kG8 || c < 2) {
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int e = 0; e < 2; ++e) pt[warp][2 * c + e][gr + 8 * r] = p[r][e];
    }

    // ---- value norms of this lane's tokens 2c, 2c + 1, 2c + 8, 2c + 9; the weight scale ----
    float nv[4][2], gv[4][2];
    float vmax = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t* vr = tile + (16 + 2 * c + (k & 1) + 8 * (k >> 1)) * rbw;
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        const int w = (grp ? kWh + E * MB1 : E * MB0) + E;
        nv[k][grp] = __uint_as_float(vr[w]);
        gv[k][grp] = __uint_as_float(vr[w + 1]) * kappa;
      }
      vmax = fmaxf(vmax, fmaxf(nv[k][0], nv[k][1]));
    }
    vmax = fmaxf(vmax, __shfl_xor_sync(kFullMask, vmax, 1));
    vmax = fmaxf(vmax, __shfl_xor_sync(kFullMask, vmax, 2));
    if (vmax > 0.f) {
      const int ex = (int)((__float_as_uint(vmax) >> 23) & 255u) - 126;  // vmax < 2^ex
      if (ex > e_run) {
        const float f = ldexpf(1.f, e_run - ex);
        corr[0] *= f;
        corr[1] *= f;
        e_run = ex;
      }
    }
    if (__any_sync(kFullMask, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
      for (int grp = 0; grp < 2; ++grp)
#pragma unroll
        for (int u = 0; u < 2 * E; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            ov[grp][u][i] *= corr[i & 1];
            oz[grp][u][i] *= corr[i & 1];
          }
    }
    const float wscale = __uint_as_float((uint32_t)(139 - e_run) << 23);  // 2^(12 - e_run)
    __syncwarp();  // pt

    // ---- value weights (B: column n = gr, q head gr mod 4, hi for gr < 4 and remainder else;
    // or q head gr, hi in set 0 and remainder in set 1) ----
    uint32_t bc[kSets][2][2], bz[kSets][2][2];
    {
      const float2 pa = *reinterpret_cast<const float2*>(&pt[warp][hq][2 * c]);
      const float2 pb = *reinterpret_cast<const float2*>(&pt[warp][hq][2 * c + 8]);
      const float pw[4] = {pa.x * wscale, pa.y * wscale, pb.x * wscale, pb.y * wscale};
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        float wc[4], wz[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          wc[k] = pw[k] * nv[k][grp];
          wz[k] = wc[k] * gv[k][grp];
        }
#pragma unroll
        for (int st = 0; st < kSets; ++st) {
          const bool rem = kG8 ? st == 1 : rem_col;
          bc[st][grp][0] = rec_split_pack(wc[0], wc[1], rem);
          bc[st][grp][1] = rec_split_pack(wc[2], wc[3], rem);
          bz[st][grp][0] = rec_split_pack(wz[0], wz[1], rem);
          bz[st][grp][1] = rec_split_pack(wz[2], wz[3], rem);
        }
      }
    }

    // ---- values: rows = coordinates (pairs 4E gr + 2u of the centroid term, 16 u + gr of
    // the sign term; row gr + 8 the next one), columns = heads ----
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const int MB = grp ? MB1 : MB0, goff = grp ? kWh : 0, IW = E * MB;
      const unsigned char* tabp = tabs[grp];
      const int bitv = 4 * E * gr * MB;
      uint32_t chv[4], sw[4][E];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t* vr = tile + (16 + 2 * c + (k & 1) + 8 * (k >> 1)) * rbw + goff;
        chv[k] = __funnelshift_r(vr[bitv >> 5], vr[(bitv >> 5) + 1], bitv & 31);
#pragma unroll
        for (int w = 0; w < E; ++w) sw[k][w] = vr[IW + w];
      }
#pragma unroll
      for (int u = 0; u < 2 * E; ++u) {
        uint2 x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          x[k] = *reinterpret_cast<const uint2*>(tabp + rec_tab_off(chv[k], 2 * MB * u, 2 * MB, lane8));
        const uint32_t h0 = __byte_perm(x[0].x, x[1].x, 0x5410), h1 = __byte_perm(x[0].x, x[1].x, 0x7632);
        const uint32_t h2 = __byte_perm(x[2].x, x[3].x, 0x5410), h3 = __byte_perm(x[2].x, x[3].x, 0x7632);
        rec_mma(ov[grp][u], h0, h1, h2, h3, bc[0][grp][0], bc[0][grp][1]);
        rec_mma(ov[grp][u], __byte_perm(x[0].y, x[1].y, 0x5410), __byte_perm(x[0].y, x[1].y, 0x7632),
                __byte_perm(x[2].y, x[3].y, 0x5410), __byte_perm(x[2].y, x[3].y, 0x7632), bc[0][grp][0], bc[0][grp][1]);
        if constexpr (kG8) rec_mma(ov[grp][u], h0, h1, h2, h3, bc[kSets - 1][grp][0], bc[kSets - 1][grp][1]);
        // sign bits 16 (u mod 2) + gr and + 8 of word u / 2: bytes bb, bb + 1 of two tokens
        const int bb = 2 * (u & 1);
        const uint32_t sel = (uint32_t)(bb | (bb + 1) << 4 | (bb + 4) << 8 | (bb + 5) << 12);
        const uint32_t z01 = __byte_perm(sw[0][u >> 1], sw[1][u >> 1], sel);
        const uint32_t z23 = __byte_perm(sw[2][u >> 1], sw[3][u >> 1], sel);
        const uint32_t s0 = rec_sign2(z01 << (15 - gr)), s1 = rec_sign2(z01 << (7 - gr));
        const uint32_t s2 = rec_sign2(z23 << (15 - gr)), s3 = rec_sign2(z23 << (7 - gr));
        rec_mma(oz[grp][u], s0, s1, s2, s3, bz[0][grp][0], bz[0][grp][1]);
        if constexpr (kG8) rec_mma(oz[grp][u], s0, s1, s2, s3, bz[kSets - 1][grp][0], bz[kSets - 1][grp][1]);
      }
    }
    __syncwarp();  // the next tile rewrites pt; the one after it this buffer
    vm0 = vm1;
    vm1 = vmn;
    buf = buf == 2 ? 0 : buf + 1;
  }
  rec_cp_wait<0>();  // (the trailing groups are empty)
  if (__any_sync(kFullMask, bad_block) && lane == 0 && a.status) atomicMax(a.status, (int32_t)kBlockOutOfRange);
  __syncthreads();  // every warp is done with its staged rows: the merge buffer may be written

  // this warp's partial: l over the lane rows, hi + lo columns, the weight scale undone
  const float unscale = ldexpf(1.f, e_run - 12);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float l = l_run[e];
    l += __shfl_xor_sync(kFullMask, l, 4);
    l += __shfl_xor_sync(kFullMask, l, 8);
    l += __shfl_xor_sync(kFullMask, l, 16);
    const int g = 2 * c + e;
    if (gr == 0 && (kG8 || c < 2) && g < G) {
      red_ml[warp][g][0] = m_run[e];
      red_ml[warp][g][1] = l;
    }
  }
#pragma unroll
  for (int grp = 0; grp < 2; ++grp)
#pragma unroll
    for (int u = 0; u < 2 * E; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // (G <= 4: hi + remainder columns)
        const float v = kG8 ? ov[grp][u][i] : ov[grp][u][i] + __shfl_xor_sync(kFullMask, ov[grp][u][i], 2);
        const float z = kG8 ? oz[grp][u][i] : oz[grp][u][i] + __shfl_xor_sync(kFullMask, oz[grp][u][i], 2);
        const int g = 2 * c + (i & 1), r = i >> 1;
        if ((kG8 || c < 2) && g < G) {
          red_acc[warp][g][grp * d + 4 * E * gr + 2 * u + r] = v * unscale;
          red_acc[warp][g][D + grp * d + 16 * u + gr + 8 * r] = z * unscale;
        }
      }
  __syncthreads();
  recipe_merge_write<kRecTcWarps, G, D>(red_ml, red_acc, (int64_t)b * a.num_q_heads + (int64_t)h * G, num_splits,
                                        split, part, warp, lane);
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
  const int64_t tiles = (a.num_tokens + kRecRows - 1) / kRecRows * a.num_kv_heads;
  const int64_t per_cta = kRecWarps;
  const int64_t want = (tiles + per_cta - 1) / per_cta;
  const size_t smem = (size_t)recipe_write_smem(d, 2 * d * (int)sizeof(T) / 4);
  auto kern = write_recipe_kernel<T, E, MB0, MB1>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRecWarps * 32, smem);
  if (err != cudaSuccess) return err;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * std::max(1, per_sm)));
  kern<<<grid, kRecWarps * 32, smem, stream>>>(static_cast<const T*>(a.raw), a.num_tokens, a.num_kv_heads, a.slots,
                                               a.pages, rc, a.signs, a.status);
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

// Dynamic shared memory of decode_recipe_tc_kernel, in words: the larger of the warps'
// staged tiles and the merge buffer.
template <int E, int G, int MB0, int MB1>
constexpr int recipe_tc_dyn_words() {
  constexpr int rbw = (E * MB0 + E + 2) + (E * MB1 + E + 2);
  constexpr int kStageWords = kRecTcWarps * kRecTcStages * 32 * rbw, kRedWords = kRecTcWarps * G * 2 * 64 * E;
  return kStageWords > kRedWords ? kStageWords : kRedWords;
}

template <int E, int G, int MB0, int MB1>
cudaError_t launch_recipe_tc(dim3 grid, cudaStream_t stream, const DecodeArgs& a, const RecipeArgs& rc,
                             const float* p_all, const DecodePlan& p, RecipeSplitView part) {
  auto kern = decode_recipe_tc_kernel<E, G, MB0, MB1>;
  const int smem = 4 * recipe_tc_dyn_words<E, G, MB0, MB1>();
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kRecTcWarps * 32, smem, stream>>>(a, rc, p_all, p.num_splits, p.blocks_per_split, part);
  return cudaGetLastError();
}

template <int E, int MB0, int MB1>
cudaError_t launch_recipe_split_g(int G, dim3 grid, cudaStream_t stream, const DecodeArgs& a, const RecipeArgs& rc,
                                  const float* p_all, const DecodePlan& p, RecipeSplitView part) {
  switch (G) {  // the tensor-core tiles at every GQA ratio
    case 1: return launch_recipe_tc<E, 1, MB0, MB1>(grid, stream, a, rc, p_all, p, part);
    case 2: return launch_recipe_tc<E, 2, MB0, MB1>(grid, stream, a, rc, p_all, p, part);
    case 4: return launch_recipe_tc<E, 4, MB0, MB1>(grid, stream, a, rc, p_all, p, part);
    case 8: return launch_recipe_tc<E, 8, MB0, MB1>(grid, stream, a, rc, p_all, p, part);
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
