// Tensor-core packed-KV row writer (fp16 / bf16 rows at head_dim 64, 128 or 256, fp32 rows at
// 64 or 128; 2 to 5 bits).
//
// TurboQuant docs: "vLLM Usage" (TQ Byte Layout, Slot Mapping, TQ Packed Page Contract:
// write_tq4_kv) and "Architecture" (PackedPageCache).
//
// A warp encodes 16 consecutive rows (t, h) at a time.
//  * Rotation.  With d = 16 j + k, H_D = H_{D/16} (x) H_16 (Sylvester order), so
//    y = H_D (s * x) is an m16n8k16 MMA per 16-column block j against
//    B_j = diag(s_j) H_16 (entries +-1: exact in fp16 / bf16, products exact in the fp32
//    accumulator), followed by the H_{D/16} butterflies across blocks, in registers.
//    (D = 256: the signs flip the A operand instead -- an XOR of fp16 sign bits -- and B
//    is H_16 itself, which keeps 32 sign masks in registers instead of 64 B fragments;
//    one CTA of 8 warps per SM.)  fp32 rows are split exactly into three bf16 parts,
//    x = hi + mid + lo (8 significant bits each), and the three MMAs accumulate into one
//    fp32 result; the products with +-1 are exact, so only the fp32 accumulation rounds,
//    as in an fp32 transform.
//  * Norm.  ||y||^2 = D ||x||^2: a sum of the thread's squares plus two quad shuffles.
//  * Quantiser.  u = y / sqrt(sum y^2) lies in [-1, 1]; N equal cells cover that range
//    and each stores (number of decision points below the cell, the first decision point
//    at or above it), with N chosen so that no decision point lies near a cell edge.
//    index = lo + (u > point): one compare, exact "#{k : boundary_k < u}" whichever cell
//    a rounding picks near an edge.  The table is replicated per lane (16 copies, 64-bit
//    entries) so the lookups are conflict free.
//  * Packing.  Bytes are assembled per row in shared memory (LSB-first fields, then the
//    fp32 norm); a token's H rows are contiguous in the page (H * row_bytes bytes), so the
//    warp stores whole token slabs with 16-byte stores.  4-bit fields fill a byte per
//    lane pair of coordinates, 2-bit ones a byte per quad; 3- and 5-bit fields cross
//    bytes, so their index pairs are staged (in the raw tile buffer the MMAs have
//    consumed) and each lane then packs 32 coordinates of a row into 3 or 5 whole words.
//  * Product rows (PROD, "QJL residual" keys: (b - 1)-bit MSE indices, D sign bits, nu,
//    gamma).  The quantiser also looks up c[idx] (a per-lane replicated copy of the
//    codebook), leaving the rotated residual r = u - c[idx] in the accumulators, and
//    gamma = ||r||.  The sketch S r of the CTA's 128 rows (8 warps x 16) is a
//    [128 x D] x [D x D] product on the 5th-generation tensor cores: each warp writes its
//    rows of r (scaled by 2^10) as fp16 hi + lo (lo x 2^12 more) into the A operand in the
//    canonical K-major layout, S sits in shared memory as fp16 hi + lo the same way, and one
//    thread issues tcgen05.mma (M 128, N D, K 16) for r_hi S_hi into one TMEM accumulator
//    and r_lo S_hi + r_hi S_lo into a second; r_hi S_hi + (r_lo S_hi + r_hi S_lo) 2^-12
//    carries ~22 bits, so a sign flips only where the projection is within ~1e-6 of zero.
//    Each warp reads its TMEM lane quarter back (32 rows x D/2 columns): one thread per row,
//    so 32 consecutive columns are a sign word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kWWarps = 8;          // warps per CTA
constexpr int kGridMaxA = 128;       // largest grid scale: 2 * 128 cells over u in [-1, 1]
constexpr int kQCells = 2 * kGridMaxA + 1;  // quantiser table entries
constexpr int kQCopies = 16;        // lane copies of the quantiser table

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16_w(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16_w_zfill(uint32_t dst, const void* src, int valid_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit_w() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait_w() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}
// d = A * B (zero accumulator input), m16n8k16, fp32 result.
template <typename T>
__device__ __forceinline__ void mma_rot(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1);
template <>
__device__ __forceinline__ void mma_rot<__half>(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
template <>
__device__ __forceinline__ void mma_rot<__nv_bfloat16>(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
// ---- tcgen05 (the sketch of product rows) ------------------------------------------------
// Shared-memory matrix descriptor of an operand in the canonical K-major layout without
// swizzle: 8-row x 16-byte core matrices of 128 contiguous bytes, `lbo` bytes between the
// two core matrices of a 16-element k-step, `sbo` bytes between 8-row groups.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | ((uint64_t)1 << 46);
}
// D[tmem] (+)= A B^T, kind::f16 (issued by one thread)
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// the mbarrier completes when every MMA issued so far by this thread has
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape, one warp)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// Waits for the phase of `bar` with parity `parity`; false after `tries` unsuccessful tries.
__device__ __forceinline__ bool mbar_wait_w(uint32_t bar, uint32_t parity, uint32_t tries) {
  for (uint32_t i = 0; i < tries; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// d = A * B + d, bf16 operands (the parts of fp32 rows)
__device__ __forceinline__ void mma_acc_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Exact split of two fp32 values into three bf16 pairs: x = hi + mid + lo.  Each
// difference below is exact in fp32 (it keeps the low bits of a number within a factor of
// two of the one rounded), and what is left after two roundings to 8 significant bits has
// at most 8 of its own.
__device__ __forceinline__ void split3_bf16(float2 x, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
  const float2 minus1 = make_float2(-1.f, -1.f);
  const float2 r1 = __ffma2_rn(__bfloat1622float2(h), minus1, x);  // x - hi, exact
  const __nv_bfloat162 m = __floats2bfloat162_rn(r1.x, r1.y);
  const float2 r2 = __ffma2_rn(__bfloat1622float2(m), minus1, r1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(r2.x, r2.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  mid = *reinterpret_cast<const uint32_t*>(&m);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// +-1 pair in the operand type: sign bits of the two halves from s0, s1 (true = negative)
template <typename T>
__device__ __forceinline__ uint32_t pm1_pair(bool neg0, bool neg1) {
  const uint32_t one = std::is_same<T, __half>::value ? 0x3C00u : 0x3F80u;
  return (one | (neg0 ? 0x8000u : 0u)) | ((one | (neg1 ? 0x8000u : 0u)) << 16);
}

struct QCell {
  int lo;       // decision points strictly below the cell
  float point;  // grid coordinate of the first decision point at or above the cell start (+inf if none)
};

struct WriteTcArgs {
  WriteArgs a;
  const float* smat;  // product rows: S, fp32 [D][D] row-major
};

// Quantiser grid g = u A + B, B = A + phi with 0 < phi < 1, cell = floor(g).  u is a
// coordinate of a unit vector, so g stays in [phi, 2A + phi] up to rounding: cells 0 to
// 2A, with no clamp (the unsigned conversion also maps a negative g or a NaN to cell 0).
// (A, phi) is the first pair, largest A first, that keeps every decision point b_k at
// least 1/64 cell from a cell edge and no two in one cell.  Deterministic, so every CTA
// picks the same grid.  Returns false when no pair qualifies (the caller then reports
// an error instead of writing).
// Run by the 32 lanes of one warp: candidate i = 4 (row of n) + phase, in the order
// n = kGridMaxA, kGridMaxA - 2, ... and phases {1/2, 1/4, 3/4, 3/8}; lane l tests the
// candidates l, l + 32, ..., and the first passing candidate in that order wins.
__device__ bool choose_grid(const float* b, int m, int lane, float& q_a, float& q_b) {
  const float phases[4] = {0.5f, 0.25f, 0.75f, 0.375f};
  constexpr int kCands = 4 * (kGridMaxA / 2 - kGridMaxA / 8 + 1);
  for (int base = 0; base < kCands; base += 32) {
    const int i = base + lane;
    const int n = kGridMaxA - 2 * (i >> 2);
    const float ga = (float)n, gb = (float)n + phases[i & 3];
    bool ok = i < kCands;
    int prev = -1;
    for (int k = 0; k < m && ok; ++k) {
      const float x = fmaf(b[k], ga, gb);
      const int cell = (int)floorf(x);
      const float f = x - (float)cell;
      ok = cell > prev && f >= 1.0f / 64 && f <= 63.0f / 64;
      prev = cell;
    }
    const unsigned hit = __ballot_sync(kFullMask, ok);
    if (hit) {
      const int src = __ffs(hit) - 1;
      q_a = __shfl_sync(kFullMask, ga, src);
      q_b = __shfl_sync(kFullMask, gb, src);
      return true;
    }
  }
  return false;
}

// CTAs per SM: one where the raw tiles of 8 warps take 8 KB each (16 rows of 256 fp16 or of
// 128 fp32 coordinates) or the sketch matrix takes 64 KB (product rows at D = 128), two
// otherwise.
template <typename T, int D, bool PROD>
__host__ __device__ constexpr int write_tc_ctas_per_sm() {
  return (D * (int)sizeof(T) >= 512 || (PROD && D == 128)) ? 1 : 2;
}
// Bytes of the shared-memory part ahead of the per-warp buffers: quantiser table, and for
// product rows the codebook copies and S hi / lo.
template <int D, bool PROD>
__host__ __device__ constexpr int write_tc_fixed_smem() {
  // product rows: codebook copies, S hi / lo (D x D fp16 each), the sketch's A operand hi / lo
  // (128 rows x D fp16 each)
  return kQCells * kQCopies * (int)sizeof(QCell) + (PROD ? 16 * 32 * 4 + 4 * D * D + 512 * D : 0);
}
template <int D, int BITS, bool PROD>
__host__ __device__ constexpr int write_tc_row_bytes() {
  return PROD ? D * BITS / 8 + D / 8 + 8 : D * BITS / 8 + 4;
}

// Product rows: BITS is the MSE index width (b - 1).
template <typename T, int D, int BITS, bool PROD>
__global__ void __launch_bounds__(kWWarps * 32, write_tc_ctas_per_sm<T, D, PROD>()) write_tc_kernel(WriteTcArgs args) {
  constexpr bool kF32Rows = std::is_same<T, float>::value;
  using OpT = typename std::conditional<kF32Rows, __nv_bfloat16, T>::type;  // MMA operand type
  static_assert(!kF32Rows || D <= 128, "fp32 rows at head_dim 64 or 128");
  static_assert(!PROD || (D <= 128 && BITS >= 2 && BITS <= 4), "product rows: D 64 / 128, 2- to 4-bit indices");
  constexpr int NB = D / 16;            // 16-column blocks
  constexpr int RB = write_tc_row_bytes<D, BITS, PROD>();  // row bytes
  constexpr int IB = D * BITS / 8;      // index bytes
  constexpr int ROWB = D * (int)sizeof(T);  // raw row bytes
  constexpr int TILE_BYTES = 16 * ROWB;
  const WriteArgs& a = args.a;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int H = a.num_kv_heads;

  // shared memory: quantiser table | per warp: 2 raw tiles + 1 packed tile
  constexpr int kQC = kQCopies;
  QCell* qtab = reinterpret_cast<QCell*>(smem);
  // product rows: codebook, 32 lane copies (entry k of lane l at 4 (32 k + l)); S hi, S lo;
  // the sketch's A operand hi, lo (all operands in the canonical K-major layout, kSbo bytes
  // between 8-row groups)
  float* ctab = reinterpret_cast<float*>(smem + kQCells * kQC * sizeof(QCell));
  unsigned char* s_hi = smem + kQCells * kQC * sizeof(QCell) + 16 * 32 * 4;
  unsigned char* s_lo = s_hi + D * D * 2;
  unsigned char* a_hi = s_lo + D * D * 2;
  unsigned char* a_lo = a_hi + 128 * D * 2;
  constexpr int kSbo = 16 * D;
  // instruction descriptor: fp32 D, fp16 A and B, both K-major, N = D, M = 128
  constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(D >> 3) << 17) | (8u << 24);
  // per warp: 2 raw tiles; once a tile's MMAs have read it, its buffer holds the 3/5-bit
  // index staging (kStage entries a row) and then the packed rows (at kPackOff)
  unsigned char* wbase = smem + write_tc_fixed_smem<D, PROD>() + warp * (2 * TILE_BYTES);
  constexpr int kStage = D / 2 + 8;
  constexpr int kPackOff = (BITS == 3 || BITS == 5) ? 16 * kStage * 2 : 0;
  static_assert(kPackOff + 16 * RB <= TILE_BYTES, "staging and packed rows must fit a raw tile buffer");
  unsigned char* raw_buf = wbase;

  // decision points (correctly rounded midpoints of neighbouring fp32 centroids) and
  // the quantiser grid
  constexpr int NC = 1 << BITS;
  __shared__ float bnd[NC - 1];
  __shared__ float grid_a, grid_b;
  __shared__ int grid_ok;
  if (threadIdx.x < NC - 1) bnd[threadIdx.x] = 0.5f * (a.centroids[threadIdx.x] + a.centroids[threadIdx.x + 1]);
  __syncthreads();
  if (warp == 0) {
    float ga = 0.f, gb = 0.f;
    const bool found = choose_grid(bnd, NC - 1, lane, ga, gb);
    if (lane == 0) {
      grid_ok = found ? 1 : 0;
      grid_a = ga;
      grid_b = gb;
      if (!found && blockIdx.x == 0) atomicMax(a.status, (int32_t)kUnsupported);
    }
  }
  __syncthreads();
  if (!grid_ok) return;  // bad codebook: write nothing
  const float q_a = grid_a, q_b = grid_b;  // grid coordinate g = u * q_a + q_b, cell = floor(g)
  // The loop works in g' = g - 1/2 (exact: q_b is a small multiple of 1/8): adding
  // 1.5 * 2^23 to g' leaves round(g') in the low mantissa bits, which is floor(g) but
  // for g within rounding of an integer, where it may be floor(g) - 1 -- harmless, as no
  // decision point lies within 1/64 cell of a cell edge.  g >= phi >= 1/4 keeps it >= 0.
  const float q_bs = q_b - 0.5f;
  for (int cell = threadIdx.x; cell < kQCells; cell += blockDim.x) {
    // cell [cell, cell + 1) in grid units: decision points below its start, first one at or above
    int below = 0;
    float point = INFINITY;
    for (int k = 0; k < NC - 1; ++k) {
      const float gk = fmaf(bnd[k], q_a, q_b);
      if (gk < (float)cell) ++below;
      else if (point == INFINITY) point = gk;
    }
    QCell q;
    q.lo = below;
    q.point = point - 0.5f;  // in g' (exact, and +inf stays +inf)
#pragma unroll
    for (int copy = 0; copy < kQC; ++copy) qtab[cell * kQC + copy] = q;
  }
  if constexpr (PROD) {
    for (int i = threadIdx.x; i < NC * 32; i += blockDim.x) ctab[i] = a.centroids[i >> 5];
    // S[n][k] (n: projection, k: coordinate) as fp16 hi and lo x 2^12, the B operand of the
    // sketch: N = D rows of D k-columns, canonical K-major
    for (int i = threadIdx.x; i < D * D; i += blockDim.x) {
      const int n = i / D, k = i - n * D;
      const float sv = __ldg(args.smat + i);
      const __half hi = __float2half_rn(sv);
      const __half lo = __float2half_rn((sv - __half2float(hi)) * 4096.0f);
      const int off = (n >> 3) * kSbo + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
      *reinterpret_cast<__half*>(s_hi + off) = hi;
      *reinterpret_cast<__half*>(s_lo + off) = lo;
    }
  }
  __syncthreads();

  // B fragments: B_j[k][n] = s[16 j + k] * (-1)^popcount(k & n); this lane holds
  // k in {2c, 2c+1} (reg 0) and {2c+8, 2c+9} (reg 1) for n = r (+8 for n-tile 1).
  // D = 256: the sign flip goes onto the A operand (asgn[j][part]: sign bits of columns
  // 16 j + 2c + 8 part, +1 in the fp16 / bf16 pair layout) and bfr[0] holds H_16 alone.
  constexpr bool kSignOnA = D == 256;
  constexpr int NBF = kSignOnA ? 1 : NB;
  uint32_t asgn[kSignOnA ? NB : 1][2];
  if constexpr (kSignOnA) {
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int k0 = 16 * j + 2 * c + 8 * part;
        asgn[j][part] = (__ldg(a.signs + k0) < 0.f ? 0x8000u : 0u) | (__ldg(a.signs + k0 + 1) < 0.f ? 0x80000000u : 0u);
      }
  }
  uint32_t bfr[NBF][2][2];
#pragma unroll
  for (int j = 0; j < NBF; ++j) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int n = r + 8 * nt;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int k0 = 2 * c + 8 * part, k1 = k0 + 1;
        const bool s0 = kSignOnA ? false : (__ldg(a.signs + 16 * j + k0) < 0.f);
        const bool s1 = kSignOnA ? false : (__ldg(a.signs + 16 * j + k1) < 0.f);
        const bool n0 = s0 ^ (__popc(k0 & n) & 1);
        const bool n1 = s1 ^ (__popc(k1 & n) & 1);
        bfr[j][nt][part] = pm1_pair<OpT>(n0, n1);
      }
    }
  }
  // shared address of cell n, this lane's copy: bits(g' + 1.5 * 2^23) * 128 + q_addr_bias
  constexpr uint32_t kMagicBits = 0x4B400000u;  // bits of 1.5 * 2^23
  const uint32_t q_addr_bias =
      smem_addr(qtab) + (uint32_t)((lane & (kQC - 1)) * sizeof(QCell)) - kMagicBits * (uint32_t)(kQC * sizeof(QCell));

  // launched as a programmatic dependent of the slot validation: the set-up above overlaps
  // it; the status word is read once that grid has completed
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (*a.status != kOk) return;  // a slot failed validation: write nothing
  // product rows: 2 D TMEM columns (D_main, D_lo of the sketch) and the MMA mbarrier
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t mma_bar;
  uint32_t tmem = 0, mma_phase = 0;
  if constexpr (PROD) {
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&tmem_slot)),
                   "n"(2 * D)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (threadIdx.x == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(&mma_bar)) : "memory");
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    tmem = tmem_slot;
  }

  const int64_t num_rows = a.num_tokens * H;
  const int64_t num_tiles = (num_rows + 15) / 16;
  const int64_t wstride = (int64_t)gridDim.x * kWWarps;
  const T* raw = static_cast<const T*>(a.raw);

  // issue the cp.async of tile `tile` into raw buffer `buf` (16 rows x ROWB bytes,
  // 16-byte chunks XOR-swizzled by row so that ldmatrix reads are conflict free)
  auto load_tile = [&](int64_t tile, int buf) {
    if (tile < num_tiles) {
      const unsigned char* src = reinterpret_cast<const unsigned char*>(raw) + tile * TILE_BYTES + lane * 16;
      const uint32_t dst0 = smem_addr(raw_buf + buf * TILE_BYTES);
      constexpr int CH = TILE_BYTES / 16, CPR = ROWB / 16;
      if ((tile + 1) * 16 <= num_rows) {  // whole tile: no per-chunk checks
#pragma unroll
        for (int k = 0; k < CH / 32; ++k) {
          const int i = lane + 32 * k, row = i / CPR, col = i % CPR;
          cp_async16_w(dst0 + row * ROWB + ((col ^ (row & 7)) << 4), src + k * 512);
        }
      } else {
        const int64_t bytes_left = (num_rows - tile * 16) * ROWB;
#pragma unroll
        for (int k = 0; k < CH / 32; ++k) {
          const int i = lane + 32 * k, row = i / CPR, col = i % CPR;
          const uint32_t dst = dst0 + row * ROWB + ((col ^ (row & 7)) << 4);
          if ((int64_t)i * 16 + 16 <= bytes_left) cp_async16_w(dst, src + k * 512);
          else cp_async16_w_zfill(dst, src - lane * 16, 0);  // past the last row: zero fill, no read
        }
      }
    }
    cp_commit_w();
  };

  // chunk i of a tile belongs to token i / d, d = H * RB / 16: a reciprocal multiply,
  // (i * ceil(2^16 / d)) >> 16, exact for i < 2^16 / d -- here i < RB <= 164 and d <= 164
  const uint32_t cpt = (uint32_t)(H * RB / 16 > 0 ? H * RB / 16 : 1);
  const uint32_t inv_cpt = (65536u + cpt - 1) / cpt;
  int64_t tile = (int64_t)blockIdx.x * kWWarps + warp;
  int buf = 0;
  load_tile(tile, 0);
  // every warp of a CTA runs the same iterations (product rows meet at CTA barriers); a warp
  // whose tile is past the end only keeps up
  for (int64_t ctile = (int64_t)blockIdx.x * kWWarps; ctile < num_tiles; ctile += wstride, tile += wstride, buf ^= 1) {
    const bool active = tile < num_tiles;
    load_tile(tile + wstride, buf ^ 1);
    unsigned char* pack_buf = raw_buf + buf * TILE_BYTES + kPackOff;
    // Re-encode of the tile rows in `rows` (bit rr: row rr) from their raw values, one row at a
    // time by the whole warp, lane l holding coordinates [l E, l E + E): the row is first
    // scaled by 2^-ex (ex the exponent of its largest |x|; exact), then rotated (warp FWHT),
    // its indices found as #{b_k < u} and OR'd into the cleared index bytes, its norm scaled
    // back; a row with a NaN or infinite coordinate gets u = 0 and its non-finite sum as the
    // norm.  Product rows also get their residual norm and their rows of the sketch operand.
    auto reencode_rows = [&](uint32_t rows) {
      constexpr int E = D / 32;
      while (rows != 0u) {
        const int rr = __ffs(rows) - 1;
        rows &= rows - 1u;
        if (tile * 16 + rr >= num_rows) continue;  // the zero-filled tail of the last tile
        const T* src = raw + (tile * 16 + rr) * (int64_t)D + lane * E;
        float x[E];
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          x[i] = to_f32(src[i]);
          m = fmaxf(m, fabsf(x[i]));
        }
        m = warp_max(m);
        int ex = 0;
        if (m > 0.f && m <= 3.402823466e38f) frexpf(m, &ex);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          x[i] = scale_pow2(x[i], -ex);
          ss = fmaf(x[i], x[i], ss);
        }
        ss = warp_sum(ss);
        const bool bad = !(ss <= 3.402823466e38f);
#pragma unroll
        for (int i = 0; i < E; ++i) x[i] *= __ldg(a.signs + lane * E + i);
        fwht_warp<E>(x);
        const float inv = (bad || !(ss > 0.f)) ? 0.f : 1.0f / sqrtf((float)D * ss);
        const float nu = bad ? ss : scale_pow2(sqrtf(ss), ex);
        unsigned char* prow = pack_buf + rr * RB;
        for (int w = lane; w < IB / 4; w += 32) reinterpret_cast<uint32_t*>(prow)[w] = 0u;
        __syncwarp();
        float rsq = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const float u = bad ? 0.f : x[i] * inv;
          int idx = 0;
          for (int k = 0; k < NC - 1; ++k) idx += u > bnd[k] ? 1 : 0;
          const int j = lane * E + i;
          const int bit = j * BITS, wi = bit >> 5, o = bit & 31;
          atomicOr(reinterpret_cast<uint32_t*>(prow) + wi, (uint32_t)idx << o);
          if (o + BITS > 32) atomicOr(reinterpret_cast<uint32_t*>(prow) + wi + 1, (uint32_t)idx >> (32 - o));
          if constexpr (PROD) {
            const float rv = u - ctab[idx * 32 + lane];
            rsq = fmaf(rv, rv, rsq);
            const float xx = rv * 1024.0f;
            const __half hi = __float2half_rn(xx);
            const __half lo = __float2half_rn((xx - __half2float(hi)) * 4096.0f);
            const int arow = 16 * warp + rr;
            const int off = (arow >> 3) * kSbo + (j >> 3) * 128 + (arow & 7) * 16 + (j & 7) * 2;
            *reinterpret_cast<__half*>(a_hi + off) = hi;
            *reinterpret_cast<__half*>(a_lo + off) = lo;
          }
        }
        if constexpr (PROD) {
          const float gamma = sqrtf(warp_sum(rsq));
          if (lane == 0) {
            *reinterpret_cast<float*>(prow + IB + D / 8) = nu;
            *reinterpret_cast<float*>(prow + IB + D / 8 + 4) = gamma;
          }
        } else {
          if (lane == 0) *reinterpret_cast<float*>(prow + IB) = nu;
        }
        __syncwarp();
      }
    };
    // slot of the tile's token `lane` for the slab store below (a global load, read early)
    int64_t my_slot = -1;
    if (16 % H == 0 && lane < 16 / H) {
      const int64_t t = tile * 16 / H + lane;
      if (t < a.num_tokens) my_slot = __ldg(a.slots + t);
    }
    cp_wait_w<1>();
    __syncwarp();
    if (active) {
    // ---- rotation: MMA per block, then butterflies across blocks ------------------
    // acc[j][nt] = (row r: cols 2c, 2c+1 | row r+8: cols 2c, 2c+1) of block j, n-tile nt
    float acc[NB][2][4];
    const uint32_t tbase = smem_addr(raw_buf + buf * TILE_BYTES);
    if constexpr (kF32Rows) {
      // A fragment of block j from the fp32 tile: a0 row r cols 16j + 2c, +1; a1 row r + 8;
      // a2, a3 the same at cols + 8 (8-byte loads from the swizzled 16-byte chunks)
      const unsigned char* tb = raw_buf + buf * TILE_BYTES;
      auto ld2 = [&](int row, int col) -> float2 {
        const int chunk = col >> 2;
        return *reinterpret_cast<const float2*>(tb + row * ROWB + ((chunk ^ (row & 7)) << 4) + (col & 3) * 4);
      };
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        uint32_t h[4], m[4], l[4];
        split3_bf16(ld2(r, 16 * j + 2 * c), h[0], m[0], l[0]);
        split3_bf16(ld2(r + 8, 16 * j + 2 * c), h[1], m[1], l[1]);
        split3_bf16(ld2(r, 16 * j + 2 * c + 8), h[2], m[2], l[2]);
        split3_bf16(ld2(r + 8, 16 * j + 2 * c + 8), h[3], m[3], l[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma_rot<OpT>(acc[j][nt], h[0], h[1], h[2], h[3], bfr[j][nt][0], bfr[j][nt][1]);
          mma_acc_bf16(acc[j][nt], m[0], m[1], m[2], m[3], bfr[j][nt][0], bfr[j][nt][1]);
          mma_acc_bf16(acc[j][nt], l[0], l[1], l[2], l[3], bfr[j][nt][0], bfr[j][nt][1]);
        }
      }
    } else {
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      // ldmatrix.x4: lanes 0-7 rows 0-7 cols 16j..+7, 8-15 rows 8-15, 16-23 rows 0-7 cols +8, 24-31 rows 8-15 cols +8
      const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int chunk = 2 * j + (lane >> 4);
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(tbase + row * ROWB + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
      if constexpr (kSignOnA) {  // a0/a1: columns 2c, 2c+1; a2/a3: columns 2c+8, 2c+9 of block j
        a0 ^= asgn[j][0];
        a1 ^= asgn[j][0];
        a2 ^= asgn[j][1];
        a3 ^= asgn[j][1];
      }
      const int jb = kSignOnA ? 0 : j;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) mma_rot<T>(acc[j][nt], a0, a1, a2, a3, bfr[jb][nt][0], bfr[jb][nt][1]);
    }
    }
    const float2 minus1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int hs = 1; hs < NB; hs <<= 1) {
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if ((j & hs) == 0) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const float2 x = make_float2(acc[j][nt][e], acc[j][nt][e + 1]);
              const float2 y = make_float2(acc[j + hs][nt][e], acc[j + hs][nt][e + 1]);
              const float2 sum = __fadd2_rn(x, y), dif = __ffma2_rn(y, minus1, x);
              acc[j][nt][e] = sum.x;
              acc[j][nt][e + 1] = sum.y;
              acc[j + hs][nt][e] = dif.x;
              acc[j + hs][nt][e + 1] = dif.y;
            }
        }
      }
    }
    // ---- norms of rows r (e = 0, 1) and r + 8 (e = 2, 3) -----------------------------
    auto row_sums = [&](float& ss0, float& ss1) {
      float2 ssv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // row r: independent chains
      float2 ssw[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // row r + 8
#pragma unroll
      for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 p = make_float2(acc[j][nt][0], acc[j][nt][1]);
          const float2 q = make_float2(acc[j][nt][2], acc[j][nt][3]);
          ssv[nt] = __ffma2_rn(p, p, ssv[nt]);
          ssw[nt] = __ffma2_rn(q, q, ssw[nt]);
        }
      ss0 = (ssv[0].x + ssv[0].y) + (ssv[1].x + ssv[1].y);
      ss1 = (ssw[0].x + ssw[0].y) + (ssw[1].x + ssw[1].y);
      ss0 += __shfl_xor_sync(kFullMask, ss0, 1);
      ss0 += __shfl_xor_sync(kFullMask, ss0, 2);
      ss1 += __shfl_xor_sync(kFullMask, ss1, 1);
      ss1 += __shfl_xor_sync(kFullMask, ss1, 2);
    };
    float ss0, ss1;
    row_sums(ss0, ss1);
    // Rows whose sum of squares leaves [2^-100, 2^100] -- rows of extreme scale (bf16 and fp32
    // coordinates beyond about 1e14 or below about 1e-16), zero rows, and rows with a NaN or
    // infinite coordinate -- are encoded here as zero rows (coordinates and row scale 0, so
    // every grid coordinate is a valid cell) and re-encoded after packing by the warp from
    // their raw values (`odd_rows`, below), away from this common path.
    const bool odd0 = !(ss0 <= 0x1p100f) || ss0 < 0x1p-100f;  // (zero rows too: their sum may have underflowed)
    const bool odd1 = !(ss1 <= 0x1p100f) || ss1 < 0x1p-100f;
    // ||x|| = sqrt(ss / D); u = y / sqrt(ss); grid coordinate g = u * q_a + q_b.
    // Every partial sum above only grows, so y^2 <= ss (1 + 2^-23) + 2^-150 for each y of
    // the row, even when ss is subnormal; adding 2^-149 under the root keeps |u| within a
    // few ulp of 1 and g inside [1/4, 2 q_a + 1/2) with no clamp (it moves ss by at most one
    // ulp, and only below 2^-124; an all-zero row gets g = q_b, i.e. u = 0).  rsqrtf (2 ulp)
    // is enough: it moves g by < 1e-4 cell and u by < 1e-6, inside the decision tolerance,
    // and the stored norm ss * rsqrt(ss) / sqrt(D) by < 1e-6 relative.
    const float rs0 = odd0 ? 0.f : rsqrtf(ss0 + 0x1p-149f), rs1 = odd1 ? 0.f : rsqrtf(ss1 + 0x1p-149f);
    const float inv_sqrt_d = 1.0f / sqrtf((float)D);
    const float nu0 = ss0 * rs0 * inv_sqrt_d, nu1 = ss1 * rs1 * inv_sqrt_d;
    // bit rr: row rr of the tile needs the re-encode (each quad votes for its rows r, r + 8)
    const uint32_t odd_b0 = __ballot_sync(kFullMask, odd0), odd_b1 = __ballot_sync(kFullMask, odd1);
    if (__builtin_expect((odd_b0 | odd_b1) != 0u, 0)) {
      // the flagged rows' coordinates may be NaN or infinite: zero them, so that with the row
      // scale 0 their grid coordinate is q_b exactly (a valid cell) and their residual finite
#pragma unroll
      for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if (odd0) acc[j][nt][0] = acc[j][nt][1] = 0.f;
          if (odd1) acc[j][nt][2] = acc[j][nt][3] = 0.f;
        }
    }
    const float ga0 = q_a * rs0, ga1 = q_a * rs1;

    // ---- quantise and pack into this warp's row buffer ------------------------------
    // the cell and the comparison both use the grid coordinate; exact for every u not
    // within a few ulp of a decision point, whichever neighbouring cell it lands in
    // g: shifted grid coordinate g'; m: g' + 1.5 * 2^23 (its bits give the cell)
    auto quant = [&](float g, float m) -> uint32_t {
      const uint32_t addr = __float_as_uint(m) * (uint32_t)(kQC * sizeof(QCell)) + q_addr_bias;
      uint32_t lo, pt;
      asm("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(lo), "=r"(pt) : "r"(addr));
      return lo + (g > __uint_as_float(pt) ? 1u : 0u);
    };
    const float2 magic2 = make_float2(12582912.0f, 12582912.0f);
    // 3/5 bits: index pairs (2 BITS bits each) of row rr, coordinates 2p, 2p + 1, at
    // stage[rr * kStage + p]; the tile's raw buffer is free once its MMAs have read it.  Rows
    // are kStage = D / 2 + 8 entries apart (16-byte aligned for the packing's loads, and 4 banks
    // apart, so the 8 rows of a store land in different banks)
    uint16_t* stage = reinterpret_cast<uint16_t*>(raw_buf + buf * TILE_BYTES);
    const uint32_t ctab_lane = smem_addr(ctab) + (uint32_t)(lane * 4);
    float rr[2] = {0.f, 0.f};  // product rows: sum of squared residuals of rows r, r + 8
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // row r (half 0) / row r + 8 (half 1)
      const float ga = half ? ga1 : ga0;
      const float2 gav = make_float2(ga, ga), gbv = make_float2(q_bs, q_bs);
      unsigned char* prow = pack_buf + (r + 8 * half) * RB;
#pragma unroll
      for (int j = 0; j < NB; ++j) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 g = __ffma2_rn(make_float2(acc[j][nt][2 * half], acc[j][nt][2 * half + 1]), gav, gbv);
          const float2 m = __fadd2_rn(g, magic2);
          const uint32_t i0 = quant(g.x, m.x);
          const uint32_t i1 = quant(g.y, m.y);
          if constexpr (PROD) {  // residual r = u - c[idx], u = y / sqrt(sum y^2)
            const float rsh = half ? rs1 : rs0;
            float c0, c1;
            asm("ld.shared.f32 %0, [%1];\n" : "=f"(c0) : "r"(ctab_lane + i0 * 128u));
            asm("ld.shared.f32 %0, [%1];\n" : "=f"(c1) : "r"(ctab_lane + i1 * 128u));
            const float e0 = fmaf(acc[j][nt][2 * half], rsh, -c0);
            const float e1 = fmaf(acc[j][nt][2 * half + 1], rsh, -c1);
            acc[j][nt][2 * half] = e0;
            acc[j][nt][2 * half + 1] = e1;
            rr[half] = fmaf(e0, e0, fmaf(e1, e1, rr[half]));
          }
          // columns 16 j + 8 nt + 2c, +1
          if (BITS == 3 || BITS == 5) {
            stage[(r + 8 * half) * kStage + 8 * j + 4 * nt + c] = (uint16_t)(i0 | (i1 << BITS));
          } else if (BITS == 4) {
            prow[8 * j + 4 * nt + c] = (unsigned char)(i0 + (i1 << 4));
          } else {
            // 2 bits: byte 4 j + 2 nt + c/2 holds columns 16 j + 8 nt + 4 (c/2) .. +3
            const uint32_t mine = i0 | (i1 << 2);
            const uint32_t other = __shfl_xor_sync(kFullMask, mine, 1);
            if ((c & 1) == 0) prow[4 * j + 2 * nt + (c >> 1)] = (unsigned char)(mine | (other << 4));
          }
        }
      }
      if constexpr (PROD) {
        rr[half] += __shfl_xor_sync(kFullMask, rr[half], 1);
        rr[half] += __shfl_xor_sync(kFullMask, rr[half], 2);
        if (c == 0) {
          *reinterpret_cast<float*>(prow + IB + D / 8) = half ? nu1 : nu0;
          *reinterpret_cast<float*>(prow + IB + D / 8 + 4) = sqrtf(rr[half]);
        }
      } else {
        if (c == 0) *reinterpret_cast<float*>(prow + IB) = half ? nu1 : nu0;
      }
    }
    if constexpr (PROD) {
      // ---- this warp's rows of the sketch's A operand: r x 2^10 as fp16 hi and lo x 2^12,
      // rows 16 warp + r (+ 8) of the CTA tile, in the canonical K-major layout.  The
      // accumulator layout already is the A layout: block j, part q holds row r (+ 8 for odd q),
      // columns 16 j + 2c, +1 (+ 8 for q >= 2).
#pragma unroll
      for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int nt = q >> 1, e = 2 * (q & 1);
          const float x0 = acc[j][nt][e] * 1024.0f, x1 = acc[j][nt][e + 1] * 1024.0f;
          const __half2 h = __floats2half2_rn(x0, x1);
          const float2 hf = __half22float2(h);
          const __half2 l = __floats2half2_rn((x0 - hf.x) * 4096.0f, (x1 - hf.y) * 4096.0f);
          const int off = (2 * warp + (q & 1)) * kSbo + (2 * j + (q >> 1)) * 128 + r * 16 + c * 4;
          *reinterpret_cast<__half2*>(a_hi + off) = h;
          *reinterpret_cast<__half2*>(a_lo + off) = l;
        }
    }
    __syncwarp();
    if constexpr (BITS == 3 || BITS == 5) {
      // group = 32 coordinates (16 pairs) of one row -> BITS words at byte 4 BITS q of the row
      constexpr int GPR = D / 32;  // groups per row
#pragma unroll
      for (int k = 0; k < 16 * GPR / 32; ++k) {
        const int g = lane + 32 * k, row = g / GPR, q = g % GPR;
        const uint4* src = reinterpret_cast<const uint4*>(stage + row * kStage + q * 16);
        const uint4 v0 = src[0], v1 = src[1];
        const uint32_t w8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t out[BITS];
#pragma unroll
        for (int w = 0; w < BITS; ++w) out[w] = 0u;
#pragma unroll
        for (int p = 0; p < 16; ++p) {  // pair p: 2 BITS bits at stream bit 2 BITS p
          const uint32_t pv = (w8[p >> 1] >> (16 * (p & 1))) & ((1u << (2 * BITS)) - 1u);
          const int bit = 2 * BITS * p, w = bit >> 5, sh = bit & 31;
          out[w] |= pv << sh;
          if (sh + 2 * BITS > 32) out[w + 1] |= pv >> (32 - sh);
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(pack_buf + row * RB + q * 4 * BITS);
#pragma unroll
        for (int w = 0; w < BITS; ++w) dst[w] = out[w];
      }
      __syncwarp();
    }

      // ---- re-encode of the rows flagged above, one row at a time by the whole warp -------
      if (__builtin_expect((odd_b0 | odd_b1) != 0u, 0)) {
        uint32_t odd_rows = 0u;  // bit rr: row rr of the tile
#pragma unroll
        for (int q = 0; q < 8; ++q) odd_rows |= ((odd_b0 >> (4 * q)) & 1u) << q | ((odd_b1 >> (4 * q)) & 1u) << (q + 8);
        reencode_rows(odd_rows);
      }
    }  // active

    if constexpr (PROD) {
      // ---- sketch S r of the CTA's 128 rows on the tensor cores (tcgen05): D_main =
      // r_hi S_hi^T, D_lo = r_lo S_hi^T + r_hi S_lo^T in TMEM, one 128 x D x 16 MMA per
      // k-step and product, issued by one thread; then each warp reads 32 rows (its TMEM lane
      // quarter) x D/2 columns back and writes their sign words to the owners' row buffers.
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      __syncthreads();
      if (threadIdx.x == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        const uint32_t ah = smem_addr(a_hi), al = smem_addr(a_lo), bh = smem_addr(s_hi), bl = smem_addr(s_lo);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (uint32_t)(256 * k);  // two 8-column core matrices per k-step
          umma_f16(tmem, umma_desc(ah + ko, 128, kSbo), umma_desc(bh + ko, 128, kSbo), kIdesc, k > 0);
          umma_f16(tmem + D, umma_desc(al + ko, 128, kSbo), umma_desc(bh + ko, 128, kSbo), kIdesc, k > 0);
          umma_f16(tmem + D, umma_desc(ah + ko, 128, kSbo), umma_desc(bl + ko, 128, kSbo), kIdesc, true);
        }
        umma_commit(smem_addr(&mma_bar));
      }
      const bool landed = mbar_wait_w(smem_addr(&mma_bar), mma_phase, kDefaultWaitTries);
      if (__syncthreads_or(!landed)) {  // the MMAs did not complete in time: stop, no rows written
        if (threadIdx.x == 0) atomicMax(a.status, (int32_t)kTimeout);
        mbar_wait_w(smem_addr(&mma_bar), mma_phase, kDefaultWaitTries);
        break;
      }
      mma_phase ^= 1u;
      asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
      const int quarter = warp & 3, part = warp >> 2;
      const int crow = 32 * quarter + lane;  // this thread's row of the CTA tile
      unsigned char* owner = smem + write_tc_fixed_smem<D, PROD>() + (crow >> 4) * (2 * TILE_BYTES) + buf * TILE_BYTES +
                             kPackOff + (crow & 15) * RB + IB;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = part * (D / 2) + 32 * cc;
        uint32_t vm[32], vl[32];
        tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)col, vm);
        tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(D + col), vl);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
        uint32_t word = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (fmaf(__uint_as_float(vl[j]), 1.0f / 4096, __uint_as_float(vm[j])) >= 0.f) word |= 1u << j;
        *reinterpret_cast<uint32_t*>(owner + 4 * (col >> 5)) = word;
      }
      asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
      __syncthreads();
    }

    if (active) {
    // ---- store: token slabs (H rows) or single rows ---------------------------------
    const int64_t row0 = tile * 16;
    if (16 % H == 0 && (H * RB) % 16 == 0) {
      constexpr int CH16 = 16 * RB / 16;  // 16-byte chunks in the tile
#pragma unroll
      for (int k = 0; k < (CH16 + 31) / 32; ++k) {
        const int i = lane + 32 * k;
        const int tt = (int)(((uint32_t)min(i, CH16 - 1) * inv_cpt) >> 16);  // token within the tile
        const int64_t slot = __shfl_sync(kFullMask, my_slot, tt);
        if (i < CH16 && slot >= 0) {
          const int off = i * 16 - tt * H * RB;
          *reinterpret_cast<uint4*>(a.pages + slot * (int64_t)(H * RB) + off) =
              *reinterpret_cast<const uint4*>(pack_buf + i * 16);
        }
      }
    } else {
      for (int i = lane; i < 16 * (RB / 4); i += 32) {
        const int rr = i / (RB / 4), w = i % (RB / 4);
        const int64_t row = row0 + rr;
        if (row < num_rows) {
          const int64_t t = row / H;
          const int hh = (int)(row - t * H);
          const int64_t slot = __ldg(a.slots + t);
          if (slot >= 0)
            reinterpret_cast<uint32_t*>(a.pages + (slot * H + hh) * (int64_t)RB)[w] =
                reinterpret_cast<const uint32_t*>(pack_buf + rr * RB)[w];
        }
      }
    }
    }  // active
    __syncwarp();
  }
  cp_wait_w<0>();
  if constexpr (PROD) {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(2 * D) : "memory");
  }
}

}  // namespace

bool write_tc_supported(const WriteArgs& a) {
  const bool dt = a.dtype == kF16 || a.dtype == kBF16 || (a.dtype == kF32 && a.head_dim <= 128);
  const bool hd = a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256;
  const bool bt = a.bits >= 2 && a.bits <= 5;
  return dt && hd && bt && a.num_kv_heads >= 1;
}

// Launches `kern` as a programmatic dependent of the previous kernel on `stream` (the slot
// validation): it may start before that kernel completes and waits for it itself.
template <typename K>
cudaError_t launch_dependent(K kern, int grid, size_t smem, cudaStream_t stream, const WriteTcArgs& t) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kern, t);
  if (err == cudaSuccess) count_launches(1);
  return err;
}

cudaError_t launch_write_tc(const WriteArgs& a, cudaStream_t stream, int grid) {
  WriteTcArgs t;
  t.a = a;
#define TQ_WTC(T, D, BITS)                                                                                    \
  if (a.head_dim == D && a.bits == BITS) {                                                                    \
    const size_t smem = write_tc_fixed_smem<D, false>() + kWWarps * (2 * 16 * D * sizeof(T));                  \
    auto kern = write_tc_kernel<T, D, BITS, false>;                                                           \
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
    if (err != cudaSuccess) return err;                                                                       \
    return launch_dependent(kern, grid, smem, stream, t);                                                     \
  }
  if (a.dtype == kF32) {
    TQ_WTC(float, 64, 2) TQ_WTC(float, 64, 3) TQ_WTC(float, 64, 4) TQ_WTC(float, 64, 5)
    TQ_WTC(float, 128, 2) TQ_WTC(float, 128, 3) TQ_WTC(float, 128, 4) TQ_WTC(float, 128, 5)
  } else if (a.dtype == kF16) {
    TQ_WTC(__half, 64, 2) TQ_WTC(__half, 64, 3) TQ_WTC(__half, 64, 4) TQ_WTC(__half, 64, 5)
    TQ_WTC(__half, 128, 2) TQ_WTC(__half, 128, 3) TQ_WTC(__half, 128, 4) TQ_WTC(__half, 128, 5)
    TQ_WTC(__half, 256, 2) TQ_WTC(__half, 256, 3) TQ_WTC(__half, 256, 4) TQ_WTC(__half, 256, 5)
  } else if (a.dtype == kBF16) {
    TQ_WTC(__nv_bfloat16, 64, 2) TQ_WTC(__nv_bfloat16, 64, 3) TQ_WTC(__nv_bfloat16, 64, 4)
    TQ_WTC(__nv_bfloat16, 64, 5) TQ_WTC(__nv_bfloat16, 128, 2) TQ_WTC(__nv_bfloat16, 128, 3)
    TQ_WTC(__nv_bfloat16, 128, 4) TQ_WTC(__nv_bfloat16, 128, 5) TQ_WTC(__nv_bfloat16, 256, 2)
    TQ_WTC(__nv_bfloat16, 256, 3) TQ_WTC(__nv_bfloat16, 256, 4) TQ_WTC(__nv_bfloat16, 256, 5)
  }
#undef TQ_WTC
  return cudaErrorInvalidValue;
}

bool write_prod_tc_supported(const WriteArgs& a) {
  const bool dt = a.dtype == kF16 || a.dtype == kBF16 || (a.dtype == kF32 && a.head_dim == 64);
  const bool hd = a.head_dim == 64 || a.head_dim == 128;
  return dt && hd && a.bits >= 3 && a.bits <= 5 && a.num_kv_heads >= 1;
}

cudaError_t launch_write_prod_tc(const WriteArgs& a, const float* smat, cudaStream_t stream, int grid) {
  WriteTcArgs t;
  t.a = a;
  t.smat = smat;
#define TQ_WTP(T, D, MB)                                                                                      \
  if (a.head_dim == D && a.bits == MB + 1) {                                                                  \
    const size_t smem = write_tc_fixed_smem<D, true>() + kWWarps * (2 * 16 * D * sizeof(T));                   \
    auto kern = write_tc_kernel<T, D, MB, true>;                                                              \
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
    if (err != cudaSuccess) return err;                                                                       \
    return launch_dependent(kern, grid, smem, stream, t);                                                     \
  }
  if (a.dtype == kF32) {
    TQ_WTP(float, 64, 2) TQ_WTP(float, 64, 3) TQ_WTP(float, 64, 4)
  } else if (a.dtype == kF16) {
    TQ_WTP(__half, 64, 2) TQ_WTP(__half, 64, 3) TQ_WTP(__half, 64, 4)
    TQ_WTP(__half, 128, 2) TQ_WTP(__half, 128, 3) TQ_WTP(__half, 128, 4)
  } else if (a.dtype == kBF16) {
    TQ_WTP(__nv_bfloat16, 64, 2) TQ_WTP(__nv_bfloat16, 64, 3) TQ_WTP(__nv_bfloat16, 64, 4)
    TQ_WTP(__nv_bfloat16, 128, 2) TQ_WTP(__nv_bfloat16, 128, 3) TQ_WTP(__nv_bfloat16, 128, 4)
  }
#undef TQ_WTP
  return cudaErrorInvalidValue;
}

}  // namespace tq
