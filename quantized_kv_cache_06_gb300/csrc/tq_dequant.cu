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
// 4-bit rows at D 64 / 128 take the tensor-core form below instead (dequant_tc_kernel).
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

// ---- tensor-core readback: 4-bit rows at D 64 / 128 ------------------------------------
// A warp takes 16-row tiles (rows in [token][head] order).  The tile's packed rows are
// brought into shared memory by 4-byte cp.async copies (rows of RBW_P words: 16-byte aligned,
// and an odd number of 16-byte chunks apart, so the 8 rows of a 128-bit load fall into
// different banks), two tiles in flight.  Block j of the inverse rotation is an m16n8k16
// MMA: A = the centroids of coordinates 16 j .. 16 j + 15 of the 16 rows, looked up per
// index byte (two coordinates) as (fp16 hi pair, fp16 lo pair x 2^12) from a table with 16
// lane copies; B = the +-1 matrix H_16 for the hi parts and +-2^-12 H_16 for the lo parts, so
// both products are exact and sum into one fp32 accumulator.  Butterflies across blocks
// finish H_D; then x s_d / sqrt(D) x nu per row, converted and stored.
namespace dtc {
constexpr int kWarps = 8;
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void wait_groups() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// fp16 pair of +-m (m = 1.0 as 0x3C00, 2^-12 as 0x0C00), negative where the flag is set
__device__ __forceinline__ uint32_t pm_pair(uint32_t m, bool neg0, bool neg1) {
  return (m | (neg0 ? 0x8000u : 0u)) | ((m | (neg1 ? 0x8000u : 0u)) << 16);
}
// two consecutive outputs (the address is a multiple of 2 elements)
__device__ __forceinline__ void store_pair(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void store_pair(__half* p, float2 v) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(v.x, v.y);
}
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}
template <int D>
struct Shape {
  static constexpr int RB = D / 2 + 4;         // row bytes at 4 bits
  static constexpr int RBW = RB / 4;           // row words
  static constexpr int P = (RBW + 3) / 4;      // 16-byte chunks a row needs
  static constexpr int RBW_P = 4 * ((P % 2) ? P : P + 1);  // padded row stride (words)
  static constexpr int TILE_W = 16 * RBW_P;    // words of a tile buffer
  static constexpr int kTable = 256 * 16 * 8;  // 16 copies of 256 (hi pair, lo pair) entries
  // 16-bit outputs: a staged output tile per warp, rows of 2 D + 16 bytes (the 4-byte writes
  // of 8 rows x 4 lanes and the 16-byte reads of a row fall into different banks)
  static constexpr int OUT_ROW = 2 * D + 16;
  static constexpr int kOutTile = 16 * OUT_ROW;
  static constexpr int kBytes = kTable + D * 4 + kWarps * 2 * TILE_W * 4 + kWarps * kOutTile;
};
}  // namespace dtc

template <typename T, int D>
__global__ void __launch_bounds__(dtc::kWarps * 32, 2) dequant_tc_kernel(DequantArgs a) {
  using S = dtc::Shape<D>;
  constexpr int NB = D / 16, RBW = S::RBW, RBW_P = S::RBW_P;
  constexpr int NW = D / 8;   // index words of a row (4 bits); the norm is word NW
  extern __shared__ __align__(16) unsigned char dsm[];
  uint2* table = reinterpret_cast<uint2*>(dsm);                  // entry b, copy k at b * 16 + k
  float* sgn_s = reinterpret_cast<float*>(dsm + S::kTable);     // s_d / sqrt(D)
  uint32_t* tiles = reinterpret_cast<uint32_t*>(dsm + S::kTable + D * 4);
  unsigned char* out_stage = dsm + S::kTable + D * 4 + dtc::kWarps * 2 * S::TILE_W * 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int H = a.num_kv_heads;
  const int64_t capacity = a.num_blocks * (int64_t)a.block_size;
  const int64_t num_rows = a.num_tokens * H;
  const int64_t num_tiles = (num_rows + 15) / 16;

  // table: entry b = (hi(c[b & 15]), hi(c[b >> 4])), ((c[b & 15] - hi) 2^12, (c[b >> 4] - hi) 2^12)
  for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
    const int b = i >> 4;
    const float c0 = __ldg(a.centroids + (b & 15)), c1 = __ldg(a.centroids + (b >> 4));
    const __half h0 = __float2half_rn(c0), h1 = __float2half_rn(c1);
    const __half l0 = __float2half_rn((c0 - __half2float(h0)) * 4096.0f);
    const __half l1 = __float2half_rn((c1 - __half2float(h1)) * 4096.0f);
    uint2 e;
    e.x = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
    e.y = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    table[i] = e;
  }
  const float rsd = 1.0f / sqrtf((float)D);
  for (int i = threadIdx.x; i < D; i += blockDim.x) sgn_s[i] = __ldg(a.signs + i) * rsd;
  __syncthreads();

  // B fragments of H_16 (hi: +-1, lo: +-2^-12): this lane holds k = 2c, 2c + 1 (part 0) and
  // 2c + 8, 2c + 9 (part 1) for n = g (n-tile 0) and g + 8 (n-tile 1)
  uint32_t bh[2][2], bl[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int n = g + 8 * nt, k0 = 2 * c + 8 * part;
      const bool n0 = __popc(k0 & n) & 1, n1 = __popc((k0 + 1) & n) & 1;
      bh[nt][part] = dtc::pm_pair(0x3C00u, n0, n1);
      bl[nt][part] = dtc::pm_pair(0x0C00u, n0, n1);
    }
  const uint32_t table_lane = dtc::smem_u32(table) + (uint32_t)((lane & 15) * 8);
  uint32_t* my_tiles = tiles + warp * 2 * S::TILE_W;
  T* out = static_cast<T*>(a.out);

  // Issue the copies of tile `tile` into buffer `buf`: lanes 2r and 2r + 1 copy row r (words
  // of their parity); rows past the end or with a negative / out-of-range slot are zero-filled.
  const bool rows32 = num_rows < (int64_t)1 << 31;  // row -> token with a 32-bit division
  const int lrow = lane >> 1, lpar = lane & 1;
  auto load_tile = [&](int64_t tile, int buf) {
    if (tile < num_tiles) {
      const int64_t row = tile * 16 + lrow;
      int64_t base = -1;  // byte offset of the row in the pages
      if (row < num_rows) {
        const int64_t t = rows32 ? (int64_t)((uint32_t)row / (uint32_t)H) : row / H;
        const int h = (int)(row - t * H);
        const int64_t slot = __ldg(a.slots + t);
        if (slot >= capacity) {
          if (h == 0 && lpar == 0 && a.status) atomicMax(a.status, (int32_t)kSlotOutOfRange);
        } else if (slot >= 0) {
          base = (slot * H + h) * (int64_t)S::RB;
        }
      }
      const bool ok = base >= 0;
      const unsigned char* src = a.pages + (ok ? base : 0) + 4 * lpar;
      const int n = ok ? 4 : 0;
      const uint32_t dst = dtc::smem_u32(my_tiles + buf * S::TILE_W + lrow * RBW_P + lpar);
#pragma unroll
      for (int k = 0; k < (RBW + 1) / 2; ++k)  // words lpar + 2k
        if (lpar + 2 * k < RBW) dtc::cp4(dst + 8 * k, src + 8 * k, n);
    }
    dtc::commit();
  };

  const int64_t wstride = (int64_t)gridDim.x * dtc::kWarps;
  int64_t tile = (int64_t)blockIdx.x * dtc::kWarps + warp;
  int buf = 0;
  load_tile(tile, 0);
  for (; tile < num_tiles; tile += wstride, buf ^= 1) {
    load_tile(tile + wstride, buf ^ 1);
    dtc::wait_groups<1>();
    __syncwarp();
    const uint32_t* tb = my_tiles + buf * S::TILE_W;
    const float nu_g = __uint_as_float(tb[g * RBW_P + NW]), nu_h = __uint_as_float(tb[(g + 8) * RBW_P + NW]);
    float acc[NB][2][4];
    // byte c of index word w of a row: its two coordinates' (hi pair, lo pair)
    auto look = [&](uint32_t w) -> uint2 {
      const uint32_t b = __byte_perm(w, 0u, 0x4440u + (uint32_t)c);
      uint2 e;
      asm("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(e.x), "=r"(e.y) : "r"(table_lane + (b << 7)));
      return e;
    };
#pragma unroll
    for (int q = 0; q < NW / 4; ++q) {
      // index words 4q .. 4q + 3 of rows g and g + 8: blocks 2q (words 4q, 4q + 1) and 2q + 1
      const uint4 x = *reinterpret_cast<const uint4*>(tb + g * RBW_P + 4 * q);
      const uint4 y = *reinterpret_cast<const uint4*>(tb + (g + 8) * RBW_P + 4 * q);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int j = 2 * q + half;
        // byte 8 j + c (word 2 j) and 8 j + 4 + c (word 2 j + 1) of rows g and g + 8
        const uint2 e0 = look(half ? x.z : x.x), e1 = look(half ? y.z : y.x);
        const uint2 e2 = look(half ? x.w : x.y), e3 = look(half ? y.w : y.y);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int xx = 0; xx < 4; ++xx) acc[j][nt][xx] = 0.f;
          dtc::mma(acc[j][nt], e0.x, e1.x, e2.x, e3.x, bh[nt][0], bh[nt][1]);
          dtc::mma(acc[j][nt], e0.y, e1.y, e2.y, e3.y, bl[nt][0], bl[nt][1]);
        }
      }
    }
    __syncwarp();  // every lane has read the tile buffer: it may be refilled
    const float2 minus1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int hs = 1; hs < NB; hs <<= 1)
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if ((j & hs) == 0) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int x = 0; x < 4; x += 2) {
              const float2 p = make_float2(acc[j][nt][x], acc[j][nt][x + 1]);
              const float2 q = make_float2(acc[j + hs][nt][x], acc[j + hs][nt][x + 1]);
              const float2 sm = __fadd2_rn(p, q), df = __ffma2_rn(q, minus1, p);
              acc[j][nt][x] = sm.x;
              acc[j][nt][x + 1] = sm.y;
              acc[j + hs][nt][x] = df.x;
              acc[j + hs][nt][x + 1] = df.y;
            }
        }
    // columns 16 j + 8 nt + 2c, +1 of rows g (x = 0, 1) and g + 8 (x = 2, 3)
    const int64_t row_g = tile * 16 + g, row_h = row_g + 8;
    const float2 ng = make_float2(nu_g, nu_g), nh = make_float2(nu_h, nu_h);
    unsigned char* ost = out_stage + warp * S::kOutTile;
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = 16 * j + 8 * nt + 2 * c;
        const float2 sv = *reinterpret_cast<const float2*>(sgn_s + col);
        const float2 vg = __fmul2_rn(__fmul2_rn(make_float2(acc[j][nt][0], acc[j][nt][1]), sv), ng);
        const float2 vh = __fmul2_rn(__fmul2_rn(make_float2(acc[j][nt][2], acc[j][nt][3]), sv), nh);
        if constexpr (sizeof(T) == 4) {  // fp32: 8-byte stores, whole 32-byte sectors per row
          if (row_g < num_rows) dtc::store_pair(out + row_g * D + col, vg);
          if (row_h < num_rows) dtc::store_pair(out + row_h * D + col, vh);
        } else {
          dtc::store_pair(reinterpret_cast<T*>(ost + g * S::OUT_ROW) + col, vg);
          dtc::store_pair(reinterpret_cast<T*>(ost + (g + 8) * S::OUT_ROW) + col, vh);
        }
      }
    if constexpr (sizeof(T) == 2) {
      // the staged tile as 16-byte chunks: a row is D / 8 chunks, lane i takes chunks i, i + 32, ..
      __syncwarp();
      constexpr int CPR = D / 8, CH = 16 * CPR;
#pragma unroll
      for (int k = 0; k < CH / 32; ++k) {
        const int i = lane + 32 * k, r = i / CPR, ch = i - r * CPR;
        const int64_t row = tile * 16 + r;
        const uint4 v = *reinterpret_cast<const uint4*>(ost + r * S::OUT_ROW + ch * 16);
        if (row < num_rows) *reinterpret_cast<uint4*>(out + row * D + ch * 8) = v;
      }
      __syncwarp();  // the next tile rewrites the staged rows
    }
  }
  dtc::wait_groups<0>();
}

template <typename T, int D>
cudaError_t launch_dequant_tc(const DequantArgs& a, cudaStream_t stream, int num_sms) {
  using S = dtc::Shape<D>;
  auto kern = dequant_tc_kernel<T, D>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  if (err != cudaSuccess) return err;
  const int64_t tiles = (a.num_tokens * a.num_kv_heads + 15) / 16;
  const int64_t ctas = (tiles + dtc::kWarps - 1) / dtc::kWarps;
  const int grid = (int)(ctas < (int64_t)num_sms * 2 ? ctas : (int64_t)num_sms * 2);
  kern<<<grid, dtc::kWarps * 32, S::kBytes, stream>>>(a);
  err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

template <typename T>
cudaError_t launch_dequant_tc_dim(const DequantArgs& a, cudaStream_t stream, int num_sms) {
  if (a.head_dim == 64) return launch_dequant_tc<T, 64>(a, stream, num_sms);
  return launch_dequant_tc<T, 128>(a, stream, num_sms);
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
  if (a.bits == 4 && (a.head_dim == 64 || a.head_dim == 128)) {  // the tensor-core form
    if (a.out_dtype == kF16) return launch_dequant_tc_dim<__half>(a, stream, num_sms);
    if (a.out_dtype == kBF16) return launch_dequant_tc_dim<__nv_bfloat16>(a, stream, num_sms);
    return launch_dequant_tc_dim<float>(a, stream, num_sms);
  }
  const int64_t rows_per_warp = 32 / (a.head_dim / 32);
  const int64_t warps_wanted = (a.num_tokens * a.num_kv_heads + rows_per_warp - 1) / rows_per_warp;
  const int64_t blocks = (warps_wanted + 7) / 8;
  const int grid = (int)(blocks < (int64_t)num_sms * 8 ? blocks : (int64_t)num_sms * 8);
  if (a.out_dtype == kF16) return launch_dim<__half>(a, stream, grid);
  if (a.out_dtype == kBF16) return launch_dim<__nv_bfloat16>(a, stream, grid);
  return launch_dim<float>(a, stream, grid);
}

}  // namespace tq
