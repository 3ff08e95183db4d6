// Multi-query mixed prefill/decode attention over packed TurboQuant pages (sm_103a,
// mma.sync f16 -> f32).
//
// TurboQuant docs: "vLLM Usage" (Runtime Dispatch: the cache plus mixed prefill/decode
// reads the packed cache) and "Architecture" (Diagnostic vs Serving Paths: keys consumed
// compressed, values accumulated from packed indices).  Query row i is one token of
// sequence q_seq[i] that attends to the first q_len[i] tokens of that sequence.
//
// Rows of one prefill chunk read the same cache blocks.  This kernel dequantises every
// 32-token tile of one kv head ONCE into shared memory (fp16, rotated space) and runs it
// against up to 64 (query row, q head) pairs with tensor-core MMAs:
//   S  = qrot Khat^T          m16n8k16, A = rotated queries, B = key tile (ldmatrix)
//   causal mask per row (token < q_len), online softmax in base 2
//   O += P' Vhat               A = P' = p * nu_v (from the S accumulators), B = value tile
//                              (ldmatrix.trans).  A tile whose largest value norm passes
//                              kMqFastValueNorm scales each row's P' by a power of two that
//                              puts its largest near 2^12 (O scaled by it before the tile and
//                              back after, both exact) and adds the fp16 remainders of P'
//                              and of the value tile; it also takes the exact key path.
// Khat holds fp16(alpha_k c[idx]) (+ the fp16 remainder for tiles that need the exact
// score), Vhat fp16(alpha_v c[idx]); the key norm multiplies the score and the value norm
// the weight, so nothing of the cache is expanded to a dense row in HBM.  The rotated
// query is split into fp16 hi + lo, and the score is hi*Khat + lo*Khat (+ hi*Klo when
// nu_k * ||q|| can exceed kMqFastBound), which keeps it at fp32-level accuracy.
//
// Work split.  CTA (window, split, kv head): a window is up to 64 / G consecutive query
// rows (64 rows of the MMA: 4 warps x 16), a split a range of split_len tokens of the
// sequence.  tq_paged_prefill takes full windows; tq_paged_decode takes one-row windows
// for the D 64/128 shapes its tensor-core kernel does not cover (3/5-bit rows, block
// sizes other than 16, GQA groups 1 and 2).  D = 256 runs 8 warps: two per row group,
// each with half of the dimensions (query fragments, score k-steps, value n-tiles); the
// half scores are summed through shared memory between the pair's two warps.  Rows of a window that belong to different sequences form segments, taken one
// after the other (each streams its own sequence; rows outside the segment are masked).
// The CTA writes one (m, l, acc[D]) partial per (row, q head, split); the split combine
// (shared with the SIMT decode) merges them and applies R^T.
//
// Per tile: every thread copies the packed words it will dequantise with cp.async into
// its own slots of a 4-stage ring, three tiles ahead.  For tile it: wait for its own
// copies -> barrier A (which also votes whether the tile needs the exact key part) ->
// dequantise into shared memory -> start the copies of tile it + 3 -> barrier B -> MMAs.
// One tile buffer: barrier A orders its reuse after every warp's math.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kMqGroups = 4;             // 16-row MMA groups per CTA
constexpr int kMqRows = 16 * kMqGroups;  // MMA rows (query row x q head) per CTA
constexpr int kMqTile = 32;             // tokens per tile
constexpr float kMqLog2e = 1.4426950408889634f;
// Largest bound nu_k * ||q_rot|| (log2 units) of a tile scored without the fp16
// remainder of the key centroids (same bound as the tensor-core decode).
constexpr float kMqFastBound = 48.0f;
constexpr float kMqSlack = 6.0f;  // log2 units the running max may lag behind the scores
// Largest value norm of a tile whose values take the fp16 path (P' = p nu_v <= 2^6 * 32,
// rounded once to fp16, and the fp16 value tile); tiles above it scale P', add both fp16
// remainders and take the exact key path (same rule as the tensor-core decode: an error
// proportional to a large norm can pass the absolute part of the 2e-3 + 2e-3 |o|
// tolerance where the output element is small).
constexpr float kMqFastValueNorm = 32.0f;
// The fp16 remainders of the key and value tiles are stored times 2^12: a remainder of a
// value below 1/4 would otherwise be an fp16 subnormal (2^-25 of absolute precision); the
// products with them are scaled back by 2^-12, exactly.
constexpr float kMqLoScale = 4096.0f;
constexpr float kMqLoUnscale = 1.0f / 4096;

constexpr int kMqStages = 4;  // raw-word ring: tiles it .. it + 2 in flight while tile it is used

// Warps per CTA.  D <= 128: one warp per 16-row group.  D = 256: two warps per group,
// each holding the query, the score contraction and the value accumulators of one half of
// the dimensions; the two half scores are summed through shared memory.
template <int D>
struct MqShape {
  static constexpr bool kSplit = D == 256;
  static constexpr int kWarps = kSplit ? 2 * kMqGroups : kMqGroups;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kDh = kSplit ? D / 2 : D;  // dimensions per warp
  static constexpr int kMinBlocks = kSplit ? 1 : 3;
};

template <int D, int KB, int VB>
struct MqSmem {
  static constexpr int kRow = 2 * D;                  // bytes per fp16 row
  static constexpr int kTileBytes = kMqTile * kRow;
  static constexpr int kOffKhi = 0;                   // [32 tokens][D], swizzled
  static constexpr int kOffKlo = kOffKhi + kTileBytes;
  static constexpr int kOffV = kOffKlo + kTileBytes;
  static constexpr int kOffQlo = kOffV + kTileBytes;  // [group][16 rows][D], swizzled
  static constexpr int kOffKn = kOffQlo + kMqGroups * 16 * kRow;  // float[32] key norms
  static constexpr int kOffVn = kOffKn + kMqTile * 4;            // float[32] value norms
  static constexpr int kOffKadd = kOffVn + kMqTile * 4;          // float[32] 0 / -inf per token
  static constexpr int kOffSeq = kOffKadd + kMqTile * 4;         // int[64] table row per window row
  static constexpr int kOffLen = kOffSeq + kMqRows * 4;          // int[64] clamped length
  static constexpr int kOffQn = kOffLen + kMqRows * 4;           // float[warps] max ||q_rot||
  // Raw-word ring, private to each thread: per stage and thread, for each of its
  // dequantisation tasks the index words, the norm, and an "in range" flag; stored
  // word-major ([stage][word][thread]) so a warp's accesses are conflict free.
  static constexpr int kThreads = MqShape<D>::kThreads;
  static constexpr int kTasks = (2 * kMqTile * (D / 32)) / kThreads;  // tasks per thread
  static constexpr int kMaxBits = KB > VB ? KB : VB;
  static constexpr int kTaskWords = kMaxBits + 2;                       // words, norm, flag
  static constexpr int kRingWords = kTasks * kTaskWords;                // per thread per stage
  static constexpr int kOffRing = (kOffQn + MqShape<D>::kWarps * 4 + 15) / 16 * 16;
  // D = 256: per warp and lane the 16 half-score partials exchanged with the partner warp
  static constexpr int kOffX = kOffRing + kMqStages * kRingWords * kThreads * 4;
  static constexpr int kBytes = kOffX + (MqShape<D>::kSplit ? MqShape<D>::kWarps * 32 * 16 * 4 : 0);
  static constexpr int kAlloc = kBytes + 1024;  // + the pad that aligns the base to 1024 bytes
  // the query hi parts are staged in the key tiles before the first tile
  static_assert(2 * kTileBytes == kMqGroups * 16 * kRow, "query staging must fit the key tiles");
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a [rows][D] fp16 tile: the chunk
// index is XORed with row % 8, so the 8 rows of an ldmatrix hit 8 different bank groups.
// Region bases are multiples of 1024 bytes and rows are 2D bytes, so the chunk bits
// (4 .. 3 + log2(D / 8)) of a row's address are free: for a compile-time step k,
// swz(row, c ^ k) = swz(row, c) ^ (k << 4), one LOP3 per address.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (2 * D) + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// D = A * B + D, m16n8k16, A row-major f16, B col-major f16, f32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {  // 2^x, hardware approximation (ex2(-inf) = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// Power-of-two scale (and its inverse) that brings a positive x to [2^11, 2^12): both exact;
// 1 and 1 for x = 0 or subnormal.
__device__ __forceinline__ void mq_tile_scale(float x, float& f, float& inv_f) {
  int e = (int)((__float_as_uint(x) >> 23) & 0xffu);
  if (e == 0) {
    f = inv_f = 1.f;
    return;
  }
  e = max(12, e);
  f = __uint_as_float((uint32_t)(265 - e) << 23);   // 2^(138 - e)
  inv_f = __uint_as_float((uint32_t)(e - 11) << 23);  // 2^(e - 138)
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void bar_pair(int id) {  // the two warps of one row group
  asm volatile("bar.sync %0, 64;\n" ::"r"(id) : "memory");
}
__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}

// The value remainders of one tile (an exact-value tile, rare): this thread's value tasks
// re-read from its ring words and expanded into the key tile's space (fp16 (alpha c - hi)
// times 2^12), between barrier C (every warp's scores done) and barrier D.  Not inlined, so
// the registers of this path do not weigh on the main loop's.
template <int VB, int MAXB, int TPT, int kTaskWords, int kMaxBits, int kThreads, int kRingWords>
__device__ __noinline__ void mq_value_remainders(uint32_t ring_base, int tid, int st, const int* comps,
                                                 const uint32_t* sts_offs, uint32_t khi_base, uint32_t vc_pair) {
  __syncthreads();  // C
#pragma unroll
  for (int j = 0; j < TPT; ++j) {
    if (comps[j] != 1) continue;
    auto ring = [&](int w) -> uint32_t {
      return ring_base + (uint32_t)(((st * kRingWords + j * kTaskWords + w) * kThreads + tid) * 4);
    };
    const bool ok = lds_u32(ring(kMaxBits + 1)) != 0u;
    uint32_t w[MAXB];
#pragma unroll
    for (int k = 0; k < MAXB; ++k) w[k] = ok ? lds_u32(ring(k)) : 0u;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t vp[4];
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        uint32_t val[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = q4 * 8 + pr * 2 + u;
          const int bit = i * VB, k = bit >> 5, sh = bit & 31;
          uint32_t f = w[k] >> sh;
          if (sh + VB > 32) f |= w[k + 1] << (32 - sh);
          val[u] = __shfl_sync(kFullMask, vc_pair, (int)f);
        }
        vp[pr] = __byte_perm(val[0], val[1], 0x7632);
      }
      sts_v4(khi_base + (sts_offs[j] ^ (uint32_t)(q4 << 4)), vp[0], vp[1], vp[2], vp[3]);
    }
  }
  __syncthreads();  // D
}

struct MqArgs {
  DecodeArgs a;
  int nsplit;     // token splits per sequence
  int split_len;  // tokens per split (multiple of 32)
  int bs_shift;   // log2(block_size) when it is a power of two, else -1
  int windows;    // ceil(rows / rows_per_window)
  int rows_per_window;  // query rows per CTA, 1 .. 64 / G (1: a decode batch, one row per sequence)
  float* part_acc;  // [rows * Hq][nsplit][D]
  float* part_ml;   // [rows * Hq][nsplit][2]
};

// Raw index words of one dequantisation task: 32 consecutive coordinates (BITS whole
// words) of one token's row, its norm, and whether the token is read at all.
template <int BITS>
struct RawTask {
  uint32_t w[BITS];
  uint32_t nrm;
  bool ok;
};

template <int D, int KB, int VB, int G>
__global__ void __launch_bounds__(MqShape<D>::kThreads, MqShape<D>::kMinBlocks) prefill_mq_kernel(MqArgs args) {
  using S = MqSmem<D, KB, VB>;
  using SH = MqShape<D>;
  constexpr int kThreads = SH::kThreads;
  constexpr bool SPLIT = SH::kSplit;
  constexpr int P = D / 32;                  // 32-coordinate parts per row
  constexpr int E = D / 32;                  // query coordinates per lane
  constexpr int KS = SH::kDh / 16;           // score k-steps of this warp
  constexpr int NT = SH::kDh / 8;            // value n-tiles of this warp
  constexpr int MQ = kMqRows / G;            // query rows per window
  constexpr int TASKS = 2 * kMqTile * P;     // K and V tasks of one tile
  constexpr int TPT = TASKS / kThreads;      // tasks per thread
  constexpr int MAXB = KB > VB ? KB : VB;
  static_assert(TPT == 1 || TPT == 2, "one or two dequantisation tasks per thread");
  static_assert(TPT == S::kTasks, "task count");
  static_assert(TPT == 2 || kThreads == 2 * kMqTile * P, "one K and one V task set");
  static_assert(kMqRows % G == 0, "group must divide the rows of a CTA");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  // region offsets assume a 256-byte aligned base (the XOR addressing needs bits 4..7 free)
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const DecodeArgs& a = args.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = warp % kMqGroups;  // this warp's 16 MMA rows: group grp
  const int dh = warp / kMqGroups;   // and dimensions [dh Dh, dh Dh + Dh) (D = 256), else 0
  const int H = a.num_kv_heads, Hq = a.num_q_heads;
  const int h = blockIdx.x % H;
  const int split = (blockIdx.x / H) % args.nsplit;
  const int window = blockIdx.x / (H * args.nsplit);
  const int i0 = window * args.rows_per_window;
  const int nrows = min(args.rows_per_window, a.batch - i0);
  const int bs = a.block_size;
  const int cap = a.max_blocks_per_seq * bs;
  const uint32_t sbase = smem_addr(smem);
  int* row_seq = reinterpret_cast<int*>(smem + S::kOffSeq);
  int* row_len = reinterpret_cast<int*>(smem + S::kOffLen);
  float* kn_s = reinterpret_cast<float*>(smem + S::kOffKn);
  float* vn_s = reinterpret_cast<float*>(smem + S::kOffVn);
  float* kadd_s = reinterpret_cast<float*>(smem + S::kOffKadd);
  float* qn_s = reinterpret_cast<float*>(smem + S::kOffQn);

  // ---- window rows: table row and clamped length -------------------------------------
  if (tid < MQ) {
    int seq = -1, len = 0;
    if (tid < nrows) {
      seq = block_table_row(a, i0 + tid);
      len = __ldg(a.seq_lens + i0 + tid);
      const bool bad = seq < 0 || len < 0 || len > cap;
      if (bad && split == 0 && h == 0 && a.status) atomicMax(a.status, (int32_t)kInvalidArg);
      len = len < 0 ? 0 : (len > cap ? cap : len);
    }
    row_seq[tid] = seq;
    row_len[tid] = len;
  }

  // ---- rotated queries of this warp's 16 MMA rows -> hi (registers) and lo (smem) ------
  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kMqLog2e / sqrtf((float)D);
  const float inv_alpha_k = 1.0f / a.k_alpha;
  const uint32_t qhi_base = sbase + S::kOffKhi + grp * 16 * S::kRow;  // staging in the key tiles
  const uint32_t qlo_base = sbase + S::kOffQlo + grp * 16 * S::kRow;
  float qn = 0.f;
  for (int m = 0; m < 16; ++m) {
    const int mr = grp * 16 + m;
    const int wrow = mr / G;
    float v[E];
    if (wrow < nrows) {
      const int64_t qr = (int64_t)(i0 + wrow) * Hq + (int64_t)h * G + mr % G;  // (row, q head)
      const int64_t base = qr * D + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        v[i] = load_query_f32(a.q, a.q_scale, qr, base + i, a.q_dtype) * __ldg(a.signs + lane * E + i);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) v[i] = 0.f;
    }
    fwht_warp<E>(v);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      v[i] *= qmul;
      ss = fmaf(v[i], v[i], ss);
      v[i] *= inv_alpha_k;  // the key tile holds alpha_k * c
    }
    qn = fmaxf(qn, sqrtf(warp_sum(ss)));
    uint32_t hi[E / 2], lo[E / 2];
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      const __half h0 = __float2half_rn(v[2 * i]), h1 = __float2half_rn(v[2 * i + 1]);
      hi[i] = half2_bits(__half2float(h0), __half2float(h1));
      lo[i] = half2_bits(v[2 * i] - __half2float(h0), v[2 * i + 1] - __half2float(h1));
    }
    // lane owns coordinates [lane E, lane E + E): chunk lane E / 8, byte offset (lane E % 8) * 2
    const uint32_t off = swz<D>(m, (lane * E) >> 3) + (uint32_t)(((lane * E) & 7) * 2);
    unsigned char* ph = smem + (qhi_base - sbase) + off;
    unsigned char* pl = smem + (qlo_base - sbase) + off;
    if (dh != 0) continue;  // D = 256: the group's first warp writes the staging
    if constexpr (E == 8) {
      *reinterpret_cast<uint4*>(ph) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(pl) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else if constexpr (E == 4) {
      *reinterpret_cast<uint2*>(ph) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(pl) = make_uint2(lo[0], lo[1]);
    } else {
      *reinterpret_cast<uint32_t*>(ph) = hi[0];
      *reinterpret_cast<uint32_t*>(pl) = lo[0];
    }
  }
  if (lane == 0) qn_s[warp] = qn;
  __syncthreads();  // row metadata, query norms and query staging visible
  const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: this lane addresses row rr of matrix mi
  // A fragments (16 rows x 16 k): matrix mi = rows (mi & 1) * 8.., k chunk 2 ks + (mi >> 1);
  // this warp's k-steps are dh KS .. dh KS + KS - 1
  const uint32_t qa_lane = swz<D>((mi & 1) * 8 + rr, mi >> 1);
  uint32_t qh[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) ldsm_x4(qh[ks], (qhi_base + qa_lane) ^ (uint32_t)((dh * KS + ks) << 5));
  float qn_cta = 0.f;
#pragma unroll
  for (int w = 0; w < SH::kWarps; ++w) qn_cta = fmaxf(qn_cta, qn_s[w]);

  // ---- per-lane softmax state: rows r and r + 8 of this warp's 16 --------------------
  const int r = lane >> 2, c = lane & 3;
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float m_thr[2] = {-INFINITY, -INFINITY};  // m_run + kMqSlack

  // dequantisation centroids: lane l holds entry l mod 2^b (a shuffle reads only the low
  // 5 bits of its source lane, so a field needs no mask)
  uint32_t kc_pair, vc_pair;  // (fp16 hi, fp16 lo * 2^12) of alpha c
  {
    const float ck = __ldg(a.k_centroids + (lane & ((1 << KB) - 1))) * a.k_alpha;
    const __half hk = __float2half_rn(ck);
    const __half lk = __float2half_rn((ck - __half2float(hk)) * kMqLoScale);
    kc_pair = (uint32_t)__half_as_ushort(hk) | ((uint32_t)__half_as_ushort(lk) << 16);
    const float cv = __ldg(a.v_centroids + (lane & ((1 << VB) - 1))) * a.v_alpha;
    const __half hv = __float2half_rn(cv);
    const __half lv = __float2half_rn((cv - __half2float(hv)) * kMqLoScale);
    vc_pair = (uint32_t)__half_as_ushort(hv) | ((uint32_t)__half_as_ushort(lv) << 16);
  }

  // task j of this thread: component (0 K, 1 V), token t of the tile, part (32
  // coordinates).  D = 128 / 256: task 0 is K and task 1 is V of (t, part) =
  // (tid / P, tid % P); D = 64: warps 0-1 take K tasks and warps 2-3 V tasks (warp-uniform).
  auto task_comp = [&](int j) -> int { return TPT == 2 ? j : (tid >= kMqTile * P ? 1 : 0); };
  auto task_rem = [&](int j) -> int { return TPT == 2 ? tid : tid % (kMqTile * P); };
  auto task_tok = [&](int j) -> int { return task_rem(j) / P; };
  auto task_part = [&](int j) -> int { return task_rem(j) % P; };

  const uint32_t khi_base = sbase + S::kOffKhi, klo_base = sbase + S::kOffKlo, v_base = sbase + S::kOffV;
  // ldmatrix lane addresses at k-step / value-tile 0 (the steps are XORed in):
  // key B fragments: matrix mi = tokens (mi >> 1) * 8.., k chunk 2 ks + (mi & 1);
  // value B fragments (transposed): tokens (mi & 1) * 8.., value chunk 2 dp + (mi >> 1)
  const uint32_t kb_lane = khi_base + swz<D>((mi >> 1) * 8 + rr, mi & 1);
  const uint32_t vb_lane = v_base + swz<D>((mi & 1) * 8 + rr, mi >> 1);
  const uint32_t ql_lane = qlo_base + qa_lane;
  // dequantisation stores of task j: chunk part * 4 + q4 of token row t -> base ^ (q4 << 4)
  uint32_t sts_off[TPT];
#pragma unroll
  for (int j = 0; j < TPT; ++j) sts_off[j] = swz<D>(task_tok(j), task_part(j) * 4);
  const int bs_shift = args.bs_shift;
  auto blk_of = [&](int T) -> int { return bs_shift >= 0 ? (T >> bs_shift) : T / bs; };
  auto off_of = [&](int T) -> int { return bs_shift >= 0 ? (T & (bs - 1)) : T % bs; };

  // ---- segments: runs of window rows with one table row ------------------------------
  int s0 = 0;
  while (s0 < nrows) {
    const int seq = row_seq[s0];
    int s1 = s0 + 1;
    while (s1 < nrows && row_seq[s1] == seq) ++s1;
    int seg_len = 0;
    for (int k = s0; k < s1; ++k) seg_len = max(seg_len, row_len[k]);
    const int t_beg = split * args.split_len;
    const int t_end = min(seg_len, t_beg + args.split_len);
    if (seq >= 0 && t_beg < t_end) {
      const int32_t* bt = a.block_table + (int64_t)seq * a.max_blocks_per_seq;
      // lengths of this lane's two rows (0 outside the segment)
      const int wA = (grp * 16 + r) / G, wB = (grp * 16 + r + 8) / G;
      const int lenA = (wA >= s0 && wA < s1) ? row_len[wA] : 0;
      const int lenB = (wB >= s0 && wB < s1) ? row_len[wB] : 0;
      const int ntiles = (t_end - t_beg + kMqTile - 1) / kMqTile;

      auto load_bid = [&](int tile, int j) -> int {
        const int T = t_beg + tile * kMqTile + task_tok(j);
        return (tile < ntiles && T < t_end) ? __ldg(bt + blk_of(T)) : -1;
      };
      // ring word w of this thread in stage st
      auto ring = [&](int st, int w) -> uint32_t {
        return sbase + S::kOffRing + (uint32_t)(((st * S::kRingWords + w) * kThreads + tid) * 4);
      };
      // Starts the copies of task j of `tile` (block `bid`) into ring stage tile % kMqStages.
      auto issue_task = [&](auto bits_tag, int tile, int j, int bid) {
        constexpr int BITS = decltype(bits_tag)::value;
        constexpr int RB = D * BITS / 8 + 4;
        const int st = tile % kMqStages;
        const int T = t_beg + tile * kMqTile + task_tok(j);
        const bool in = tile < ntiles && T < t_end;
        const bool okb = bid >= 0 && (int64_t)bid < a.num_blocks;
        if (in && !okb && a.status) atomicMax(a.status, (int32_t)kBlockOutOfRange);
        const bool ok = in && okb;
        sts_u32(ring(st, j * S::kTaskWords + S::kMaxBits + 1), ok ? 1u : 0u);
        if (ok) {
          const uint8_t* pages = task_comp(j) == 0 ? a.k_pages : a.v_pages;
          const uint32_t* row =
              reinterpret_cast<const uint32_t*>(pages + (((int64_t)bid * bs + off_of(T)) * H + h) * RB);
#pragma unroll
          for (int k = 0; k < BITS; ++k) cp_async4(ring(st, j * S::kTaskWords + k), row + task_part(j) * BITS + k);
          if (task_part(j) == 0) cp_async4(ring(st, j * S::kTaskWords + S::kMaxBits), row + (RB - 4) / 4);
        }
      };
      auto issue_tile = [&](int tile, const int (&bid)[TPT]) {
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
          if (task_comp(j) == 0) issue_task(std::integral_constant<int, KB>{}, tile, j, bid[j]);
          else issue_task(std::integral_constant<int, VB>{}, tile, j, bid[j]);
        }
        cp_async_commit();
      };

      // prologue: block ids of tiles 0 .. kMqStages - 1, copies of tiles 0 .. kMqStages - 2
      int bids[kMqStages][TPT];
#pragma unroll
      for (int u = 0; u < kMqStages; ++u)
#pragma unroll
        for (int j = 0; j < TPT; ++j) bids[u][j] = load_bid(u, j);
#pragma unroll
      for (int u = 0; u < kMqStages - 1; ++u) issue_tile(u, bids[u]);
      int bid_pref[TPT];  // block ids of tile it + kMqStages - 1
#pragma unroll
      for (int j = 0; j < TPT; ++j) bid_pref[j] = bids[kMqStages - 1][j];

      for (int it = 0; it < ntiles; ++it) {
        const int T0 = t_beg + it * kMqTile;
        // ---- this thread's words of tile it (its own copies: no barrier needed) -------
        cp_async_wait<kMqStages - 2>();
        RawTask<MAXB> raw[TPT];
        {
          const int st = it % kMqStages;
#pragma unroll
          for (int j = 0; j < TPT; ++j) {
            raw[j].ok = lds_u32(ring(st, j * S::kTaskWords + S::kMaxBits + 1)) != 0u;
#pragma unroll
            for (int k = 0; k < MAXB; ++k)
              raw[j].w[k] = raw[j].ok ? lds_u32(ring(st, j * S::kTaskWords + k)) : 0u;
            raw[j].nrm = (raw[j].ok && task_part(j) == 0) ? lds_u32(ring(st, j * S::kTaskWords + S::kMaxBits)) : 0u;
          }
        }
        // ---- A: exact-score and exact-value votes; every warp is done with the previous
        // tile.  One barrier votes on both; only a tile that needs either (rare) takes one
        // more to tell them apart.
        int kflag = 0, vflag = 0;
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
          if (task_part(j) != 0 || !raw[j].ok) continue;
          if (task_comp(j) == 0) kflag |= fabsf(__uint_as_float(raw[j].nrm)) * qn_cta > kMqFastBound;
          else vflag |= fabsf(__uint_as_float(raw[j].nrm)) > kMqFastValueNorm;
        }
        // an exact-value tile also takes the exact key path
        bool exact = false, exact_v = false;
        if (__syncthreads_or(kflag | vflag)) {
          exact = true;
          exact_v = __syncthreads_or(vflag) != 0;
        }

        // ---- dequantise the tile into shared memory --------------------------------
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
          const int t = task_tok(j), part = task_part(j);
          if (task_comp(j) == 0) {
            if (part == 0) {
              kn_s[t] = raw[j].ok ? __uint_as_float(raw[j].nrm) : 0.f;
              kadd_s[t] = raw[j].ok ? 0.f : -INFINITY;
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {  // 8 coordinates per 16-byte chunk
              uint32_t val[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int i = q4 * 8 + u;  // coordinate within the part
                const int bit = i * KB, k = bit >> 5, sh = bit & 31;
                uint32_t f = raw[j].w[k] >> sh;
                if (sh + KB > 32) f |= raw[j].w[k + 1] << (32 - sh);
                val[u] = __shfl_sync(kFullMask, kc_pair, (int)f);
              }
              const uint32_t off = sts_off[j] ^ (uint32_t)(q4 << 4);
              sts_v4(khi_base + off, __byte_perm(val[0], val[1], 0x5410), __byte_perm(val[2], val[3], 0x5410),
                     __byte_perm(val[4], val[5], 0x5410), __byte_perm(val[6], val[7], 0x5410));
              if (exact)
                sts_v4(klo_base + off, __byte_perm(val[0], val[1], 0x7632), __byte_perm(val[2], val[3], 0x7632),
                       __byte_perm(val[4], val[5], 0x7632), __byte_perm(val[6], val[7], 0x7632));
            }
          } else {
            if (part == 0) vn_s[t] = raw[j].ok ? __uint_as_float(raw[j].nrm) : 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t vp[4];
#pragma unroll
              for (int pr = 0; pr < 4; ++pr) {
                uint32_t val[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int i = q4 * 8 + pr * 2 + u;
                  const int bit = i * VB, k = bit >> 5, sh = bit & 31;
                  uint32_t f = raw[j].w[k] >> sh;
                  if (sh + VB > 32) f |= raw[j].w[k + 1] << (32 - sh);
                  val[u] = __shfl_sync(kFullMask, vc_pair, (int)f);
                }
                vp[pr] = __byte_perm(val[0], val[1], 0x5410);
              }
              sts_v4(v_base + (sts_off[j] ^ (uint32_t)(q4 << 4)), vp[0], vp[1], vp[2], vp[3]);
            }
          }
        }

        // ---- copies of tile it + kMqStages - 1 (its stage was read in iteration it - 1) --
        issue_tile(it + kMqStages - 1, bid_pref);
#pragma unroll
        for (int j = 0; j < TPT; ++j) bid_pref[j] = load_bid(it + kMqStages, j);
        __syncthreads();  // B: the tile is in shared memory

        // ---- math: skipped by a warp whose rows all end before the tile (such a warp
        // still takes part in an exact-value tile's barriers and remainder tile) ---------
        const bool live = __any_sync(kFullMask, T0 < lenA || T0 < lenB);
        if (!live && !exact_v) continue;  // (its copies are issued)
        // Exact-value tiles: once every warp's scores are done (barrier C), the key tile
        // is free; the fp16 remainders of the value tile go there (re-read from this
        // thread's ring words of the tile), visible after barrier D.
        auto value_remainders = [&]() {
          int comps[TPT];
#pragma unroll
          for (int j = 0; j < TPT; ++j) comps[j] = task_comp(j);
          mq_value_remainders<VB, MAXB, TPT, S::kTaskWords, S::kMaxBits, kThreads, S::kRingWords>(
              sbase + S::kOffRing, tid, it % kMqStages, comps, sts_off, khi_base, vc_pair);
        };
        float s[4][4];
#pragma unroll
        for (int jn = 0; jn < 4; ++jn)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[jn][e] = 0.f;
        auto scores = [&](auto exact_tag) {
          constexpr bool EX = decltype(exact_tag)::value;
          if (EX) {
            // q_hi * key_lo first (key_lo carries 2^12), scaled back before the main products
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const uint32_t kaddr = kb_lane ^ (uint32_t)((dh * KS + ks) << 5);
#pragma unroll
              for (int jp = 0; jp < 2; ++jp) {
                uint32_t kl[4];
                ldsm_x4(kl, kaddr + (uint32_t)(jp * 16 * S::kRow) + (uint32_t)(S::kOffKlo - S::kOffKhi));
                mma_f16(s[2 * jp], qh[ks], kl[0], kl[1]);
                mma_f16(s[2 * jp + 1], qh[ks], kl[2], kl[3]);
              }
            }
#pragma unroll
            for (int jn = 0; jn < 4; ++jn)
#pragma unroll
              for (int e = 0; e < 4; ++e) s[jn][e] *= kMqLoUnscale;
          }
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t ql[4];
            ldsm_x4(ql, ql_lane ^ (uint32_t)((dh * KS + ks) << 5));
            const uint32_t kaddr = kb_lane ^ (uint32_t)((dh * KS + ks) << 5);
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
              const uint32_t koff = kaddr + (uint32_t)(jp * 16 * S::kRow);  // tokens 16 jp ..
              uint32_t kb[4];
              ldsm_x4(kb, koff);
              mma_f16(s[2 * jp], qh[ks], kb[0], kb[1]);
              mma_f16(s[2 * jp + 1], qh[ks], kb[2], kb[3]);
              mma_f16(s[2 * jp], ql, kb[0], kb[1]);
              mma_f16(s[2 * jp + 1], ql, kb[2], kb[3]);
            }
          }
        };
        if (live) {
        if (exact) scores(std::true_type{});
        else scores(std::false_type{});
        if constexpr (SPLIT) {  // sum the two half-dimension scores of the row group
          float4* xb = reinterpret_cast<float4*>(smem + S::kOffX);
#pragma unroll
          for (int jn = 0; jn < 4; ++jn) xb[(warp * 32 + lane) * 4 + jn] = make_float4(s[jn][0], s[jn][1], s[jn][2], s[jn][3]);
          bar_pair(1 + grp);
          const int partner = warp ^ kMqGroups;
#pragma unroll
          for (int jn = 0; jn < 4; ++jn) {
            const float4 pv = xb[(partner * 32 + lane) * 4 + jn];
            s[jn][0] += pv.x;  // fp addition commutes: both warps get the same sums
            s[jn][1] += pv.y;
            s[jn][2] += pv.z;
            s[jn][3] += pv.w;
          }
        }
        }  // live

        if (exact_v) value_remainders();
        if (!live) continue;

        // scores: x nu_k, invalid tokens -inf, causal mask per row
#pragma unroll
        for (int jn = 0; jn < 4; ++jn) {
          const int tok = 8 * jn + 2 * c;
          const float2 kn = *reinterpret_cast<const float2*>(kn_s + tok);
          const float2 ka = *reinterpret_cast<const float2*>(kadd_s + tok);
          s[jn][0] = fmaf(s[jn][0], kn.x, ka.x);
          s[jn][1] = fmaf(s[jn][1], kn.y, ka.y);
          s[jn][2] = fmaf(s[jn][2], kn.x, ka.x);
          s[jn][3] = fmaf(s[jn][3], kn.y, ka.y);
          if (T0 + tok >= lenA) s[jn][0] = -INFINITY;
          if (T0 + tok + 1 >= lenA) s[jn][1] = -INFINITY;
          if (T0 + tok >= lenB) s[jn][2] = -INFINITY;
          if (T0 + tok + 1 >= lenB) s[jn][3] = -INFINITY;
        }
        // online softmax for rows r (e = 0, 1) and r + 8 (e = 2, 3); 4 lanes share a row.
        // The running max only moves when a score passes it by more than kMqSlack, so
        // p = 2^(s - m) <= 2^kMqSlack; most tiles move no max and skip the rescale.
        float mx[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          mx[hr] = -INFINITY;
#pragma unroll
          for (int jn = 0; jn < 4; ++jn) mx[hr] = fmaxf(mx[hr], fmaxf(s[jn][2 * hr], s[jn][2 * hr + 1]));
        }
        if (__any_sync(kFullMask, mx[0] > m_thr[0] || mx[1] > m_thr[1])) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float mt = fmaxf(mx[hr], __shfl_xor_sync(kFullMask, mx[hr], 1));
            mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 2));
            const float mn = mt > m_thr[hr] ? mt : m_run[hr];
            const float corr = mn == m_run[hr] ? 1.f : ex2(m_run[hr] - mn);
            m_run[hr] = mn;
            m_thr[hr] = mn + kMqSlack;
            l_run[hr] *= corr;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o[nt][2 * hr] *= corr;
              o[nt][2 * hr + 1] *= corr;
            }
          }
        }
        const float m_use[2] = {m_run[0] == -INFINITY ? 0.f : m_run[0], m_run[1] == -INFINITY ? 0.f : m_run[1]};
        // O += P' Vhat: k-step s2 covers tokens 16 s2 .. 16 s2 + 15.  EXV adds P'_lo Vhat_hi
        // and P'_hi Vhat_lo (the remainders sit in the key tile's space).
        auto values = [&](auto exv_tag) {
          constexpr bool EXV = decltype(exv_tag)::value;
          float pw[4][4];  // P' = p nu_v (the fast path packs each column group at once)
          uint32_t pa[2][4], pl[2][4];
#pragma unroll
          for (int jn = 0; jn < 4; ++jn) {
            const float2 vn = *reinterpret_cast<const float2*>(vn_s + 8 * jn + 2 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p = ex2(s[jn][e] - m_use[e >> 1]);
              l_run[e >> 1] += p;
              pw[jn][e] = p > 0.f ? p * ((e & 1) ? vn.y : vn.x) : 0.f;
            }
            if (!EXV) {
              pa[jn >> 1][(jn & 1) * 2 + 0] = half2_bits(pw[jn][0], pw[jn][1]);
              pa[jn >> 1][(jn & 1) * 2 + 1] = half2_bits(pw[jn][2], pw[jn][3]);
            }
          }
          float inv_f[2] = {1.f, 1.f};
          if (EXV) {  // per row: the largest P' to [2^11, 2^12), O by the same power of two
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              float pm = 0.f;
#pragma unroll
              for (int jn = 0; jn < 4; ++jn) pm = fmaxf(pm, fmaxf(pw[jn][2 * hr], pw[jn][2 * hr + 1]));
              pm = fmaxf(pm, __shfl_xor_sync(kFullMask, pm, 1));
              pm = fmaxf(pm, __shfl_xor_sync(kFullMask, pm, 2));
              float f;
              mq_tile_scale(pm, f, inv_f[hr]);
#pragma unroll
              for (int jn = 0; jn < 4; ++jn) {
                pw[jn][2 * hr] *= f;
                pw[jn][2 * hr + 1] *= f;
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                o[nt][2 * hr] *= f;
                o[nt][2 * hr + 1] *= f;
              }
            }
          }
          // EXV: pa = fp16 P' (scaled), pl = its fp16 remainders
#pragma unroll
          for (int jn = 0; jn < 4 && EXV; ++jn) {
            const uint32_t h01 = half2_bits(pw[jn][0], pw[jn][1]), h23 = half2_bits(pw[jn][2], pw[jn][3]);
            pa[jn >> 1][(jn & 1) * 2 + 0] = h01;
            pa[jn >> 1][(jn & 1) * 2 + 1] = h23;
            {
              const __half2 x01 = *reinterpret_cast<const __half2*>(&h01);
              const __half2 x23 = *reinterpret_cast<const __half2*>(&h23);
              pl[jn >> 1][(jn & 1) * 2 + 0] = half2_bits(pw[jn][0] - __low2float(x01), pw[jn][1] - __high2float(x01));
              pl[jn >> 1][(jn & 1) * 2 + 1] = half2_bits(pw[jn][2] - __low2float(x23), pw[jn][3] - __high2float(x23));
            }
          }
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
#pragma unroll
            for (int dp = 0; dp < NT / 2; ++dp) {
              const uint32_t vaddr = (vb_lane ^ (uint32_t)((dh * (NT / 2) + dp) << 5)) + (uint32_t)(s2 * 16 * S::kRow);
              uint32_t vb[4];
              ldsm_x4_t(vb, vaddr);
              mma_f16(o[2 * dp], pa[s2], vb[0], vb[1]);
              mma_f16(o[2 * dp + 1], pa[s2], vb[2], vb[3]);
              if (EXV) {
                mma_f16(o[2 * dp], pl[s2], vb[0], vb[1]);
                mma_f16(o[2 * dp + 1], pl[s2], vb[2], vb[3]);
              }
            }
          }
          if (EXV) {
            // value remainders (stored x 2^12, in the key tile's space) against P'_hi 2^-12:
            // scaling an fp16 by a power of two is exact while it stays normal, and the
            // weights that leave the normal range are 2^-13 of the tile's largest or less
            const __half2 unscale = __float2half2_rn(kMqLoUnscale);
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                __half2 x = *reinterpret_cast<const __half2*>(&pa[s2][k]);
                x = __hmul2(x, unscale);
                pa[s2][k] = *reinterpret_cast<const uint32_t*>(&x);
              }
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
#pragma unroll
              for (int dp = 0; dp < NT / 2; ++dp) {
                const uint32_t vaddr = (vb_lane ^ (uint32_t)((dh * (NT / 2) + dp) << 5)) + (uint32_t)(s2 * 16 * S::kRow);
                uint32_t vl[4];
                ldsm_x4_t(vl, vaddr - v_base + khi_base);
                mma_f16(o[2 * dp], pa[s2], vl[0], vl[1]);
                mma_f16(o[2 * dp + 1], pa[s2], vl[2], vl[3]);
              }
            }
          }
          if (EXV) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o[nt][0] *= inv_f[0];
              o[nt][1] *= inv_f[0];
              o[nt][2] *= inv_f[1];
              o[nt][3] *= inv_f[1];
            }
          }
        };
        if (exact_v) values(std::true_type{});
        else values(std::false_type{});
      }
    }
    cp_async_wait<0>();  // no copy of this segment outlives it
    s0 = s1;
  }

  // ---- partials: (m, l, acc / alpha_v) per (row, q head) of this window and split ------
  const float inv_alpha_v = 1.0f / a.v_alpha;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    float l = l_run[hr];
    l += __shfl_xor_sync(kFullMask, l, 1);
    l += __shfl_xor_sync(kFullMask, l, 2);
    const int mr = grp * 16 + r + 8 * hr;
    const int wrow = mr / G;
    if (wrow < nrows) {
      const int64_t slot = ((int64_t)(i0 + wrow) * Hq + (int64_t)h * G + mr % G) * args.nsplit + split;
      float* acc = args.part_acc + slot * D + dh * SH::kDh;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float2*>(acc + 8 * nt + 2 * c) =
            make_float2(o[nt][2 * hr] * inv_alpha_v, o[nt][2 * hr + 1] * inv_alpha_v);
      if (c == 0 && dh == 0) {
        args.part_ml[slot * 2 + 0] = m_run[hr];
        args.part_ml[slot * 2 + 1] = l;
      }
    }
  }
}

template <int D, int KB, int VB, int G>
cudaError_t launch_mq_one(const MqArgs& m, int grid, cudaStream_t stream) {
  constexpr int bytes = MqSmem<D, KB, VB>::kAlloc;
  auto kern = prefill_mq_kernel<D, KB, VB, G>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  kern<<<grid, MqShape<D>::kThreads, bytes, stream>>>(m);
  err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

template <int D, int KB, int VB>
cudaError_t launch_mq_g(const MqArgs& m, int grid, cudaStream_t stream) {
  switch (m.a.num_q_heads / m.a.num_kv_heads) {
    case 1: return launch_mq_one<D, KB, VB, 1>(m, grid, stream);
    case 2: return launch_mq_one<D, KB, VB, 2>(m, grid, stream);
    case 4: return launch_mq_one<D, KB, VB, 4>(m, grid, stream);
    case 8: return launch_mq_one<D, KB, VB, 8>(m, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_mq_bits(const MqArgs& m, int grid, cudaStream_t stream) {
  const int kb = m.a.k_bits, vb = m.a.v_bits;
  if (kb == 4 && vb == 4) return launch_mq_g<D, 4, 4>(m, grid, stream);
  if (kb == 4 && vb == 2) return launch_mq_g<D, 4, 2>(m, grid, stream);
  if (kb == 2 && vb == 4) return launch_mq_g<D, 2, 4>(m, grid, stream);
  if (kb == 2 && vb == 2) return launch_mq_g<D, 2, 2>(m, grid, stream);
  if (kb == 3 && vb == 3) return launch_mq_g<D, 3, 3>(m, grid, stream);
  if (kb == 5 && vb == 5) return launch_mq_g<D, 5, 5>(m, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

bool prefill_mq_supported(const DecodeArgs& a) {
  const int G = a.num_kv_heads > 0 ? a.num_q_heads / a.num_kv_heads : 0;
  // exactly the instantiations in launch_mq_bits
  const bool bits = ((a.k_bits == 2 || a.k_bits == 4) && (a.v_bits == 2 || a.v_bits == 4)) ||
                    (a.k_bits == a.v_bits && (a.k_bits == 3 || a.k_bits == 5));
  return (a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256) && bits && (G == 1 || G == 2 || G == 4 || G == 8) &&
         a.block_size >= 1;
}

MqPlan plan_prefill_mq(const DecodeArgs& a, int num_sms, bool one_row_per_window) {
  MqPlan p{};
  const int G = std::max(1, a.num_kv_heads > 0 ? a.num_q_heads / a.num_kv_heads : 1);
  const int rows_per_window = one_row_per_window ? 1 : std::max(1, kMqRows / G);
  p.rows_per_window = rows_per_window;
  p.windows = (std::max(0, a.batch) + rows_per_window - 1) / rows_per_window;
  const long long cap = (long long)std::max(0, a.max_blocks_per_seq) * std::max(1, a.block_size);
  const long long units = std::max(1LL, (long long)p.windows * std::max(1, a.num_kv_heads));
  const long long target = 6LL * num_sms;  // about two waves of three resident CTAs per SM
  long long nsplit = (target + units - 1) / units;
  // splits of >= 1024 tokens (>= 256 for one-row windows, whose partials are small)
  const long long min_len = one_row_per_window ? 256 : 1024;
  nsplit = std::max(1LL, std::min(nsplit, std::max(1LL, (cap + min_len - 1) / min_len)));
  long long len = (cap + nsplit - 1) / nsplit;
  len = std::max(32LL, (len + 31) / 32 * 32);
  p.split_len = (int)std::min(len, (long long)1 << 30);
  p.nsplit = (int)std::max(1LL, (cap + p.split_len - 1) / p.split_len);
  p.workspace_bytes = (size_t)std::max(0, a.batch) * a.num_q_heads * p.nsplit * (a.head_dim + 2) * sizeof(float) + 16;
  return p;
}

cudaError_t launch_prefill_mq(const DecodeArgs& a, const MqPlan& p, cudaStream_t stream) {
  if (a.status) {
    cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
  }
  if (a.batch == 0) return cudaSuccess;
  MqArgs m;
  m.a = a;
  m.nsplit = p.nsplit;
  m.split_len = p.split_len;
  m.bs_shift = -1;
  for (int k = 0; k < 31; ++k)
    if (a.block_size == (1 << k)) m.bs_shift = k;
  m.windows = p.windows;
  m.rows_per_window = p.rows_per_window;
  m.part_acc = static_cast<float*>(a.workspace);
  m.part_ml = m.part_acc + (size_t)a.batch * a.num_q_heads * p.nsplit * a.head_dim;
  const long long grid = (long long)p.windows * p.nsplit * a.num_kv_heads;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t err = a.head_dim == 64    ? launch_mq_bits<64>(m, (int)grid, stream)
                    : a.head_dim == 128 ? launch_mq_bits<128>(m, (int)grid, stream)
                    : a.head_dim == 256 ? launch_mq_bits<256>(m, (int)grid, stream)
                                        : cudaErrorInvalidValue;
  if (err != cudaSuccess) return err;
  return launch_combine_splits(m.part_acc, m.part_ml, a.batch * a.num_q_heads, p.nsplit, a.head_dim, a.signs, a.out,
                               a.out_dtype, stream);
}

}  // namespace tq
