// Tensor-core paged decode over packed TurboQuant pages (sm_103a, mma.sync f16 -> f32).
//
// TurboQuant docs: "vLLM Usage" (TQ Packed Page Contract: decode_tq4_paged) and
// "Architecture" (Diagnostic vs Serving Paths: keys consumed compressed, packed-V).
//
// Work split.  The blocks of all sequences form one flat list (sequence-major); CTA i
// of C owns the contiguous range [N*i/C, N*(i+1)/C).  Every CTA is busy for the same
// number of blocks whatever the length mix, and a CTA emits one split partial per
// (sequence it touches, warp slot), so the combine pass reads C + B partials at most.
//
// Per CTA: WPH warps per kv head (warp w: head w % H, block slot w / H).  A stage holds
// WPH consecutive blocks; their whole K and V slabs (block_size * H * row_bytes bytes,
// contiguous in the page tensor) are brought into shared memory by one bulk async copy
// each, issued by a producer warp (the CTA's last warp, which does no math) and
// completed on a per-stage "full" mbarrier.  Every consumer warp signals a per-stage
// "empty" mbarrier when it is done with the stage, and the producer waits on it before
// it refills the buffers.  No CTA-wide barrier in the main loop.  (A consumer warp that
// also issues the copies delays them by its own math and serialises copy and compute.)
//
// Scores.  For a 16-token tile of one kv head the warp computes S[16 tok x 8 q-heads]
// = Khat[16 x D] * qrot^T with m16n8k16 MMAs.  The A operand is looked up from the
// packed bytes: each 2b-bit field (two neighbouring coordinates) indexes a table of
// (fp16 hi, fp16 lo) centroid pairs, replicated per lane to avoid bank conflicts; the
// query is split into fp16 hi + lo as well, and hi*hi + lo*hi + hi*lo carries ~22
// significant bits, so the score keeps fp32-level accuracy even for very large norms.
// The k order inside a fragment is a fixed permutation of the coordinates; the query
// fragment follows the same permutation.  3- and 5-bit rows have fields that cross word
// boundaries: each lane takes a contiguous window of whole fields and extracts them with
// shifts (funnel shifts across words) into the address of its own table copy; 3-bit rows
// look up a pair of coordinates per 6-bit field, 5-bit rows one coordinate per field.
//
// Values.  Accumulated in rotated space with the contraction over (token, parity):
// O'[pair][2g + e] += sum_t Vhat[t][2 pair + e] * P'[g][t], so one table entry gives
// both coordinates of a pair of one token.  V centroids are stored as fp16(alpha * c),
// alpha chosen on the host so that alpha * c lands near fp16 grid points; 1/alpha is
// applied when the partial is written.
//
// Large norms.  Nothing bounds a row's norm (the writer takes any raw row), so tiles whose
// largest value norm passes kFastValueNorm take an exact path: the value weights
// P' = p * nu_v of each q head are scaled by a power of two that puts their largest near
// 2^12 (the accumulators scaled by the same power before the tile and back after it, both
// exact), then split into fp16 hi + lo, with the value table entries split the same way:
// V_hi P'_hi + V_lo P'_hi + V_hi P'_lo carries ~22 significant bits for every weight the
// output can feel.  Such tiles also take the exact key path (the error of the hi-only key
// scores, ~1e-3 of p at the fast bound, would otherwise be multiplied by the large norm).
// Other tiles have P' <= 2^kRescaleSlack * kFastValueNorm = 2048, well inside fp16.
//
// Softmax: online, base 2 (log2 e folded into the query), per q head.  Rows of tokens
// past the sequence end are masked (score -inf, value norm 0: their bytes are stale);
// blocks with an out-of-range id are skipped and reported through the status word.
// The kernels are instantiated and launched by tq_decode_tc.cu.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kBS = 16;       // tokens per block (the only block size this kernel takes)
constexpr float kLog2eTc = 1.4426950408889634f;

struct BlockMeta {
  int b;      // sequence
  int j;      // block index within the sequence
  int ntok;   // valid tokens in the block (1..16); 0 = no block in this slot
  int valid;  // block id inside [0, num_blocks)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// mbarrier and bulk-copy primitives (shared-window addresses).  Every wait is bounded:
// after `tries` unsuccessful tries the caller reports kTimeout and stops.  The waits of the
// pipeline take TcArgs::wait_tries (normally kDefaultWaitTries); the producer's final
// drain of its own copies always takes kDefaultWaitTries, so no copy is in flight when
// the CTA exits.

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(tx) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `bar` with parity `parity` to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t tries) {
  for (uint32_t i = 0; i < tries; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// that completes `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Shared load from an absolute shared-window address.  Not volatile: its address is
// computed from data read after the stage's wait, which orders it.
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32_off128(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1+128];\n" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t ld32(const unsigned char* p) { return *reinterpret_cast<const uint32_t*>(p); }

// 2^x with the hardware approximation (denormal results flush to zero): the softmax
// weights it produces are relative to the running max, so tiny values do not matter.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// Power-of-two scale (and its inverse) that brings a positive x to [2^11, 2^12): both
// exact; 1 and 1 for x = 0 or subnormal (nothing there that could reach the output).
__device__ __forceinline__ void tile_scale(float x, float& f, float& inv_f) {
  int e = (int)((__float_as_uint(x) >> 23) & 0xffu);  // biased exponent of x (x >= 0)
  if (e == 0) {
    f = inv_f = 1.f;
    return;
  }
  e = max(12, e);  // x < 2^-115: clamp, its terms are far below anything the output feels
  f = __uint_as_float((uint32_t)(265 - e) << 23);   // 2^(138 - e)
  inv_f = __uint_as_float((uint32_t)(e - 11) << 23);  // 2^(e - 138)
}

// D = A * B + D, m16n8k16, A row-major f16, B col-major f16, f32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Split x into fp16 hi + fp16 lo with the remainder scaled by 2^kLoShift:
// x ~= hi + lo * 2^-kLoShift to ~22 significant bits.  (The remainder of a value below 1/4
// would fall into fp16's subnormal range, where only 2^-25 of absolute precision is left;
// the products with lo parts are multiplied by 2^-kLoShift when they are summed, exactly.)
constexpr int kLoShift = 12;
constexpr float kLoScale = 4096.0f;        // 2^kLoShift
constexpr float kLoUnscale = 1.0f / 4096;  // 2^-kLoShift
__device__ __forceinline__ void split_half(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn((x - __half2float(hi)) * kLoScale);
}

// Field i of width W (bits [W i, W i + W)) of a window of words w (i compile-time).
template <int W>
__device__ __forceinline__ uint32_t win_field(const uint32_t* w, int i) {
  const int bit = W * i, wi = bit >> 5, sh = bit & 31;
  return (sh <= 32 - W ? (w[wi] >> sh) : __funnelshift_r(w[wi], w[wi + 1], sh)) & ((1u << W) - 1u);
}
// The same field shifted to bits [7, 7 + W) and OR'd into `lane_base`: the shared address
// of entry `field` of a per-lane replicated table of 128-byte entries.
template <int W>
__device__ __forceinline__ uint32_t win_addr(const uint32_t* w, int i, uint32_t lane_base) {
  const int bit = W * i, wi = bit >> 5, sh = bit & 31;
  uint32_t x;
  if (sh <= 32 - W) x = sh >= 7 ? (w[wi] >> (sh - 7)) : (w[wi] << (7 - sh));
  else x = __funnelshift_r(w[wi], w[wi + 1], sh - 7);
  return (x & (((1u << W) - 1u) << 7)) | lane_base;
}

// PROD: product-quantised ("QJL residual") key rows -- KB-bit MSE indices, then D sign bits,
// then fp32 nu and gamma.
template <int D, int KB, int VB, int G, int WPH, bool PROD = false>
struct TcCfg {
  static constexpr int kRBK = D * KB / 8 + (PROD ? D / 8 + 8 : 4);  // row bytes
  static constexpr int kKNormOff = D * KB / 8 + (PROD ? D / 8 : 0);   // byte of nu in a K row
  static constexpr int kSignOff = D * KB / 8;                          // product rows: sign bits
  static constexpr int kRBV = D * VB / 8 + 4;
  static constexpr int kWK = D * KB / 32;              // index words per K row
  static constexpr int kWV = D * VB / 32;
  static constexpr bool kKWin = KB == 3 || KB == 5;    // window mode: 3- and 5-bit rows
  // (and 2-bit values at D = 64, whose 4 index words do not split into 8 word columns)
  static constexpr bool kVWin = VB == 3 || VB == 5 || (VB == 2 && D == 64);
  static constexpr int kPWK = kKWin ? 1 : 16 / KB;      // pairs per word (2- and 4-bit rows)
  static constexpr int kPWV = kVWin ? 1 : 16 / VB;
  static constexpr int kKSteps = D / 16;               // score k-steps
  static constexpr int kMTiles = D / 32;               // value m-tiles
  static constexpr int kNT = (2 * G + 7) / 8;          // value n-tiles (N = 2G)
  // Byte-field table T (4-bit indices): 256 entries x 256 bytes, [0, 128) the fp16 hi
  // parts of the K centroid pairs and [128, 256) the V pairs fp16(alpha c), 32 lane
  // copies each so lookups are bank conflict free.  T sits at a 64 KB aligned shared
  // address, so one PRMT of (packed word, T base | lane * 4) yields the absolute
  // address of an entry.
  static constexpr bool kHasT = KB == 4 || VB == 4;
  // The small tables (K lo parts of byte fields, read only by tiles that need the exact
  // score, and the nibble-field tables of 2-bit indices) have one copy each and live in
  // the fixed part of the shared memory.
  // Window mode (3- and 5-bit rows, whose fields cross word boundaries).  K: lane c of a
  // row owns the pairs [c D/8, (c + 1) D/8), KB D/128 whole words from word KB D/128 c,
  // taken in chunks of KB words (32 coordinates, 8 k-steps) -- at D = 64, 16 KB bits from
  // bit 16 KB c (half-word aligned), 4 k-steps; k-step s takes pairs c D/8 + 2s and + 2s + 1.
  // V: lane r owns the pairs [r D/16, (r + 1) D/16) of a token row (D = 64: 8 VB bits from
  // bit 8 VB r, byte aligned; D = 128: 16 VB bits from bit 16 VB r, half-word aligned;
  // D = 256: VB whole words); m-tile i takes pairs r D/16 + 2i and + 2i + 1.  2-bit values at
  // D = 64 take this mode with 4-bit pair fields (a 16-entry pair table).  3-bit rows look up a pair per 6-bit
  // field in a 64-entry table of (fp16 hi, fp16 hi) pairs; 5-bit rows look up each
  // coordinate in a 32-entry table of (fp16 hi, fp16 lo x 2^12) and join two with a PRMT.
  // Each table is replicated per lane (entry e of lane l at e * 128 + 4 l) in an 8 KB slot
  // aligned to 8 KB, so the address of an entry is the field, shifted to bit 7, OR'd into
  // (table base | lane * 4).  K and V widths are independent: each component takes its own
  // form.
  static constexpr int kKLaneWords = KB * D / 128;  // K words per lane and row (window mode)
  // Table region: T (64 KB, 64 KB aligned) when either width is 4, then an 8 KB slot for a
  // window-mode K table and one for a window-mode V table; empty for 2-bit rows.
  static constexpr int kWinSlot = 64 * 128;
  static constexpr int kKWOff = kHasT ? 256 * 256 : 0;
  static constexpr int kVWOff = kKWOff + (kKWin ? kWinSlot : 0);
  // product rows: the sign table, (+-1, +-1) fp16 pairs for the four bits of a nibble, per
  // lane (entry n of lane l at 256 n + 8 l), in one more slot
  static constexpr int kSgnOff = kVWOff + (kVWin ? kWinSlot : 0);
  static constexpr int kTBytes = kSgnOff + (PROD ? kWinSlot : 0);
  static constexpr int kTAlign = kHasT ? 256 * 256 : kWinSlot;
  static_assert(kKWin || kWK % 4 == 0, "K row must split into 4 interleaved word columns");
  static_assert(kVWin || kWV % 8 == 0, "V row must split into 8 interleaved word columns");
  static_assert(G == 4 || G == 8, "GQA group 4 or 8");
  static_assert(KB >= 2 && KB <= 5 && VB >= 2 && VB <= 5, "2- to 5-bit indices");
  static_assert(!(kKWin || kVWin) || D == 64 || D == 128 || D == 256, "window mode at head_dim 64, 128 or 256");
  static_assert(!PROD || KB <= 4, "product rows: 2- to 4-bit MSE indices");
};

struct TcArgs {
  DecodeArgs a;
  int num_ctas;           // C
  int k_tok_stride;       // smem bytes per token in a K slab (H*RBK + pad)
  int v_tok_stride;
  int k_slab_smem;        // bytes of the K part of a block buffer
  int v_slab_smem;
  int k_row_copy;         // 1: K copied one token row at a time (padded rows); 0: one slab copy
  int v_row_copy;
  float v_alpha;          // V centroid scale
  float k_alpha;          // K centroid scale
  int nst;                // pipeline stages (WPH block buffers each), 2..kMaxStages
  int n_lo;               // block buffers below the T table
  int buf_lo;             // dynamic-smem offset of buffer 0
  int buf_hi;             // dynamic-smem offset of buffer n_lo
  int buf_bytes;          // bytes per block buffer
  int t_off;              // dynamic-smem offset of T (64 KB aligned shared address)
  uint32_t wait_tries;    // tries of a pipeline wait before it reports kTimeout
  float* part_acc;        // [WPH*(C+B)][Hq][D]
  float* part_ml;         // [WPH*(C+B)][Hq][2]
  const float* p_all;     // product rows: p = S q~ per (sequence, q head), [B][Hq][D]
  float sketch;           // product rows: sqrt(pi / 2) / D
  int* prefix;            // [B+1] block prefix sums (written by CTA 0)
};

// Fixed part of the dynamic shared memory (offsets from its start).
constexpr int kMaxStages = 8;
constexpr int kOffBar = 0;                                  // full[kMaxStages], empty[kMaxStages]
constexpr int kOffMeta = kOffBar + 2 * kMaxStages * 8;      // BlockMeta[kMaxStages][WPH <= 2]
constexpr int kOffScan = kOffMeta + kMaxStages * 2 * 16;    // int[36]
constexpr int kOffK2 = kOffScan + 36 * 4;                   // nibble K table, 16 x 8 bytes
constexpr int kOffV2 = kOffK2 + 16 * 8;                     // nibble V table (hi, lo), 16 x 8 bytes
constexpr int kOffL = kOffV2 + 16 * 8;                      // byte K lo table, 256 x 4 bytes
constexpr int kOffVL = kOffL + 256 * 4;                     // byte V lo table, 256 x 4 bytes
constexpr int kOffK3L = kOffVL + 256 * 4;                   // 6-bit K lo table, 64 x 4 bytes
constexpr int kOffV3L = kOffK3L + 64 * 4;                   // 6-bit V lo table, 64 x 4 bytes
constexpr int kMiscBytes = (kOffV3L + 64 * 4 + 127) / 128 * 128;

constexpr float kRescaleSlack = 6.0f;  // log2 units the running max may lag behind
// Largest bound nu_k * ||q_rot|| (log2 units) of a tile scored with the fp16-hi key part
// only.  With the alpha scaling the hi part is within ~1e-4 relative of the fp32
// centroid, so the score error of such a tile stays far below the output tolerance;
// tiles above the bound (rows with very large norms) add the fp16-lo part.
constexpr float kFastScoreBound = 48.0f;
// Largest value norm of a tile whose values take the fp16 path (P' and the value table
// each rounded once to fp16, ~2^-12 relative): there the output error stays far below
// the 2e-3 + 2e-3 |o| tolerance.  Tiles with a larger norm add the fp16 remainders of
// both (V_hi P'_hi + V_lo P'_hi + V_hi P'_lo, ~2^-22 relative), since a rounding error
// proportional to a large norm can exceed the absolute part of the tolerance wherever
// the output element itself is small.
constexpr float kFastValueNorm = 32.0f;

// At most 9 warps (8 consumers + the producer).  The register file is granted to a CTA
// in groups of 4 warps, so 288 threads take 12 warps' worth: 168 registers a thread at most
// (a launch at more registers is refused).
template <int D, int KB, int VB, int G, int WPH, bool PROD = false>
__global__ void __launch_bounds__(32 * 9, 1) decode_tc_kernel(TcArgs args) {
  using Cfg = TcCfg<D, KB, VB, G, WPH, PROD>;
  const DecodeArgs& a = args.a;
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = a.num_kv_heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int ncons = nwarps - 1;  // consumer warps; warp ncons is the producer
  const int cta = blockIdx.x, C = args.num_ctas;
  const int B = a.batch;
  const int cap = a.max_blocks_per_seq * kBS;
  const int nst = args.nst;

  const uint32_t smem_base = smem_u32(smem);
  const uint32_t t_base = smem_base + (uint32_t)args.t_off;
  if (Cfg::kTBytes > 0 && (t_base & (uint32_t)(Cfg::kTAlign - 1)) != 0u) {  // layout for another shared window
    if (tid == 0 && a.status) atomicMax(a.status, (int32_t)kUnsupported);
    return;
  }
  unsigned char* lutT = smem + args.t_off;
  unsigned char* lutL = smem + kOffL;
  unsigned char* lutK2 = smem + kOffK2;
  unsigned char* lutV2 = smem + kOffV2;
  unsigned char* lutVL = smem + kOffVL;
  unsigned char* lutK3L = smem + kOffK3L;
  unsigned char* lutV3L = smem + kOffV3L;
  unsigned char* lutKW = smem + args.t_off + Cfg::kKWOff;  // window-mode tables (3- and 5-bit rows)
  unsigned char* lutVW = smem + args.t_off + Cfg::kVWOff;
  BlockMeta* meta = reinterpret_cast<BlockMeta*>(smem + kOffMeta);
  int* scan_tmp = reinterpret_cast<int*>(smem + kOffScan);
  auto bar_full = [&](int i) -> uint32_t { return smem_base + kOffBar + 8u * i; };
  auto bar_empty = [&](int i) -> uint32_t { return smem_base + kOffBar + 8u * (kMaxStages + i); };
  auto buf_off = [&](int slot, int u) -> int {
    const int idx = slot * WPH + u;
    return idx < args.n_lo ? args.buf_lo + idx * args.buf_bytes : args.buf_hi + (idx - args.n_lo) * args.buf_bytes;
  };

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), (uint32_t)ncons);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }

  // ---- flat block list: N, this CTA's range, its first and last sequence ------------
  auto nblocks_of = [&](int b) -> int {
    int len = __ldg(a.seq_lens + b);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    return (len + kBS - 1) / kBS;
  };
  int local = 0;
  bool bad_len = false;
  for (int b = tid; b < B; b += nthreads) {
    const int len = __ldg(a.seq_lens + b);
    bad_len |= (len < 0 || len > cap);
    local += nblocks_of(b);
  }
  if (cta == 0 && a.status && __any_sync(kFullMask, bad_len) && lane == 0) atomicMax(a.status, (int32_t)kInvalidArg);
  local = (int)__reduce_add_sync(kFullMask, (unsigned)local);
  if (lane == 0) scan_tmp[warp] = local;
  __syncthreads();
  long long N = 0;
  for (int w = 0; w < nwarps; ++w) N += scan_tmp[w];
  const long long g_lo = N * cta / C, g_hi = N * (cta + 1) / C;
  __syncthreads();
  if (tid == 0) {
    scan_tmp[32] = -1;
    scan_tmp[33] = -1;
    scan_tmp[34] = 0;
  }
  int carry = 0;
  for (int base = 0; base < B; base += nthreads) {
    const int b = base + tid;
    const int nb = b < B ? nblocks_of(b) : 0;
    int incl = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    __syncthreads();
    if (lane == 31) scan_tmp[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int w = 0; w < nwarps; ++w) {
      if (w < warp) wbase += scan_tmp[w];
      total += scan_tmp[w];
    }
    const int excl = carry + wbase + incl - nb;
    if (b < B) {
      if (cta == 0) args.prefix[b] = excl;
      if (nb > 0 && excl <= g_lo && g_lo < excl + nb) {
        scan_tmp[32] = b;
        scan_tmp[34] = (int)(g_lo - excl);
      }
      if (nb > 0 && excl <= g_hi - 1 && g_hi - 1 < excl + nb) scan_tmp[33] = b;
    }
    carry += total;
  }
  if (cta == 0 && tid == 0) args.prefix[B] = carry;
  __syncthreads();  // also: barriers initialised
  // the combine grid may be scheduled now; it waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  if (g_lo >= g_hi) return;  // nothing to do (uniform; no copy was issued)
  const int b_first = scan_tmp[32], b_last = scan_tmp[33], j_first = scan_tmp[34];
  const int nstages = (int)((g_hi - g_lo + WPH - 1) / WPH);

  // ---- producer state: block cursor of lane u < WPH, blocks g_lo + WPH*st + u ---------
  int cb = b_first, cj = j_first, cnb = nblocks_of(b_first);
  long long cg = g_lo;
  auto cursor_advance = [&](int steps) {
    cg += steps;
    cj += steps;
    while (cg < g_hi && cj >= cnb) {
      cj -= cnb;
      ++cb;
      cnb = nblocks_of(cb);
    }
  };
  const bool producer = warp == ncons;
  if (producer && lane < WPH) cursor_advance(lane);
  // The metadata of a stage is loaded (global reads in flight) one stage before it is
  // stored, so the producer does not wait on those reads when it issues the copies.
  BlockMeta pend_m{0, 0, 0, 0};
  int pend_len = 0, pend_bid = -1;
  auto meta_load = [&]() {  // producer lanes < WPH: the next stage of this lane's cursor
    pend_m = BlockMeta{0, 0, 0, 0};
    pend_bid = -1;
    pend_len = 0;
    if (cg < g_hi) {
      pend_len = __ldg(a.seq_lens + cb);
      pend_m.b = cb;
      pend_m.j = cj;
      pend_bid = __ldg(a.block_table + (int64_t)cb * a.max_blocks_per_seq + cj);
      pend_m.ntok = 1;  // marks a real block until meta_store fills the count
      cursor_advance(WPH);
    }
  };
  // Stores the pending metadata into ring slot `slot`; returns the block id to copy (-1: none).
  auto meta_store = [&](int slot) -> int {
    BlockMeta m = pend_m;
    int bid = -1;
    if (m.ntok) {
      const int len = pend_len < 0 ? 0 : (pend_len > cap ? cap : pend_len);
      m.ntok = min(kBS, len - m.j * kBS);
      m.valid = (pend_bid >= 0 && (int64_t)pend_bid < a.num_blocks);
      if (!m.valid && a.status)
        atomicMax(a.status, (int32_t)kBlockOutOfRange);
      bid = m.valid ? pend_bid : -1;
    }
    meta[slot * WPH + lane] = m;
    return bid;
  };

  // ---- copies -------------------------------------------------------------------------
  const int kraw = H * Cfg::kRBK, vraw = H * Cfg::kRBV;
  const int k_slab = kBS * kraw, v_slab = kBS * vraw;
  const uint32_t blk_tx = (uint32_t)(k_slab + v_slab);
  // Producer step (all lanes of the producer): metadata of the next stage into ring slot `slot`, then
  // the copies of its valid blocks on full[slot].  The caller has made sure the slot's
  // buffers are free.
  auto produce = [&](int slot) {
    int bid = -1;
    if (lane < WPH) {
      bid = meta_store(slot);
      meta_load();
    }
    __syncwarp();
    int bids[WPH];
    uint32_t tx = 0;
#pragma unroll
    for (int u = 0; u < WPH; ++u) {
      bids[u] = __shfl_sync(kFullMask, bid, u);
      if (bids[u] >= 0) tx += blk_tx;
    }
    if (lane == 0) mbar_arrive_expect_tx(bar_full(slot), tx);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < WPH; ++u) {
      if (bids[u] < 0) continue;
      const unsigned char* ksrc = a.k_pages + (int64_t)bids[u] * k_slab;
      const unsigned char* vsrc = a.v_pages + (int64_t)bids[u] * v_slab;
      const uint32_t kdst = smem_base + (uint32_t)buf_off(slot, u);
      const uint32_t vdst = kdst + (uint32_t)args.k_slab_smem;
      if (lane < 16) {
        if (args.k_row_copy)
          bulk_g2s(kdst + lane * args.k_tok_stride, ksrc + lane * kraw, (uint32_t)kraw, bar_full(slot));
        else if (lane == 0)
          bulk_g2s(kdst, ksrc, (uint32_t)k_slab, bar_full(slot));
      } else {
        const int t = lane - 16;
        if (args.v_row_copy)
          bulk_g2s(vdst + t * args.v_tok_stride, vsrc + t * vraw, (uint32_t)vraw, bar_full(slot));
        else if (t == 0)
          bulk_g2s(vdst, vsrc, (uint32_t)v_slab, bar_full(slot));
      }
    }
  };

  // ---- consumer state ----------------------------------------------------------------
  const int h = warp;  // consumer warp h: kv head h of every block
  const int r = lane >> 2, c = lane & 3;
  const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
  const float qmul = scale * kLog2eTc / sqrtf((float)D);
  const float inv_alpha_k = 1.0f / args.k_alpha;
  const int kts = args.k_tok_stride, vts = args.v_tok_stride;
  const uint32_t t_lane = t_base | (uint32_t)(lane * 4);  // T base (bits 16-31) | lane copy
  // value-B selectors: the P value goes to the low half when (r & 1) == 0, else the high half
  const int hsel = (r >> 1) & 1;
  const uint32_t sel_b = (r & 1) ? (0x0044u | ((2u * hsel) << 8) | ((2u * hsel + 1u) << 12))
                                 : ((2u * hsel) | ((2u * hsel + 1u) << 4) | 0x4400u);

  // Table lookups for field e of word w.  4-bit fields: one PRMT places byte e of w at
  // bits 8-15 of (T base | lane * 4), the absolute address of this lane's copy.
  auto t_addr = [&](uint32_t w, int e) -> uint32_t { return __byte_perm(w, t_lane, 0x7604u | ((uint32_t)e << 4)); };
  auto k_hi = [&](uint32_t w, int e) -> uint32_t {
    if (KB == 4) return lds32(t_addr(w, e));
    return ld32(lutK2 + (((w >> (4 * e)) & 15u) << 3));
  };
  auto k_lo = [&](uint32_t w, int e) -> uint32_t {
    if (KB == 4) return ld32(lutL + (((w >> (8 * e)) & 255u) << 2));
    return ld32(lutK2 + (((w >> (4 * e)) & 15u) << 3) + 4);
  };
  auto v_lookup = [&](uint32_t w, int e) -> uint32_t {
    if (VB == 4) return lds32_off128(t_addr(w, e));
    return ld32(lutV2 + (((w >> (4 * e)) & 15u) << 3));
  };
  auto v_lookup_lo = [&](uint32_t w, int e) -> uint32_t {  // fp16 remainders of the same pair
    if (VB == 4) return ld32(lutVL + (((w >> (8 * e)) & 255u) << 2));
    return ld32(lutV2 + (((w >> (4 * e)) & 15u) << 3) + 4);
  };

  // Window mode: the A registers of pair j of a window w (fp16 hi parts of coordinates 2j,
  // 2j + 1; and their remainders, for the exact paths).
  const uint32_t kw_lane = (t_base + (uint32_t)Cfg::kKWOff) | (uint32_t)(lane * 4);  // K table, this lane's copy
  const uint32_t vw_lane = (t_base + (uint32_t)Cfg::kVWOff) | (uint32_t)(lane * 4);
  using KBt = std::integral_constant<int, KB>;
  using VBt = std::integral_constant<int, VB>;
  auto win_hi = [&](auto bits_tag, const uint32_t* w, int j, uint32_t lane_base) -> uint32_t {
    constexpr int WB = decltype(bits_tag)::value;
    if constexpr (WB == 3) return lds32(win_addr<6>(w, j, lane_base));
    else if constexpr (WB == 2) return lds32(win_addr<4>(w, j, lane_base));
    else return __byte_perm(lds32(win_addr<5>(w, 2 * j, lane_base)), lds32(win_addr<5>(w, 2 * j + 1, lane_base)), 0x5410u);
  };
  // remainders: 3-bit pairs from their one-copy table, 2-bit pairs from the nibble table
  // (hi, lo) entries, 5-bit coordinates from the high halves of their own entries
  auto win_lo = [&](auto bits_tag, const uint32_t* w, int j, uint32_t lane_base, const unsigned char* lo3) -> uint32_t {
    constexpr int WB = decltype(bits_tag)::value;
    if constexpr (WB == 3) return ld32(lo3 + (win_field<6>(w, j) << 2));
    else if constexpr (WB == 2) return ld32(lutV2 + (win_field<4>(w, j) << 3) + 4);
    else return __byte_perm(lds32(win_addr<5>(w, 2 * j, lane_base)), lds32(win_addr<5>(w, 2 * j + 1, lane_base)), 0x7632u);
  };
  // V window of token row `row` for this lane (pairs [r D/16, (r + 1) D/16)), from bit 0
  auto v_window = [&](const unsigned char* row, uint32_t (&w)[5]) {
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = 0u;
    if (D == 64) {  // 8 VB bits from bit 8 VB r: two words hold them at any byte offset
      const int bit0 = 8 * VB * r;
      const int wi = bit0 >> 5;
      const uint32_t sh = (uint32_t)(bit0 & 31);
      const uint32_t x0 = ld32(row + wi * 4), x1 = ld32(row + wi * 4 + 4);
      w[0] = __funnelshift_r(x0, x1, sh);
      w[1] = x1 >> sh;
    } else if (D == 128) {
      constexpr int NL = (VB + 1) / 2;  // words spanning 16 VB bits from a half-word offset
      const int wi = (VB * r) >> 1;
      const uint32_t sh = 16u * (uint32_t)(r & 1);
      uint32_t x[NL];
#pragma unroll
      for (int i = 0; i < NL; ++i) x[i] = ld32(row + (wi + i) * 4);
#pragma unroll
      for (int i = 0; i + 1 < NL; ++i) w[i] = __funnelshift_r(x[i], x[i + 1], sh);
      w[NL - 1] = x[NL - 1] >> sh;
    } else {
#pragma unroll
      for (int i = 0; i < VB; ++i) w[i] = ld32(row + (VB * r + i) * 4);
    }
  };

  // K window of row `row` for this lane at D = 64 (pairs [8c, 8c + 8)): 16 KB bits from bit
  // 16 KB c, half-word aligned
  auto k_window64 = [&](const unsigned char* row, uint32_t (&w)[3]) {
    constexpr int NL = (KB + 1) / 2;
    const int wi = (KB * c) >> 1;
    const uint32_t sh = 16u * (uint32_t)(c & 1);
    uint32_t x[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) x[i] = ld32(row + (wi + i) * 4);
#pragma unroll
    for (int i = 0; i + 1 < NL; ++i) w[i] = __funnelshift_r(x[i], x[i + 1], sh);
    w[NL - 1] = x[NL - 1] >> sh;
#pragma unroll
    for (int i = NL; i < 3; ++i) w[i] = 0u;
  };

  // Query B fragments.  G = 4: one set whose columns 0-3 hold the fp16 hi part of the
  // rotated query and columns 4-7 (the unused half of the n = 8 MMA) its fp16 lo part,
  // so one MMA yields both products.  G = 8: separate hi and lo sets.
  constexpr int kQSets = G == 4 ? 1 : 2;
  uint32_t bq[kQSets][Cfg::kKSteps][2];
  uint32_t pq[kQSets][Cfg::kKSteps][2];  // product rows: p = S q~, same layout (unused otherwise)
  float qnorm_max = 0.f;  // max over this warp's heads of ||rotated query|| (log2 units)
  float o_acc[Cfg::kNT][Cfg::kMTiles][4];
  float m_run[2], l_run[2], m_thr[2];  // running max, sum, and max + kRescaleSlack per head
  int cur_b = -1;

  auto reset_state = [&]() {
#pragma unroll
    for (int nt = 0; nt < Cfg::kNT; ++nt)
#pragma unroll
      for (int i = 0; i < Cfg::kMTiles; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_acc[nt][i][e] = 0.f;
    m_run[0] = m_run[1] = m_thr[0] = m_thr[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
  };
  // Multiplies the value accumulators of each q head by its factor cv[e] (held by the
  // score-layout lanes: lane (r, c) has heads 2c, 2c+1; the value layout has head c + 4 nt).
  auto rescale_values = [&](const float (&cv)[2]) {
#pragma unroll
    for (int nt = 0; nt < Cfg::kNT; ++nt) {
      const int g = c + 4 * nt;
      const int srcl = (g >> 1) & 3;  // lane (r'=0, c'=g>>1)
      const float c0 = __shfl_sync(kFullMask, cv[0], srcl);
      const float c1 = __shfl_sync(kFullMask, cv[1], srcl);
      const float cg = (g & 1) ? c1 : c0;
#pragma unroll
      for (int i = 0; i < Cfg::kMTiles; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_acc[nt][i][e] *= cg;
    }
  };

  // B fragments from per-lane natural-order values x[g][i] (coordinate lane E + i of head g):
  // the fp16 hi / lo split of the pair order the K rows use.
  auto build_frags = [&](const float (&x)[G][D / 32], uint32_t (&frag)[kQSets][Cfg::kKSteps][2]) {
    constexpr int E = D / 32;
    const int gq = G == 4 ? (r & 3) : r;  // this lane's B column -> q head
#pragma unroll
    for (int s = 0; s < Cfg::kKSteps; ++s) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = 2 * s + u;
        const int jw = q / Cfg::kPWK, e = q % Cfg::kPWK;
        // pair index (coordinates 2p, 2p+1) of local pair u of k-step s on this lane column
        const int p = Cfg::kKWin ? (D / 8) * c + q : Cfg::kPWK * (c + 4 * jw) + e;
        const int src = (2 * p) / E;
        const int off = (2 * p) % E;  // identical on every lane (see the pair layout)
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float v0 = __shfl_sync(kFullMask, x[g][off], src);
          const float v1 = __shfl_sync(kFullMask, x[g][(off + 1) % E], E == 1 ? src + 1 : src);
          if (g == gq) {
            x0 = v0;
            x1 = v1;
          }
        }
        __half h0, l0, h1, l1;
        split_half(x0, h0, l0);
        split_half(x1, h1, l1);
        __half2 hh = __halves2half2(h0, h1), ll = __halves2half2(l0, l1);
        if (G == 4) {
          frag[0][s][u] = r < 4 ? *reinterpret_cast<uint32_t*>(&hh) : *reinterpret_cast<uint32_t*>(&ll);
        } else {
          frag[0][s][u] = *reinterpret_cast<uint32_t*>(&hh);
          frag[kQSets - 1][s][u] = *reinterpret_cast<uint32_t*>(&ll);
        }
      }
    }
  };

  // Rotated query of sequence b for this warp's G heads -> hi/lo B fragments.
  auto load_query = [&](int b) {
    constexpr int E = D / 32;
    float qr[G][E];
    qnorm_max = 0.f;
    // all G*E loads of this lane in flight at once (one dtype branch outside the loops)
    const int64_t base = ((int64_t)b * a.num_q_heads + (int64_t)h * G) * D + lane * E;
    if (a.q_dtype == kF16) {
      const __half* q16 = static_cast<const __half*>(a.q) + base;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < E; ++i) qr[g][i] = __half2float(q16[g * D + i]);
    } else if (a.q_dtype == kBF16) {
      const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q) + base;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < E; ++i) qr[g][i] = __bfloat162float(qb[g * D + i]);
    } else {
      const float* qf = static_cast<const float*>(a.q) + base;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < E; ++i) qr[g][i] = __ldg(qf + g * D + i);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int i = 0; i < E; ++i) qr[g][i] *= __ldg(a.signs + lane * E + i);
      fwht_warp<E>(qr[g]);
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        qr[g][i] *= qmul;
        ss = fmaf(qr[g][i], qr[g][i], ss);
        qr[g][i] *= inv_alpha_k;  // the K tables hold alpha * c
      }
      qnorm_max = fmaxf(qnorm_max, sqrtf(warp_sum(ss)));
    }
    build_frags(qr, bq);
    if constexpr (PROD) {  // p = S q~ of the same heads, into the sketch fragments
      // p is written by the projection grid this one may depend on programmatically: wait
      // for it (immediate once it has completed, or without such a launch), plain loads
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      const float* pb = args.p_all + base;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < E; ++i) qr[g][i] = pb[g * D + i];
      build_frags(qr, pq);
    }
  };

  const float inv_alpha = 1.0f / args.v_alpha;
  // Writes this warp's partial for sequence b (empty when `empty`).
  auto flush = [&](int b, bool empty) {
    const int64_t slot = (int64_t)cta + b;
    float lsum[2] = {l_run[0], l_run[1]};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      lsum[e] += __shfl_xor_sync(kFullMask, lsum[e], 4);
      lsum[e] += __shfl_xor_sync(kFullMask, lsum[e], 8);
      lsum[e] += __shfl_xor_sync(kFullMask, lsum[e], 16);
    }
    if (r == 0) {  // score layout: lane (r, c) holds q heads 2c, 2c+1
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int g = 2 * c + e;
        if (g < G) {
          float* ml = args.part_ml + (slot * a.num_q_heads + (int64_t)h * G + g) * 2;
          ml[0] = empty ? -INFINITY : m_run[e];
          ml[1] = empty ? 0.f : lsum[e];
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < Cfg::kNT; ++nt) {  // value layout: q head c + 4 nt
      const int g = c + 4 * nt;
      if (g < G) {
        float* acc = args.part_acc + (slot * a.num_q_heads + (int64_t)h * G + g) * D;
#pragma unroll
        for (int i = 0; i < Cfg::kMTiles; ++i) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int q = 2 * i + half;
            const int pv = Cfg::kVWin ? (D / 16) * r + q : Cfg::kPWV * (r + 8 * (q / Cfg::kPWV)) + (q % Cfg::kPWV);
            float2 v;
            v.x = empty ? 0.f : o_acc[nt][i][2 * half] * inv_alpha;
            v.y = empty ? 0.f : o_acc[nt][i][2 * half + 1] * inv_alpha;
            *reinterpret_cast<float2*>(acc + 2 * pv) = v;
          }
        }
      }
    }
  };

  // Move this warp to sequence b: close the current one and any non-empty sequences
  // of this CTA in between (they get empty partials), then load b's query.
  auto enter_sequence = [&](int b) {
    const int from = cur_b;
    if (from >= 0) flush(from, false);
    for (int x = (from < 0 ? b_first : from + 1); x < b; ++x)
      if (nblocks_of(x) > 0) flush(x, true);
    reset_state();
    cur_b = b;
    load_query(b);
  };

  // NTL (1 or 2) consecutive 16-token tiles of this warp's kv head in one sequence:
  // scores, one joint online-softmax update, values.  Only the last tile may be partial
  // (ntok_last tokens).  Two tiles give two independent lookup/MMA chains per phase.
  auto tiles = [&](auto ntl_tag, const unsigned char* kblk0, const unsigned char* kblk1, int ntok_last) {
    constexpr int NTL = decltype(ntl_tag)::value;
    const unsigned char* kbase[NTL];
    const unsigned char* vbase[NTL];
    kbase[0] = kblk0 + h * Cfg::kRBK;
    if (NTL == 2) kbase[NTL - 1] = kblk1 + h * Cfg::kRBK;
    float kn[NTL][2], vn[NTL][2];
    float kmax = 0.f;
#pragma unroll
    for (int t = 0; t < NTL; ++t) {
      vbase[t] = kbase[t] - h * Cfg::kRBK + args.k_slab_smem + h * Cfg::kRBV;
      kn[t][0] = __uint_as_float(ld32(kbase[t] + r * kts + Cfg::kKNormOff));
      kn[t][1] = __uint_as_float(ld32(kbase[t] + (r + 8) * kts + Cfg::kKNormOff));
      vn[t][0] = __uint_as_float(ld32(vbase[t] + r * vts + Cfg::kWV * 4));
      vn[t][1] = __uint_as_float(ld32(vbase[t] + (r + 8) * vts + Cfg::kWV * 4));
      kmax = fmaxf(kmax, fmaxf(fabsf(kn[t][0]), fabsf(kn[t][1])));
    }
    // Rows past the sequence end hold stale bytes (a NaN norm, say): their value norm is 0
    // before any arithmetic sees it (their scores are masked below).
    if (ntok_last < kBS) {
      if (r >= ntok_last) vn[NTL - 1][0] = 0.f;
      if (r + 8 >= ntok_last) vn[NTL - 1][1] = 0.f;
    }
    float vmax = 0.f;
#pragma unroll
    for (int t = 0; t < NTL; ++t) vmax = fmaxf(vmax, fmaxf(vn[t][0], vn[t][1]));
    // Precision switch: tiles whose largest |score| bound nu_k * ||q|| stays within
    // kFastScoreBound take the fp16-hi key path (rounding error ~1e-4 relative after the
    // alpha scaling); otherwise (large-norm rows), and in every exact-value tile, the
    // fp16-lo key part is added as well.  Stale rows past the sequence end can only select
    // the exact path, which is correct for any tile.  One vote in the common case.
    const bool pv = vmax > kFastValueNorm;
    bool exact = false, exact_v = false;
    if (__any_sync(kFullMask, pv || kmax * qnorm_max > kFastScoreBound)) {
      exact = true;
      exact_v = __any_sync(kFullMask, pv);
    }
    float sacc[NTL][4];
#pragma unroll
    for (int t = 0; t < NTL; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[t][e] = 0.f;
    if (!exact) {
      // G = 4: columns 0-3 get key_hi * q_hi, 4-7 key_hi * q_lo; each tile runs its even and
      // odd k-steps as two chains.  G = 8: a q_lo chain per tile.
      float sacc1[NTL][4];
#pragma unroll
      for (int t = 0; t < NTL; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc1[t][e] = 0.f;
      auto kstep = [&](int t, int s, uint32_t h00, uint32_t h10, uint32_t h01, uint32_t h11) {
        if (G == 8) {
          mma16816(sacc[t], h00, h10, h01, h11, bq[0][s][0], bq[0][s][1]);
          mma16816(sacc1[t], h00, h10, h01, h11, bq[kQSets - 1][s][0], bq[kQSets - 1][s][1]);
        } else {
          mma16816((s & 1) ? sacc1[t] : sacc[t], h00, h10, h01, h11, bq[0][s][0], bq[0][s][1]);
        }
      };
      if constexpr (Cfg::kKWin && D == 64) {
        uint32_t w0[NTL][3], w1[NTL][3];
#pragma unroll
        for (int t = 0; t < NTL; ++t) {
          k_window64(kbase[t] + r * kts, w0[t]);
          k_window64(kbase[t] + (r + 8) * kts, w1[t]);
        }
#pragma unroll
        for (int s8 = 0; s8 < 4; ++s8)
#pragma unroll
          for (int t = 0; t < NTL; ++t)
            kstep(t, s8, win_hi(KBt{}, w0[t], 2 * s8, kw_lane), win_hi(KBt{}, w1[t], 2 * s8, kw_lane),
                  win_hi(KBt{}, w0[t], 2 * s8 + 1, kw_lane), win_hi(KBt{}, w1[t], 2 * s8 + 1, kw_lane));
      } else if constexpr (Cfg::kKWin) {
        // chunks of KB words of this lane's window: 16 pairs, 8 k-steps each
#pragma unroll
        for (int ch = 0; ch < D / 128; ++ch) {
          uint32_t w0[NTL][KB], w1[NTL][KB];
#pragma unroll
          for (int t = 0; t < NTL; ++t)
#pragma unroll
            for (int i = 0; i < KB; ++i) {
              w0[t][i] = ld32(kbase[t] + r * kts + (Cfg::kKLaneWords * c + KB * ch + i) * 4);
              w1[t][i] = ld32(kbase[t] + (r + 8) * kts + (Cfg::kKLaneWords * c + KB * ch + i) * 4);
            }
#pragma unroll
          for (int s8 = 0; s8 < 8; ++s8)
#pragma unroll
            for (int t = 0; t < NTL; ++t)
              kstep(t, 8 * ch + s8, win_hi(KBt{}, w0[t], 2 * s8, kw_lane), win_hi(KBt{}, w1[t], 2 * s8, kw_lane),
                    win_hi(KBt{}, w0[t], 2 * s8 + 1, kw_lane), win_hi(KBt{}, w1[t], 2 * s8 + 1, kw_lane));
        }
      } else {
#pragma unroll
        for (int jw = 0; jw < Cfg::kWK / 4; ++jw) {
          uint32_t w0[NTL], w1[NTL];
#pragma unroll
          for (int t = 0; t < NTL; ++t) {
            w0[t] = ld32(kbase[t] + r * kts + (c + 4 * jw) * 4);
            w1[t] = ld32(kbase[t] + (r + 8) * kts + (c + 4 * jw) * 4);
          }
#pragma unroll
          for (int e2 = 0; e2 < Cfg::kPWK; e2 += 2) {
            const int s = (jw * Cfg::kPWK + e2) >> 1;
#pragma unroll
            for (int t = 0; t < NTL; ++t)
              kstep(t, s, k_hi(w0[t], e2), k_hi(w1[t], e2), k_hi(w0[t], e2 + 1), k_hi(w1[t], e2 + 1));
          }
        }
      }
      // G = 8: sacc1 holds key_hi * q_lo (q_lo scaled by 2^12); G = 4: the odd k-steps, same
      // column scales as sacc
#pragma unroll
      for (int t = 0; t < NTL; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[t][e] = G == 8 ? fmaf(sacc1[t][e], kLoUnscale, sacc[t][e]) : sacc[t][e] + sacc1[t][e];
    } else {
      // adds key_lo * q_hi (G = 4: key_lo * [q_hi | q_lo])
#pragma unroll
      for (int t = 0; t < NTL; ++t) {
        float sacc1[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
        auto kstep_ex = [&](int s, uint32_t h00, uint32_t h10, uint32_t h01, uint32_t h11, uint32_t l00,
                            uint32_t l10, uint32_t l01, uint32_t l11) {
          mma16816(sacc[t], h00, h10, h01, h11, bq[0][s][0], bq[0][s][1]);
          if (G == 8) mma16816(sacc1, h00, h10, h01, h11, bq[kQSets - 1][s][0], bq[kQSets - 1][s][1]);
          mma16816(sacc2, l00, l10, l01, l11, bq[0][s][0], bq[0][s][1]);
        };
        if constexpr (Cfg::kKWin && D == 64) {
          uint32_t w0[3], w1[3];
          k_window64(kbase[t] + r * kts, w0);
          k_window64(kbase[t] + (r + 8) * kts, w1);
#pragma unroll
          for (int s8 = 0; s8 < 4; ++s8) {
            const int j0 = 2 * s8, j1 = 2 * s8 + 1;
            kstep_ex(s8, win_hi(KBt{}, w0, j0, kw_lane), win_hi(KBt{}, w1, j0, kw_lane),
                     win_hi(KBt{}, w0, j1, kw_lane), win_hi(KBt{}, w1, j1, kw_lane),
                     win_lo(KBt{}, w0, j0, kw_lane, lutK3L), win_lo(KBt{}, w1, j0, kw_lane, lutK3L),
                     win_lo(KBt{}, w0, j1, kw_lane, lutK3L), win_lo(KBt{}, w1, j1, kw_lane, lutK3L));
          }
        } else if constexpr (Cfg::kKWin) {
#pragma unroll
          for (int ch = 0; ch < D / 128; ++ch) {
            uint32_t w0[KB], w1[KB];
#pragma unroll
            for (int i = 0; i < KB; ++i) {
              w0[i] = ld32(kbase[t] + r * kts + (Cfg::kKLaneWords * c + KB * ch + i) * 4);
              w1[i] = ld32(kbase[t] + (r + 8) * kts + (Cfg::kKLaneWords * c + KB * ch + i) * 4);
            }
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8) {
              const int j0 = 2 * s8, j1 = 2 * s8 + 1;
              kstep_ex(8 * ch + s8, win_hi(KBt{}, w0, j0, kw_lane), win_hi(KBt{}, w1, j0, kw_lane),
                       win_hi(KBt{}, w0, j1, kw_lane), win_hi(KBt{}, w1, j1, kw_lane),
                       win_lo(KBt{}, w0, j0, kw_lane, lutK3L), win_lo(KBt{}, w1, j0, kw_lane, lutK3L),
                       win_lo(KBt{}, w0, j1, kw_lane, lutK3L), win_lo(KBt{}, w1, j1, kw_lane, lutK3L));
            }
          }
        } else {
#pragma unroll
          for (int jw = 0; jw < Cfg::kWK / 4; ++jw) {
            const uint32_t w0 = ld32(kbase[t] + r * kts + (c + 4 * jw) * 4);
            const uint32_t w1 = ld32(kbase[t] + (r + 8) * kts + (c + 4 * jw) * 4);
#pragma unroll
            for (int e2 = 0; e2 < Cfg::kPWK; e2 += 2)
              kstep_ex((jw * Cfg::kPWK + e2) >> 1, k_hi(w0, e2), k_hi(w1, e2), k_hi(w0, e2 + 1), k_hi(w1, e2 + 1),
                       k_lo(w0, e2), k_lo(w1, e2), k_lo(w0, e2 + 1), k_lo(w1, e2 + 1));
          }
        }
        // sacc1 (key_hi * q_lo) and sacc2 (key_lo * q) each carry one 2^12 scale
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[t][e] = fmaf(sacc1[e] + sacc2[e], kLoUnscale, sacc[t][e]);
      }
    }
    if constexpr (PROD) {
      // sketch term of product rows: gamma kappa <p, 2 z - 1>.  The A operand is the +-1 pairs
      // of the row's sign bits (the nibble of k-step s holds both pairs of the lane), the B
      // operand p = S q~ split like the query; added to the MSE score before the fold (for
      // G = 4 the p_lo columns carry the same 2^12 as the q_lo ones).
      const uint32_t sgn_lane = (t_base + (uint32_t)Cfg::kSgnOff) | (uint32_t)(lane * 8);
      auto sign_pairs = [&](const unsigned char* row, int s) -> uint2 {
        const int q = 2 * s, jw = q / Cfg::kPWK, e = q % Cfg::kPWK;
        const int bo = 2 * (Cfg::kKWin ? (D / 8) * c + q : Cfg::kPWK * (c + 4 * jw) + e);  // first sign bit
        const uint32_t w = ld32(row + Cfg::kSignOff + (bo >> 5) * 4);
        return lds64(sgn_lane | (((w >> (bo & 31)) & 15u) << 8));
      };
#pragma unroll
      for (int t = 0; t < NTL; ++t) {
        float z0[4] = {0.f, 0.f, 0.f, 0.f}, z1[4] = {0.f, 0.f, 0.f, 0.f};
        const unsigned char* ra = kbase[t] + r * kts;
        const unsigned char* rb = kbase[t] + (r + 8) * kts;
        const float g0 = __uint_as_float(ld32(ra + Cfg::kKNormOff + 4)) * args.sketch;
        const float g1 = __uint_as_float(ld32(rb + Cfg::kKNormOff + 4)) * args.sketch;
#pragma unroll
        for (int s = 0; s < Cfg::kKSteps; ++s) {
          const uint2 za = sign_pairs(ra, s), zb = sign_pairs(rb, s);
          mma16816(z0, za.x, zb.x, za.y, zb.y, pq[0][s][0], pq[0][s][1]);
          if (G == 8) mma16816(z1, za.x, zb.x, za.y, zb.y, pq[kQSets - 1][s][0], pq[kQSets - 1][s][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float zz = G == 8 ? fmaf(z1[e], kLoUnscale, z0[e]) : z0[e];  // G = 8: z1 holds p_lo x 2^12
          sacc[t][e] = fmaf(e < 2 ? g0 : g1, zz, sacc[t][e]);
        }
      }
    }
    float sc[NTL][4];
#pragma unroll
    for (int t = 0; t < NTL; ++t) {
      if (G == 4) {
        // fold the q_lo columns (lanes c = 2, 3; q_lo scaled by 2^12) onto the q_hi columns
        // (lanes c = 0, 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[t][e] = fmaf(__shfl_xor_sync(kFullMask, sacc[t][e], 2), kLoUnscale, sacc[t][e]);
      }
      sc[t][0] = sacc[t][0] * kn[t][0];
      sc[t][1] = sacc[t][1] * kn[t][0];
      sc[t][2] = sacc[t][2] * kn[t][1];
      sc[t][3] = sacc[t][3] * kn[t][1];
    }
    if (ntok_last < kBS) {  // last block of a sequence: mask the rows past its end
      if (r >= ntok_last) sc[NTL - 1][0] = sc[NTL - 1][1] = -INFINITY;
      if (r + 8 >= ntok_last) sc[NTL - 1][2] = sc[NTL - 1][3] = -INFINITY;
    }

    // --- online softmax (q heads 2c, 2c+1 on this lane).  The running max only moves
    // when a score passes it by more than kRescaleSlack, so p = 2^(s - m) <= 2^slack.
    // Most tiles move no max: one compare per score and a vote replace the reduction.
    float smax[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      smax[e] = fmaxf(sc[0][e], sc[0][2 + e]);
#pragma unroll
      for (int t = 1; t < NTL; ++t) smax[e] = fmaxf(smax[e], fmaxf(sc[t][e], sc[t][2 + e]));
    }
    if (__any_sync(kFullMask, smax[0] > m_thr[0] || smax[1] > m_thr[1])) {
      float corr[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mt = smax[e];
        mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 16));
        const float mn = mt > m_thr[e] ? mt : m_run[e];
        corr[e] = m_run[e] == mn ? 1.f : fast_exp2(m_run[e] - mn);
        l_run[e] *= corr[e];
        m_run[e] = mn;
        m_thr[e] = mn + kRescaleSlack;
      }
      rescale_values(corr);
    }
    float pvf[NTL][4];  // P' = p nu_v: [t][e] token r, [t][2 + e] token r + 8 (heads 2c, 2c+1)
#pragma unroll
    for (int t = 0; t < NTL; ++t) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p0 = fast_exp2(sc[t][e] - m_run[e]), p1 = fast_exp2(sc[t][2 + e] - m_run[e]);
        l_run[e] += p0 + p1;
        pvf[t][e] = p0 * vn[t][0];
        pvf[t][2 + e] = p1 * vn[t][1];
      }
    }

    // --- values ------------------------------------------------------------------------
    // EXV: tiles with a value norm above kFastValueNorm add the fp16 remainders of the
    // table entries and of P'.
    auto values = [&](auto exv_tag) {
      constexpr bool EXV = decltype(exv_tag)::value;
      // EXV: q = fp16 remainders of P' (P'_lo), u = P' 2^-12 (pairs with the V_lo entries,
      // which carry 2^12)
      uint32_t p01[NTL], p23[NTL], q01[NTL], q23[NTL], u01[NTL], u23[NTL];
#pragma unroll
      for (int t = 0; t < NTL; ++t) {
        p01[t] = pack_half2(pvf[t][0], pvf[t][1]);  // token r:   heads 2c, 2c+1
        p23[t] = pack_half2(pvf[t][2], pvf[t][3]);  // token r+8: heads 2c, 2c+1
        if (EXV) {
          const __half2 h01 = *reinterpret_cast<const __half2*>(&p01[t]);
          const __half2 h23 = *reinterpret_cast<const __half2*>(&p23[t]);
          q01[t] = pack_half2(pvf[t][0] - __low2float(h01), pvf[t][1] - __high2float(h01));
          q23[t] = pack_half2(pvf[t][2] - __low2float(h23), pvf[t][3] - __high2float(h23));
          u01[t] = pack_half2(pvf[t][0] * kLoUnscale, pvf[t][1] * kLoUnscale);
          u23[t] = pack_half2(pvf[t][2] * kLoUnscale, pvf[t][3] * kLoUnscale);
        }
      }
#pragma unroll
      for (int t = 0; t < NTL; ++t) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {  // tokens {c, c+4} (ks=0) and {c+8, c+12} (ks=1)
          const int t0 = c + 8 * ks, t1 = c + 4 + 8 * ks;
          uint32_t bv[Cfg::kNT][2], bl[Cfg::kNT][2], bu[Cfg::kNT][2];
#pragma unroll
          for (int nt = 0; nt < Cfg::kNT; ++nt) {
            const int cs = 2 * nt + (r >> 2);  // source lane column: q head (4 nt + r/2) / 2
            const uint32_t src = ks == 0 ? p01[t] : p23[t];
            const uint32_t x0 = __shfl_sync(kFullMask, src, 4 * c + cs);
            const uint32_t x1 = __shfl_sync(kFullMask, src, 4 * (c + 4) + cs);
            bv[nt][0] = __byte_perm(x0, 0u, sel_b);
            bv[nt][1] = __byte_perm(x1, 0u, sel_b);
            if (EXV) {
              const uint32_t srcl = ks == 0 ? q01[t] : q23[t];
              const uint32_t y0 = __shfl_sync(kFullMask, srcl, 4 * c + cs);
              const uint32_t y1 = __shfl_sync(kFullMask, srcl, 4 * (c + 4) + cs);
              bl[nt][0] = __byte_perm(y0, 0u, sel_b);
              bl[nt][1] = __byte_perm(y1, 0u, sel_b);
              const uint32_t srcu = ks == 0 ? u01[t] : u23[t];
              const uint32_t z0 = __shfl_sync(kFullMask, srcu, 4 * c + cs);
              const uint32_t z1 = __shfl_sync(kFullMask, srcu, 4 * (c + 4) + cs);
              bu[nt][0] = __byte_perm(z0, 0u, sel_b);
              bu[nt][1] = __byte_perm(z1, 0u, sel_b);
            }
          }
          // m-tile i: the A fragment (pairs q = 2i (row r), 2i+1 (row r+8) of tokens t0, t1)
          auto vstep = [&](int i, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t l0, uint32_t l1,
                           uint32_t l2, uint32_t l3) {
#pragma unroll
            for (int nt = 0; nt < Cfg::kNT; ++nt) mma16816(o_acc[nt][i], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
            if (EXV) {
#pragma unroll
              for (int nt = 0; nt < Cfg::kNT; ++nt) {
                mma16816(o_acc[nt][i], l0, l1, l2, l3, bu[nt][0], bu[nt][1]);  // V_lo 2^12 * P' 2^-12
                mma16816(o_acc[nt][i], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);  // V_hi * P'_lo
              }
            }
          };
          if constexpr (Cfg::kVWin) {
            uint32_t wa[5], wb[5];
            v_window(vbase[t] + t0 * vts, wa);
            v_window(vbase[t] + t1 * vts, wb);
#pragma unroll
            for (int i = 0; i < Cfg::kMTiles; ++i) {
              const int j0 = 2 * i, j1 = 2 * i + 1;
              // the remainder lookups are dead code (and dropped) unless EXV
              vstep(i, win_hi(VBt{}, wa, j0, vw_lane), win_hi(VBt{}, wa, j1, vw_lane), win_hi(VBt{}, wb, j0, vw_lane),
                    win_hi(VBt{}, wb, j1, vw_lane), win_lo(VBt{}, wa, j0, vw_lane, lutV3L),
                    win_lo(VBt{}, wa, j1, vw_lane, lutV3L), win_lo(VBt{}, wb, j0, vw_lane, lutV3L),
                    win_lo(VBt{}, wb, j1, vw_lane, lutV3L));
            }
          } else {
#pragma unroll
            for (int jw = 0; jw < Cfg::kWV / 8; ++jw) {
              const uint32_t wa = ld32(vbase[t] + t0 * vts + (r + 8 * jw) * 4);
              const uint32_t wb = ld32(vbase[t] + t1 * vts + (r + 8 * jw) * 4);
#pragma unroll
              for (int e = 0; e < Cfg::kPWV; e += 2)
                vstep((jw * Cfg::kPWV + e) >> 1, v_lookup(wa, e), v_lookup(wa, e + 1), v_lookup(wb, e),
                      v_lookup(wb, e + 1), v_lookup_lo(wa, e), v_lookup_lo(wa, e + 1), v_lookup_lo(wb, e),
                      v_lookup_lo(wb, e + 1));
            }
          }
        }
      }
    };
    if (exact_v) {
      // per q head, scale the weights so that the largest lands in [2^11, 2^12) and the
      // accumulators by the same power of two, exactly; undone after the tile
      float f[2], inv_f[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float pm = 0.f;
#pragma unroll
        for (int t = 0; t < NTL; ++t) pm = fmaxf(pm, fmaxf(pvf[t][e], pvf[t][2 + e]));
        pm = fmaxf(pm, __shfl_xor_sync(kFullMask, pm, 4));
        pm = fmaxf(pm, __shfl_xor_sync(kFullMask, pm, 8));
        pm = fmaxf(pm, __shfl_xor_sync(kFullMask, pm, 16));
        tile_scale(pm, f[e], inv_f[e]);
#pragma unroll
        for (int t = 0; t < NTL; ++t) {
          pvf[t][e] *= f[e];
          pvf[t][2 + e] *= f[e];
        }
      }
      rescale_values(f);
      values(std::true_type{});
      rescale_values(inv_f);
    } else {
      values(std::false_type{});
    }
  };
  using One = std::integral_constant<int, 1>;
  using Two = std::integral_constant<int, 2>;

  // ---- main pipeline -----------------------------------------------------------------
  // Stage st lives in ring slot st % nst; full[slot] completes when its copies landed,
  // empty[slot] when every consumer warp is done with it.
  if (producer) {
    int S = 0;
    for (; S < nstages; ++S) {
      const int ps = S % nst;
      if (S >= nst && !mbar_wait(bar_empty(ps), (uint32_t)(((S / nst) - 1) & 1), args.wait_tries)) break;
      if (S == 0 && lane < WPH) meta_load();
      produce(ps);
    }
    if (S < nstages && lane == 0 && a.status) atomicMax(a.status, (int32_t)kTimeout);
    // let this CTA's copies land before the producer leaves (the consumers normally
    // have already waited for all of them)
    for (int s2 = (S > nst ? S - nst : 0); s2 < S; ++s2)
      mbar_wait(bar_full(s2 % nst), (uint32_t)((s2 / nst) & 1), kDefaultWaitTries);
    return;
  }
  {
      // ---- tables (consumer warps; the producer is already streaming) ------------------
    if (KB == 4) {
      // lane k of every consumer warp splits centroid k once; the entries then take their
      // two halves with shuffles instead of global loads in the loop
      __half k_hi_l, k_lo_l;
      split_half(__ldg(a.k_centroids + (lane & 15)) * args.k_alpha, k_hi_l, k_lo_l);
      const uint32_t k_pair_l = (uint32_t)__half_as_ushort(k_hi_l) | ((uint32_t)__half_as_ushort(k_lo_l) << 16);
      for (int i = tid; i < 256 * 32; i += 32 * ncons) {
        const int f = i >> 5, copy = i & 31;
        const uint32_t pa = __shfl_sync(kFullMask, k_pair_l, f & 15);  // (hi, lo) of c[f & 15]
        const uint32_t pb = __shfl_sync(kFullMask, k_pair_l, f >> 4);
        *reinterpret_cast<uint32_t*>(lutT + f * 256 + copy * 4) = __byte_perm(pa, pb, 0x5410);
        if (copy == 0) *reinterpret_cast<uint32_t*>(lutL + f * 4) = __byte_perm(pa, pb, 0x7632);
      }
    } else if (KB == 2) {
      for (int f = tid; f < 16; f += 32 * ncons) {
        __half ha, la, hb, lb;
        split_half(__ldg(a.k_centroids + (f & 3)) * args.k_alpha, ha, la);
        split_half(__ldg(a.k_centroids + (f >> 2)) * args.k_alpha, hb, lb);
        __half2 hi2 = __halves2half2(ha, hb), lo2 = __halves2half2(la, lb);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t*>(&hi2);
        v.y = *reinterpret_cast<uint32_t*>(&lo2);
        *reinterpret_cast<uint2*>(lutK2 + f * 8) = v;
      }
    }
    if (VB == 4) {
      __half v_hi_l, v_lo_l;
      split_half(__ldg(a.v_centroids + (lane & 15)) * args.v_alpha, v_hi_l, v_lo_l);
      const uint32_t v_pair_l = (uint32_t)__half_as_ushort(v_hi_l) | ((uint32_t)__half_as_ushort(v_lo_l) << 16);
      for (int i = tid; i < 256 * 32; i += 32 * ncons) {
        const int f = i >> 5, copy = i & 31;
        const uint32_t pa = __shfl_sync(kFullMask, v_pair_l, f & 15);  // (hi, lo) of c[f & 15]
        const uint32_t pb = __shfl_sync(kFullMask, v_pair_l, f >> 4);
        *reinterpret_cast<uint32_t*>(lutT + f * 256 + 128 + copy * 4) = __byte_perm(pa, pb, 0x5410);
        if (copy == 0) *reinterpret_cast<uint32_t*>(lutVL + f * 4) = __byte_perm(pa, pb, 0x7632);
      }
    } else if (VB == 2) {
      for (int f = tid; f < 16; f += 32 * ncons) {
        __half ha, la, hb, lb;
        split_half(__ldg(a.v_centroids + (f & 3)) * args.v_alpha, ha, la);
        split_half(__ldg(a.v_centroids + (f >> 2)) * args.v_alpha, hb, lb);
        __half2 hi2 = __halves2half2(ha, hb), lo2 = __halves2half2(la, lb);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t*>(&hi2);
        v.y = *reinterpret_cast<uint32_t*>(&lo2);
        *reinterpret_cast<uint2*>(lutV2 + f * 8) = v;
      }
    }
    if constexpr (Cfg::kKWin || Cfg::kVWin) {
      // window-mode tables, one copy per lane.  3-bit: entry f = the fp16 hi parts of
      // (c[f & 7], c[f >> 3]), their remainders (x 2^12) in one copy.  5-bit: entry e =
      // (fp16 hi, fp16 lo x 2^12) of c[e].
#pragma unroll
      for (int comp = 0; comp < 2; ++comp) {
        const int cb = comp == 0 ? KB : VB;
        if ((comp == 0 && !Cfg::kKWin) || (comp == 1 && !Cfg::kVWin)) continue;
        const float* cents = comp == 0 ? a.k_centroids : a.v_centroids;
        const float alpha = comp == 0 ? args.k_alpha : args.v_alpha;
        unsigned char* tab = comp == 0 ? lutKW : lutVW;
        unsigned char* tlo = comp == 0 ? lutK3L : lutV3L;
        __half hi_l, lo_l;
        split_half(__ldg(cents + (lane & (cb == 3 ? 7 : (cb == 2 ? 3 : 31)))) * alpha, hi_l, lo_l);
        const uint32_t pair_l = (uint32_t)__half_as_ushort(hi_l) | ((uint32_t)__half_as_ushort(lo_l) << 16);
        for (int i = tid; i < (cb == 3 ? 64 : (cb == 2 ? 16 : 32)) * 32; i += 32 * ncons) {
          const int f = i >> 5, copy = i & 31;
          if (cb == 2) {  // entry f = the fp16 hi parts of (c[f & 3], c[f >> 2]); remainders in lutV2
            const uint32_t pa = __shfl_sync(kFullMask, pair_l, f & 3);
            const uint32_t pb = __shfl_sync(kFullMask, pair_l, f >> 2);
            *reinterpret_cast<uint32_t*>(tab + f * 128 + copy * 4) = __byte_perm(pa, pb, 0x5410);
          } else if (cb == 3) {
            const uint32_t pa = __shfl_sync(kFullMask, pair_l, f & 7);  // (hi, lo) of c[f & 7]
            const uint32_t pb = __shfl_sync(kFullMask, pair_l, f >> 3);
            *reinterpret_cast<uint32_t*>(tab + f * 128 + copy * 4) = __byte_perm(pa, pb, 0x5410);
            if (copy == 0) *reinterpret_cast<uint32_t*>(tlo + f * 4) = __byte_perm(pa, pb, 0x7632);
          } else {
            *reinterpret_cast<uint32_t*>(tab + f * 128 + copy * 4) = __shfl_sync(kFullMask, pair_l, f);
          }
        }
      }
    }
    if constexpr (PROD) {  // sign table: entry n = (+-1, +-1), (+-1, +-1) of the 4 bits of n
      unsigned char* sg = smem + args.t_off + Cfg::kSgnOff;
      for (int i = tid; i < 16 * 32; i += 32 * ncons) {
        const int n = i >> 5, copy = i & 31;
        uint2 v;
        v.x = ((n & 1) ? 0x3C00u : 0xBC00u) | (((n & 2) ? 0x3C00u : 0xBC00u) << 16);
        v.y = ((n & 4) ? 0x3C00u : 0xBC00u) | (((n & 8) ? 0x3C00u : 0xBC00u) << 16);
        *reinterpret_cast<uint2*>(sg + n * 256 + copy * 8) = v;
      }
    }
  asm volatile("bar.sync 1, %0;\n" ::"r"(32 * ncons) : "memory");  // consumer warps only
  }
  // the first block belongs to b_first: its query is read while the first copies land
  reset_state();
  cur_b = b_first;
  load_query(b_first);
  int slot = 0;
  uint32_t par = 0;
  for (int st = 0; st < nstages; ++st) {
    if (!mbar_wait(bar_full(slot), par, args.wait_tries)) {
      if (lane == 0 && a.status) atomicMax(a.status, (int32_t)kTimeout);
      return;
    }
    const BlockMeta m0 = meta[slot * WPH];
    const BlockMeta m1 = meta[slot * WPH + WPH - 1];
    if (WPH == 2 && m0.ntok == kBS && m0.valid && m1.ntok != 0 && m1.valid && m1.b == m0.b) {
      if (m0.b != cur_b) enter_sequence(m0.b);
      tiles(Two{}, smem + buf_off(slot, 0), smem + buf_off(slot, 1), m1.ntok);
    } else {
#pragma unroll
      for (int u = 0; u < WPH; ++u) {
        const BlockMeta m = u == 0 ? m0 : m1;
        if (m.ntok != 0) {
          if (m.b != cur_b) enter_sequence(m.b);
          if (m.valid) tiles(One{}, smem + buf_off(slot, u), nullptr, m.ntok);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty(slot));
    if (++slot == nst) {
      slot = 0;
      par ^= 1u;
    }
  }
  // close the last sequence and any later non-empty ones this CTA owns
  if (cur_b < 0) {
    for (int x = b_first; x <= b_last; ++x)
      if (nblocks_of(x) > 0) flush(x, true);
  } else {
    flush(cur_b, false);
    for (int x = cur_b + 1; x <= b_last; ++x)
      if (nblocks_of(x) > 0) flush(x, true);
  }
}

// One warp per (sequence, q head): merge the partials of the CTAs that touched the
// sequence, normalise, apply R^T (FWHT + sign flip) and store.  The (m, l) and the
// accumulator of up to kCombineBatch partials are loaded together (one round trip);
// longer spans loop over batches with a running rescale.
constexpr int kCombineBatch = 4;

template <int E>
__global__ void __launch_bounds__(256)
combine_tc_kernel(DecodeArgs a, int num_ctas, const float* __restrict__ part_acc, const float* __restrict__ part_ml,
                  const int* __restrict__ prefix) {
  constexpr int D = 32 * E;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // launched as a programmatic dependent of the split kernel: wait until that grid has
  // completed and its partials are visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (row >= a.batch * a.num_q_heads) return;
  const int b = row / a.num_q_heads, j = row - b * a.num_q_heads;
  const long long N = prefix[a.batch];
  const long long p0 = prefix[b], p1 = prefix[b + 1];
  float v[E];
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = 0.f;
  if (p1 > p0) {
    const long long C = num_ctas;
    // CTA i owns blocks [N i / C, N (i + 1) / C); block g belongs to CTA ((g + 1) C - 1) / N.
    // With N >= C every CTA from the owner of p0 to the owner of p1 - 1 wrote a partial for
    // this sequence; with N < C some ranges are empty, and the writers are exactly the
    // owners of the sequence's blocks, one each.
    const bool dense = N >= C;
    const long long f = ((p0 + 1) * C - 1) / N, l = (p1 * C - 1) / N;  // first / last CTA
    const long long cnt = dense ? l - f + 1 : p1 - p0;                  // partials to merge
    float mx = -INFINITY, lsum = 0.f;
    for (long long k0 = 0; k0 < cnt; k0 += kCombineBatch) {
      float ms[kCombineBatch], ls[kCombineBatch], acc[kCombineBatch][E];
#pragma unroll
      for (int u = 0; u < kCombineBatch; ++u) {
        const long long k = k0 + u;
        const bool live = k < cnt;
        const long long i = !live ? 0 : (dense ? f + k : ((p0 + k + 1) * C - 1) / N);
        const int64_t s = (i + b) * a.num_q_heads + j;
        ms[u] = live ? part_ml[s * 2] : -INFINITY;
        ls[u] = live ? part_ml[s * 2 + 1] : 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k) acc[u][k] = live ? part_acc[s * D + lane * E + k] : 0.f;
      }
      float bm = mx;
#pragma unroll
      for (int u = 0; u < kCombineBatch; ++u) bm = fmaxf(bm, ms[u]);
      const float cr = mx == -INFINITY ? 0.f : exp2f(mx - bm);  // rescale of what came before
      lsum *= cr;
#pragma unroll
      for (int k = 0; k < E; ++k) v[k] *= cr;
#pragma unroll
      for (int u = 0; u < kCombineBatch; ++u) {
        const float w = ms[u] == -INFINITY ? 0.f : exp2f(ms[u] - bm);
        lsum = fmaf(w, ls[u], lsum);
#pragma unroll
        for (int k = 0; k < E; ++k) v[k] = fmaf(w, acc[u][k], v[k]);
      }
      mx = bm;
    }
    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) v[k] *= inv;
  }
  fwht_warp<E>(v);
  const float rs = 1.0f / sqrtf((float)D);
#pragma unroll
  for (int k = 0; k < E; ++k)
    store_from_f32(a.out, (int64_t)row * D + lane * E + k, a.out_dtype, v[k] * __ldg(a.signs + lane * E + k) * rs);
}

template <int D, int KB, int VB, int G, int WPH, bool PROD = false>
cudaError_t launch_tc_typed(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream,
                            const float* p_all = nullptr) {
  using Cfg = TcCfg<D, KB, VB, G, WPH, PROD>;
  TcArgs t{};
  t.a = a;
  t.num_ctas = p.num_splits;
  const int H = a.num_kv_heads;
  const int kraw = H * Cfg::kRBK, vraw = H * Cfg::kRBV;
  // Each K and V slab arrives as one bulk copy, unpadded.  (Per-token row copies would
  // allow padded, conflict-free strides, but many small bulk copies do not keep enough
  // bytes in flight; for 8 heads of 128 4-bit coordinates the unpadded K stride costs a
  // 2-way conflict on the 8 index-word loads of a tile, the V stride none.)
  t.k_row_copy = 0;
  t.v_row_copy = 0;
  t.k_tok_stride = kraw;
  t.v_tok_stride = vraw;
  t.k_slab_smem = (kBS * t.k_tok_stride + 15) / 16 * 16;
  t.v_slab_smem = (kBS * t.v_tok_stride + 15) / 16 * 16;
  t.v_alpha = a.v_alpha > 0.f ? a.v_alpha : 1.0f;
  t.k_alpha = a.k_alpha > 0.f ? a.k_alpha : 1.0f;
  t.wait_tries = wait_tries();

  // Shared-memory layout: [misc | buffers ... | table region (T: 64 KB at a 64 KB aligned
  // shared address; 3-bit pair tables: 16 KB at an 8 KB aligned one) | buffers ...].  Dynamic shared memory starts right after the per-block
  // reserved bytes in the shared window (the kernel checks the T alignment it gets).
  int dev = 0, reserved = 0, max_dyn = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&max_dyn, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  t.buf_bytes = (t.k_slab_smem + t.v_slab_smem + 127) / 128 * 128;
  int total_bufs = 0;
  t.buf_lo = kMiscBytes;
  if (Cfg::kTBytes > 0) {
    int t_off = (Cfg::kTAlign - reserved % Cfg::kTAlign) % Cfg::kTAlign;
    while (t_off < kMiscBytes) t_off += Cfg::kTAlign;
    t.t_off = t_off;
    t.n_lo = (t_off - kMiscBytes) / t.buf_bytes;
    t.buf_hi = t_off + Cfg::kTBytes;
    total_bufs = t.n_lo + std::max(0, (max_dyn - t.buf_hi) / t.buf_bytes);
  } else {
    t.t_off = 0;
    t.n_lo = (max_dyn - t.buf_lo) / t.buf_bytes;
    t.buf_hi = 0;
    total_bufs = t.n_lo;
  }
  t.nst = std::min(kMaxStages, total_bufs / WPH);
  if (t.nst < 2) return cudaErrorInvalidConfiguration;
  const int nbuf = t.nst * WPH;
  size_t smem = 0;
  if (Cfg::kTBytes > 0) {
    smem = (size_t)t.t_off + Cfg::kTBytes;
    if (nbuf > t.n_lo) smem = (size_t)t.buf_hi + (size_t)(nbuf - t.n_lo) * t.buf_bytes;
  } else {
    smem = (size_t)t.buf_lo + (size_t)nbuf * t.buf_bytes;
  }

  const int B = a.batch, Hq = a.num_q_heads;
  const int64_t slots = (int64_t)p.num_splits + B;
  t.part_acc = static_cast<float*>(a.workspace);
  t.part_ml = t.part_acc + slots * Hq * D;
  t.prefix = reinterpret_cast<int*>(t.part_ml + slots * Hq * 2);
  t.p_all = p_all;
  t.sketch = 1.2533141373155003f / (float)D;  // sqrt(pi / 2) / D
  auto kern = decode_tc_kernel<D, KB, VB, G, WPH, PROD>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if constexpr (PROD) {
    // a programmatic dependent of the projection p = S q~ (the previous launch on the
    // stream): the block-table scan and the first page copies overlap its tail; the
    // consumer warps wait for it before they read p
    cudaLaunchConfig_t kcfg{};
    kcfg.gridDim = dim3(p.num_splits);
    kcfg.blockDim = dim3(32 * (H + 1));
    kcfg.dynamicSmemBytes = smem;
    kcfg.stream = stream;
    cudaLaunchAttribute kattr[1];
    kattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    kattr[0].val.programmaticStreamSerializationAllowed = 1;
    kcfg.attrs = kattr;
    kcfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&kcfg, kern, t);
  } else {
    kern<<<p.num_splits, 32 * (H + 1), smem, stream>>>(t);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  count_launches(1);
  const int rows = B * Hq;
  // programmatic dependent launch: the combine's launch overlaps the split kernel's tail
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((rows + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, combine_tc_kernel<D / 32>, a, p.num_splits, (const float*)t.part_acc,
                           (const float*)t.part_ml, (const int*)t.prefix);
  if (err == cudaSuccess) count_launches(1);
  return err;
}


// One instantiation per translation unit line: the forms are split over several .cu files
// (tq_decode_tc*.cu) so that they compile in parallel.
#define TQ_TC_CASE(D, KB, VB, GG, WPH)                                                             \
  if (a.head_dim == D && a.k_bits == KB && a.v_bits == VB && a.num_q_heads / a.num_kv_heads == GG) \
    return launch_tc_typed<D, KB, VB, GG, WPH>(a, p, stream);
#define TQ_TC_VBITS(D, KB, WPH)                                                                      \
  TQ_TC_CASE(D, KB, 2, 4, WPH) TQ_TC_CASE(D, KB, 3, 4, WPH) TQ_TC_CASE(D, KB, 4, 4, WPH)            \
  TQ_TC_CASE(D, KB, 5, 4, WPH) TQ_TC_CASE(D, KB, 2, 8, WPH) TQ_TC_CASE(D, KB, 3, 8, WPH)            \
  TQ_TC_CASE(D, KB, 4, 8, WPH) TQ_TC_CASE(D, KB, 5, 8, WPH)
// product-quantised key rows at D = 128: MB-bit MSE indices (a.k_bits = MB + 1), every V width
#define TQ_TCP_CASE(MB, VB, GG)                                                                \
  if (a.k_bits == MB + 1 && a.v_bits == VB) return launch_tc_typed<128, MB, VB, GG, 2, true>(a, p, stream, p_all);
#define TQ_TCP_V(MB, GG) TQ_TCP_CASE(MB, 2, GG) TQ_TCP_CASE(MB, 3, GG) TQ_TCP_CASE(MB, 4, GG) TQ_TCP_CASE(MB, 5, GG)

}  // namespace
}  // namespace tq

namespace tq {
// Launchers of the instantiated forms, one per translation unit: each returns
// cudaErrorNotSupported for a shape it does not hold.  D 128 / 256 / 64 at K width 2 and 4
// (part a / c / e), 3 and 5 (part b / d / f), every V width, G 4 / 8.
cudaError_t launch_tc_part_a(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
cudaError_t launch_tc_part_b(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
cudaError_t launch_tc_part_c(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
cudaError_t launch_tc_part_d(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
cudaError_t launch_tc_part_e(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
cudaError_t launch_tc_part_f(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
// Product-quantised key rows, GQA group 8 (tq_decode_tc_q.cu).
cudaError_t launch_tc_prod_g8(const DecodeArgs& a, const DecodePlan& p, const float* p_all, cudaStream_t stream);
}  // namespace tq
