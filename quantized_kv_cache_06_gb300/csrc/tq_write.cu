// Packed-KV row writer: rotate, quantise, bit-pack and scatter rows into uint8 pages.
//
// TurboQuant docs: "vLLM Usage" (TQ Byte Layout, Slot Mapping, TQ Packed Page
// Contract: write_tq4_kv) and "Architecture" (PackedPageCache).
//
// One warp encodes one (token, kv head) row.  Lane l owns coordinates
// [l*E, l*E + E) of the D = 32*E row, so the sign flip, the norm, the
// Walsh-Hadamard butterflies and the quantisation all run in registers and
// shuffles.  The packed row is assembled in shared memory and written back as
// 32-bit words (rows are 4-byte aligned for D >= 32).
#include <algorithm>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_qjl.h"

namespace tq {
namespace {

constexpr int kWriteWarps = 8;

__global__ void validate_slots_kernel(const int64_t* __restrict__ slots, int64_t n, int64_t limit,
                                      int32_t* __restrict__ status) {
  // the tensor-core writer is a programmatic dependent of this kernel: it may be scheduled
  // now, does its set-up, and waits for this grid before it reads the status word
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    bad |= __ldg(slots + i) >= limit;
  if (__any_sync(kFullMask, bad) && (threadIdx.x & 31) == 0) atomicMax(status, (int32_t)kSlotOutOfRange);
}

template <typename T, int E>
__global__ void __launch_bounds__(kWriteWarps * 32)
write_rows_kernel(const T* __restrict__ raw, int64_t num_rows, int num_kv_heads, int bits,
                  const int64_t* __restrict__ slots, uint8_t* __restrict__ pages,
                  const float* __restrict__ signs, const float* __restrict__ centroids,
                  const int32_t* __restrict__ status) {
  constexpr int D = 32 * E;
  __shared__ float boundary[32];
  __shared__ uint32_t rowbuf[kWriteWarps][D * 5 / 32 + 1];

  const int nc = 1 << bits;
  // Decision points: correctly rounded midpoints of neighbouring fp32 centroids.
  if (threadIdx.x < nc - 1) boundary[threadIdx.x] = 0.5f * (centroids[threadIdx.x] + centroids[threadIdx.x + 1]);
  __syncthreads();
  if (*status != kOk) return;  // a slot failed validation: write nothing

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int index_words = D * bits / 32;
  const int row_words = index_words + 1;
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  float sg[E];
#pragma unroll
  for (int i = 0; i < E; ++i) sg[i] = __ldg(signs + lane * E + i);
  uint32_t* buf = rowbuf[warp];

  for (int64_t r = (int64_t)blockIdx.x * kWriteWarps + warp; r < num_rows; r += (int64_t)gridDim.x * kWriteWarps) {
    const int64_t t = r / num_kv_heads;
    const int h = (int)(r - t * num_kv_heads);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // "Slot Mapping": negative slots are ignored

    float v[E];
    load_chunk<T, E>(raw + r * D + lane * E, v);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(v[i], v[i], ss);
    ss = warp_sum(ss);
    // A row whose sum of squares leaves [2^-100, 2^100] is scaled by an exact power of two
    // 2^-ex from its largest |x| first (u is scale free; the norm is scaled back).
    int ex = 0;
    if (!(ss >= 0x1p-100f && ss <= 0x1p100f)) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) m = fmaxf(m, fabsf(v[i]));
      m = warp_max(m);
      if (m > 0.f && m <= 3.402823466e38f) {  // zero and non-finite rows keep their sums
        frexpf(m, &ex);
        ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          v[i] = scale_pow2(v[i], -ex);
          ss = fmaf(v[i], v[i], ss);
        }
        ss = warp_sum(ss);
      }
    }
    const float nu_s = sqrtf(ss);  // norm of the (scaled) row
    const float nu = scale_pow2(nu_s, ex);
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] *= sg[i];
    fwht_warp<E>(v);
    // y = H(s*x)/(sqrt(D) nu); a zero row and a row with a non-finite sum (NaN or infinite
    // input) get u = 0, the zero row's indices, the latter with its non-finite norm
    const bool bad = !(nu_s <= 3.402823466e38f);
    const float inv = (nu_s > 0.f && !bad) ? inv_sqrt_d / nu_s : 0.f;

    for (int w = lane; w < row_words; w += 32) buf[w] = 0u;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float u = bad ? 0.f : v[i] * inv;
      int idx = 0;  // #{k : boundary_k < u}, branch-free binary search
      for (int s = nc >> 1; s > 0; s >>= 1)
        if (u > boundary[idx + s - 1]) idx += s;
      const int bit = (lane * E + i) * bits;
      const int w = bit >> 5, o = bit & 31;
      atomicOr(&buf[w], (uint32_t)idx << o);
      if (o + bits > 32) atomicOr(&buf[w + 1], (uint32_t)idx >> (32 - o));
    }
    __syncwarp();
    if (lane == 0) buf[index_words] = __float_as_uint(nu);
    __syncwarp();
    uint32_t* dst = reinterpret_cast<uint32_t*>(pages + (slot * num_kv_heads + h) * (int64_t)(row_words * 4));
    for (int w = lane; w < row_words; w += 32) dst[w] = buf[w];
    __syncwarp();
  }
}

template <typename T>
cudaError_t launch_write_typed(const WriteArgs& a, cudaStream_t stream, int grid) {
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  const T* raw = static_cast<const T*>(a.raw);
#define TQ_WRITE_CASE(E)                                                                              \
  case 32 * E:                                                                                        \
    write_rows_kernel<T, E><<<grid, kWriteWarps * 32, 0, stream>>>(raw, rows, a.num_kv_heads, a.bits, \
                                                                   a.slots, a.pages, a.signs,         \
                                                                   a.centroids, a.status);            \
    break;
  switch (a.head_dim) {
    TQ_WRITE_CASE(1)
    TQ_WRITE_CASE(2)
    TQ_WRITE_CASE(4)
    TQ_WRITE_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef TQ_WRITE_CASE
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

}  // namespace

int device_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

cudaError_t launch_validate_slots(const WriteArgs& a, cudaStream_t stream, int num_sms) {
  const int vgrid = (int)std::min<int64_t>((a.num_tokens + 255) / 256, (int64_t)num_sms * 4);
  validate_slots_kernel<<<vgrid, 256, 0, stream>>>(a.slots, a.num_tokens, a.num_blocks * a.block_size, a.status);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) count_launches(1);
  return err;
}

// Status word of the writes called without a caller status word (tq_write_kv /
// tq_write_kv_prod with status_dev == NULL): one file-scope device int per device, its
// address looked up once per device with that device current.
namespace {
__device__ int32_t g_internal_write_status;
std::mutex g_internal_status_mutex;
int32_t* g_internal_status_ptr[128] = {};
}  // namespace

cudaError_t internal_write_status(int32_t** ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_internal_status_mutex);
  if (g_internal_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_internal_write_status);
    if (err != cudaSuccess) return err;
    g_internal_status_ptr[dev] = static_cast<int32_t*>(p);
  }
  *ptr = g_internal_status_ptr[dev];
  return cudaSuccess;
}

cudaError_t launch_write(const WriteArgs& a, cudaStream_t stream) {
  cudaError_t err = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  if (a.num_tokens == 0) return cudaSuccess;
  const int sms = device_sms();
  err = launch_validate_slots(a, stream, sms);
  if (err != cudaSuccess) return err;
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  if (a.head_dim == 16) return launch_write_d16(a, stream);
  if (write_tc_supported(a)) {
    // 16-row tiles, 8 warps per CTA, two CTAs per SM resident
    const int64_t tiles = (rows + 15) / 16;
    const int tgrid = (int)std::max<int64_t>(1, std::min<int64_t>((tiles + 7) / 8, (int64_t)sms * 2));
    return launch_write_tc(a, stream, tgrid);
  }
  const int grid = (int)std::min<int64_t>((rows + kWriteWarps - 1) / kWriteWarps, (int64_t)sms * 16);
  switch (a.dtype) {
    case kF32: return launch_write_typed<float>(a, stream, grid);
    case kF16: return launch_write_typed<__half>(a, stream, grid);
    case kBF16: return launch_write_typed<__nv_bfloat16>(a, stream, grid);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
