// Host side of the C ABI declared in include/tq.h: argument checks, rotation signs,
// the Lloyd-Max codebook, and the kernel launches.
//
// The codebook is solved here independently of the test oracle: cell masses and
// first moments come from composite Gauss-Legendre quadrature of the coordinate
// density, and the initial centroids from bisection on the quadrature CDF.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "tq.h"
#include "tq_internal.h"
#include "tq_qjl.h"
#include "tq_recipe.h"

namespace {

thread_local std::string g_last_error;

tq_status fail(tq_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

tq_status ok() {
  g_last_error.clear();
  return TQ_OK;
}

bool pow2_dim_ok(int d) { return d >= 16 && d <= 256 && (d & (d - 1)) == 0; }
bool bits_ok(int b) { return b >= 2 && b <= 5; }
bool dtype_ok(int t) { return t == TQ_F32 || t == TQ_F16 || t == TQ_BF16; }
size_t dtype_size(int t) { return t == TQ_F32 ? 4 : 2; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

tq_status check_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(TQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- codebook

// Gauss-Legendre nodes and weights on [-1, 1] (Newton iteration on P_n).
void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
  x.assign(n, 0.0);
  w.assign(n, 0.0);
  for (int i = 0; i < (n + 1) / 2; ++i) {
    double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
    double pn = 0.0, dp = 1.0;
    for (int it = 0; it < 100; ++it) {
      double p_prev = 1.0, p = z;
      for (int k = 2; k <= n; ++k) {
        const double p_next = ((2.0 * k - 1.0) * z * p - (k - 1.0) * p_prev) / k;
        p_prev = p;
        p = p_next;
      }
      pn = p;
      dp = n * (z * p - p_prev) / (z * z - 1.0);
      const double dz = pn / dp;
      z -= dz;
      if (std::fabs(dz) < 1e-17) break;
    }
    x[i] = -z;
    x[n - 1 - i] = z;
    w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
  }
}

struct CoordDensity {
  double log_c, p;
  std::vector<double> gx, gw;
  explicit CoordDensity(int d) {
    log_c = std::lgamma(d / 2.0) - 0.5 * std::log(M_PI) - std::lgamma((d - 1) / 2.0);
    p = (d - 3) / 2.0;
    gauss_legendre(24, gx, gw);
  }
  double f(double x) const {
    const double t = 1.0 - x * x;
    return t <= 0.0 ? 0.0 : std::exp(log_c + p * std::log1p(-x * x));
  }
  // (integral of f, integral of x f) over [lo, hi], 8 panels of 24-point Gauss-Legendre.
  std::pair<double, double> moments(double lo, double hi) const {
    const int panels = 8;
    const double h = (hi - lo) / panels;
    double m0 = 0.0, m1 = 0.0;
    for (int k = 0; k < panels; ++k) {
      const double a = lo + k * h, mid = a + 0.5 * h;
      for (size_t i = 0; i < gx.size(); ++i) {
        const double x = mid + 0.5 * h * gx[i];
        const double fx = gw[i] * 0.5 * h * f(x);
        m0 += fx;
        m1 += x * fx;
      }
    }
    return {m0, m1};
  }
};

std::vector<double> solve_lloyd_max(int d, int bits) {
  const int n = 1 << bits;
  CoordDensity dens(d);
  // Initial centroids: (k + 1/2)/n quantiles by bisection on the quadrature CDF.
  std::vector<double> c(n);
  for (int k = 0; k < n; ++k) {
    const double target = (k + 0.5) / n;
    double lo = -1.0, hi = 1.0;
    for (int it = 0; it < 60; ++it) {
      const double mid = 0.5 * (lo + hi);
      const double cdf = 0.5 + (mid >= 0 ? dens.moments(0.0, mid).first : -dens.moments(mid, 0.0).first);
      (cdf < target ? lo : hi) = mid;
    }
    c[k] = 0.5 * (lo + hi);
  }
  std::vector<double> edges(n + 1), cn(n);
  for (int iter = 0; iter < 1000000; ++iter) {
    edges[0] = -1.0;
    edges[n] = 1.0;
    for (int k = 1; k < n; ++k) edges[k] = 0.5 * (c[k - 1] + c[k]);
    double moved = 0.0;
    for (int k = 0; k < n; ++k) {
      const auto mm = dens.moments(edges[k], edges[k + 1]);
      cn[k] = mm.second / mm.first;
      moved = std::fmax(moved, std::fabs(cn[k] - c[k]));
    }
    c.swap(cn);
    if (moved < 1e-14) break;
  }
  // The density is even: make the solution exactly odd-symmetric.
  std::vector<double> s(n);
  for (int k = 0; k < n; ++k) s[k] = 0.5 * (c[k] - c[n - 1 - k]);
  return s;
}

std::mutex g_cb_mutex;
std::map<std::pair<int, int>, std::vector<float>> g_cb_cache;

const std::vector<float>& codebook_f32(int d, int bits) {
  std::lock_guard<std::mutex> lock(g_cb_mutex);
  auto key = std::make_pair(d, bits);
  auto it = g_cb_cache.find(key);
  if (it != g_cb_cache.end()) return it->second;
  const std::vector<double> c = solve_lloyd_max(d, bits);
  std::vector<float> c32(c.size());
  for (size_t i = 0; i < c.size(); ++i) c32[i] = (float)c[i];
  return g_cb_cache.emplace(key, std::move(c32)).first->second;
}

// Nearest fp16 value of a positive double (ties to even), written out from the fp16
// format: 11 significant bits, exponent floor at 2^-14 (subnormal spacing 2^-24).
double round_to_fp16(double x) {
  int e = 0;
  std::frexp(x, &e);  // x = m 2^e, m in [0.5, 1)
  const int ee = e < -13 ? -13 : e;
  const double ulp = std::ldexp(1.0, ee - 11);
  return std::nearbyint(x / ulp) * ulp;
}

// Scale alpha in [1, 2) that brings every alpha * |c_k| closest to an fp16 grid point
// (the tensor-core decode stores V centroids as fp16(alpha * c) and divides by alpha
// afterwards); minimises the largest relative rounding error.  Cached per (D, b).
std::mutex g_alpha_mutex;
std::map<std::pair<int, int>, float> g_alpha_cache;

float fp16_scale_for(int d, int bits) {
  const std::vector<float>& c = codebook_f32(d, bits);
  std::lock_guard<std::mutex> lock(g_alpha_mutex);
  auto key = std::make_pair(d, bits);
  auto it = g_alpha_cache.find(key);
  if (it != g_alpha_cache.end()) return it->second;
  std::vector<double> mags;
  for (float v : c)
    if (v > 0.f) mags.push_back(v);
  float best = 1.0f;
  double best_err = 1e300;
  const int steps = 1 << 18;
  for (int i = 0; i < steps; ++i) {
    const float alpha = (float)(1.0 + (double)i / steps);
    double worst = 0.0;
    for (double m : mags) {
      const double exact = (double)alpha * m;
      const double stored = round_to_fp16((double)(alpha * (float)m));
      worst = std::fmax(worst, std::fabs(stored - exact) / exact);
      if (worst >= best_err) break;
    }
    if (worst < best_err) {
      best_err = worst;
      best = alpha;
    }
  }
  g_alpha_cache.emplace(key, best);
  return best;
}

int current_device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return sms > 0 ? sms : 1;
}

tq_status decode_shape_check(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                             int max_blocks_per_seq, int block_size) {
  if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 0 || block_size < 1)
    return fail(TQ_ERR_INVALID_ARG, "decode: invalid sizes (batch=%d, q_heads=%d, kv_heads=%d, max_blocks=%d, block_size=%d)",
                batch, num_q_heads, num_kv_heads, max_blocks_per_seq, block_size);
  if (num_q_heads % num_kv_heads != 0)
    return fail(TQ_ERR_INVALID_ARG, "decode: num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads, num_kv_heads);
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(TQ_ERR_UNSUPPORTED, "decode: GQA group %d not supported (1, 2, 4 or 8)", g);
  return ok();
}

// The decode kernel choice also depends on k_bits / v_bits, which the workspace queries do
// not take: the largest workspace over the SIMT, tensor-core and multi-query plans.
size_t decode_workspace_any_bits(tq::DecodeArgs a, int sms) {
  a.k_bits = a.v_bits = 0;
  size_t need = tq::plan_decode(a, sms).workspace_bytes;  // SIMT plan
  need = std::max(need, tq::plan_prefill_mq(a, sms, true).workspace_bytes);
  a.k_bits = a.v_bits = 4;  // the tensor-core plan where the shapes have one, else the multi-query plan
  need = std::max(need, tq::plan_decode(a, sms).workspace_bytes);
  return need;
}

tq::DecodeArgs make_decode_args(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                int max_blocks_per_seq, int block_size) {
  tq::DecodeArgs a{};
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.block_size = block_size;
  return a;
}

tq_status decode_impl(const char* name, const void* q, tq_dtype q_dtype, int batch, int num_q_heads,
                          int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                          const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, const float* signs, const float* k_centroids,
                          const float* v_centroids, float scale, void* out, tq_dtype out_dtype,
                          void* workspace, size_t workspace_bytes, int32_t* status_dev,
                          void* stream, const int32_t* bt_rows, int bt_num_rows, const float* q_scale = nullptr) {
  tq_status st = decode_shape_check(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  if (st != TQ_OK) return st;
  if (!bits_ok(k_bits) || !bits_ok(v_bits))
    return fail(TQ_ERR_UNSUPPORTED, "k_bits %d / v_bits %d: must be 2, 3, 4 or 5", k_bits, v_bits);
  // int8 query codes (q_dtype 3) only come with their scales, from tq_paged_prefill_int8q
  const bool int8q = q_scale != nullptr && (int)q_dtype == tq::kI8;
  if ((!dtype_ok(q_dtype) && !int8q) || !dtype_ok(out_dtype)) return fail(TQ_ERR_INVALID_ARG, "%s: unknown dtype", name);
  if (num_blocks < 0) return fail(TQ_ERR_INVALID_ARG, "%s: num_blocks < 0", name);
  if (batch > 0 && (!q || !k_pages || !v_pages || !seq_lens || !signs || !k_centroids || !v_centroids || !out ||
                    (max_blocks_per_seq > 0 && !block_table)))
    return fail(TQ_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (batch > 0 && int8q && !aligned(q_scale, 4)) return fail(TQ_ERR_INVALID_ARG, "%s: misaligned q_scales", name);
  if (batch > 0 && (!aligned(q, int8q ? 1 : dtype_size(q_dtype)) || !aligned(out, dtype_size(out_dtype)) ||
                    !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(block_table, 4) ||
                    !aligned(seq_lens, 4)))
    return fail(TQ_ERR_INVALID_ARG, "%s: misaligned pointer (pages need 16-byte alignment)", name);
  tq::DecodeArgs a = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  a.q = q;
  a.q_dtype = (int)q_dtype;
  a.k_pages = k_pages;
  a.k_bits = k_bits;
  a.v_pages = v_pages;
  a.v_bits = v_bits;
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.signs = signs;
  a.k_centroids = k_centroids;
  a.v_centroids = v_centroids;
  a.scale = scale;
  a.out = out;
  a.out_dtype = (int)out_dtype;
  a.workspace = workspace;
  a.status = status_dev;
  a.v_alpha = 1.0f;
  a.k_alpha = 1.0f;
  a.bt_rows = bt_rows;
  a.bt_num_rows = bt_num_rows;
  a.q_scale = int8q ? q_scale : nullptr;
  if (batch > 0 && (tq::tc_decode_supported(a) || tq::prefill_mq_supported(a))) {
    a.v_alpha = fp16_scale_for(head_dim, v_bits);
    a.k_alpha = fp16_scale_for(head_dim, k_bits);
  }
  if (bt_rows && tq::prefill_mq_supported(a)) {
    // mixed prefill/decode: query rows of one sequence share each dequantised key/value tile
    const tq::MqPlan plan = tq::plan_prefill_mq(a, current_device_sms(), false);
    if (batch > 0 && (workspace_bytes < plan.workspace_bytes || !workspace || !aligned(workspace, 16)))
      return fail(TQ_ERR_INVALID_ARG, "%s: workspace must be >= %zu bytes and 16-byte aligned (got %zu)", name,
                  plan.workspace_bytes, workspace_bytes);
    return check_cuda(tq::launch_prefill_mq(a, plan, static_cast<cudaStream_t>(stream)), name);
  }
  tq::DecodePlan plan = tq::plan_decode(a, current_device_sms());
  if (int8q && plan.kernel != 1) {
    // int8 query codes are read by the multi-query kernel (taken above for every shape it
    // covers) and the SIMT kernels; any other shape runs the SIMT plan
    tq::DecodeArgs s = a;
    s.k_bits = s.v_bits = 0;
    plan = tq::plan_decode(s, current_device_sms());
  }
  if (batch > 0 && (workspace_bytes < plan.workspace_bytes || !workspace || !aligned(workspace, 16)))
    return fail(TQ_ERR_INVALID_ARG, "%s: workspace must be >= %zu bytes and 16-byte aligned (got %zu)", name,
                plan.workspace_bytes, workspace_bytes);
  return check_cuda(tq::launch_decode(a, plan, static_cast<cudaStream_t>(stream)), name);
}


// Tries of a bounded device wait for the next launches; < 0 means the default.
std::atomic<int64_t> g_wait_limit{-1};

// A write called with status_dev == NULL: runs `launch` with the library's own status word
// (one per device, shared, so these calls are serialised), waits for the stream and
// returns the code the kernels left there.
std::mutex g_sync_write_mutex;

template <typename Launch>
tq_status write_with_own_status(const char* name, cudaStream_t stream, Launch launch) {
  std::lock_guard<std::mutex> lock(g_sync_write_mutex);
  int32_t* st = nullptr;
  tq_status r = check_cuda(tq::internal_write_status(&st), name);
  if (r != TQ_OK) return r;
  r = check_cuda(launch(st), name);
  if (r != TQ_OK) return r;
  int32_t code = 0;
  r = check_cuda(cudaMemcpyAsync(&code, st, sizeof(code), cudaMemcpyDeviceToHost, stream), name);
  if (r != TQ_OK) return r;
  r = check_cuda(cudaStreamSynchronize(stream), name);
  if (r != TQ_OK) return r;
  if (code == TQ_ERR_SLOT_OUT_OF_RANGE)
    return fail(TQ_ERR_SLOT_OUT_OF_RANGE, "%s: a slot is >= num_blocks * block_size; no row was written", name);
  if (code != TQ_OK) return fail((tq_status)code, "%s: device status %d", name, (int)code);
  return ok();
}

}  // namespace

namespace tq {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
uint32_t wait_tries() {
  const int64_t v = g_wait_limit.load(std::memory_order_relaxed);
  if (v < 0) return kDefaultWaitTries;
  return v > (int64_t)kDefaultWaitTries ? kDefaultWaitTries : (uint32_t)v;
}
}  // namespace tq

extern "C" {

const char* tq_last_error(void) { return g_last_error.c_str(); }

uint64_t tq_launch_count(void) { return tq::g_launches.load(std::memory_order_relaxed); }

int64_t tq_set_wait_limit(int64_t tries) {
  const int64_t prev = g_wait_limit.exchange(tries < 0 ? -1 : tries);
  return prev < 0 ? (int64_t)tq::kDefaultWaitTries : prev;
}

int64_t tq_row_bytes(int head_dim, int bits) {
  if (!pow2_dim_ok(head_dim) || !bits_ok(bits)) return -1;
  return ((int64_t)head_dim * bits + 7) / 8 + 4;
}

tq_status tq_build_rotation(int head_dim, uint64_t seed, float* signs_host) {
  if (!signs_host) return fail(TQ_ERR_INVALID_ARG, "tq_build_rotation: signs_host is NULL");
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  uint64_t state = seed;
  for (int i = 0; i < head_dim; ++i) {
    state += 0x9E3779B97F4A7C15ull;  // splitmix64 (Steele, Lea & Flood 2014)
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    signs_host[i] = (z >> 63) ? -1.0f : 1.0f;
  }
  return ok();
}

tq_status tq_codebook(int head_dim, int bits, float* centroids_host, float* boundaries_host) {
  if (!centroids_host) return fail(TQ_ERR_INVALID_ARG, "tq_codebook: centroids_host is NULL");
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  // 1 bit: the MSE part of the 2-bit groups of the recipe rows
  if (bits < 1 || bits > 5) return fail(TQ_ERR_UNSUPPORTED, "bits %d: must be 1 .. 5", bits);
  const std::vector<float>& c = codebook_f32(head_dim, bits);
  std::memcpy(centroids_host, c.data(), c.size() * sizeof(float));
  if (boundaries_host)
    for (size_t k = 0; k + 1 < c.size(); ++k)
      boundaries_host[k] = (float)(0.5 * ((double)c[k] + (double)c[k + 1]));
  return ok();
}

tq_status tq_write_kv(const void* raw, tq_dtype raw_dtype, int64_t num_tokens, int num_kv_heads,
                      int head_dim, int bits, const int64_t* slots, uint8_t* pages,
                      int64_t num_blocks, int block_size, const float* signs,
                      const float* centroids, int32_t* status_dev, void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 0 || block_size < 1)
    return fail(TQ_ERR_INVALID_ARG, "tq_write_kv: invalid sizes (tokens=%lld, kv_heads=%d, blocks=%lld, block_size=%d)",
                (long long)num_tokens, num_kv_heads, (long long)num_blocks, block_size);
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  if (!bits_ok(bits)) return fail(TQ_ERR_UNSUPPORTED, "bits %d: must be 2, 3, 4 or 5", bits);
  if (!dtype_ok(raw_dtype)) return fail(TQ_ERR_INVALID_ARG, "tq_write_kv: unknown raw dtype %d", (int)raw_dtype);
  if (num_tokens > 0 && (!raw || !slots || !pages || !signs || !centroids))
    return fail(TQ_ERR_INVALID_ARG, "tq_write_kv: null pointer argument");
  if (num_tokens > 0 && (!aligned(raw, 16) || !aligned(pages, 16) || !aligned(slots, 8) || !aligned(signs, 4) ||
                         !aligned(centroids, 4) || !aligned(status_dev, 4)))
    return fail(TQ_ERR_INVALID_ARG, "tq_write_kv: raw and pages must be 16-byte aligned, slots 8-byte aligned");
  tq::WriteArgs a{raw, (int)raw_dtype, num_tokens, num_kv_heads, head_dim, bits, slots, pages,
                  num_blocks, block_size, signs, centroids, status_dev};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!status_dev)
    return write_with_own_status("tq_write_kv", s, [&](int32_t* st) {
      a.status = st;
      return tq::launch_write(a, s);
    });
  return check_cuda(tq::launch_write(a, s), "tq_write_kv launch");
}

tq_status tq_dequant_rows(const uint8_t* pages, int bits, int64_t num_blocks, int block_size, int num_kv_heads,
                          int head_dim, const int64_t* slots, int64_t num_tokens, const float* signs,
                          const float* centroids, void* out, tq_dtype out_dtype, int32_t* status_dev,
                          void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 0 || block_size < 1)
    return fail(TQ_ERR_INVALID_ARG, "tq_dequant_rows: invalid sizes (tokens=%lld, kv_heads=%d, blocks=%lld, block_size=%d)",
                (long long)num_tokens, num_kv_heads, (long long)num_blocks, block_size);
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  if (!bits_ok(bits)) return fail(TQ_ERR_UNSUPPORTED, "bits %d: must be 2, 3, 4 or 5", bits);
  if (!dtype_ok(out_dtype)) return fail(TQ_ERR_INVALID_ARG, "tq_dequant_rows: unknown out dtype %d", (int)out_dtype);
  if (num_tokens > 0 && (!pages || !slots || !signs || !centroids || !out))
    return fail(TQ_ERR_INVALID_ARG, "tq_dequant_rows: null pointer argument");
  if (num_tokens > 0 && (!aligned(pages, 16) || !aligned(slots, 8) || !aligned(signs, 4) || !aligned(centroids, 4) ||
                         !aligned(out, 16) || !aligned(status_dev, 4)))
    return fail(TQ_ERR_INVALID_ARG, "tq_dequant_rows: pages and out must be 16-byte aligned, slots 8-byte aligned");
  tq::DequantArgs a{pages, bits, num_blocks, block_size, num_kv_heads, head_dim, slots, num_tokens,
                    signs, centroids, out, (int)out_dtype, status_dev};
  if (!tq::dequant_supported(a))
    return fail(TQ_ERR_UNSUPPORTED, "tq_dequant_rows: head_dim %d with %d bits has no kernel", head_dim, bits);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status_dev) {
    tq_status st = check_cuda(cudaMemsetAsync(status_dev, 0, sizeof(int32_t), s), "tq_dequant_rows status reset");
    if (st != TQ_OK) return st;
  }
  return check_cuda(tq::launch_dequant(a, s, current_device_sms()), "tq_dequant_rows launch");
}

size_t tq_paged_decode_workspace(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size) {
  if (decode_shape_check(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size) != TQ_OK)
    return 0;
  tq::DecodeArgs a = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  return decode_workspace_any_bits(a, current_device_sms());
}

tq_status tq_paged_decode(const void* q, tq_dtype q_dtype, int batch, int num_q_heads,
                          int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                          const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, const float* signs, const float* k_centroids,
                          const float* v_centroids, float scale, void* out, tq_dtype out_dtype,
                          void* workspace, size_t workspace_bytes, int32_t* status_dev,
                          void* stream) {
  return decode_impl("tq_paged_decode", q, q_dtype, batch, num_q_heads, num_kv_heads, head_dim, k_pages, k_bits,
                     v_pages, v_bits, num_blocks, block_size, block_table, max_blocks_per_seq, seq_lens, signs,
                     k_centroids, v_centroids, scale, out, out_dtype, workspace, workspace_bytes, status_dev, stream,
                     nullptr, 0);
}

size_t tq_paged_prefill_workspace(int num_q_rows, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int block_size) {
  // The larger of the row-mapped decode plan and the multi-query plan (which one runs
  // depends on k_bits / v_bits, which this query does not take).
  size_t need =
      tq_paged_decode_workspace(num_q_rows, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  if (need == 0) return 0;
  tq::DecodeArgs a =
      make_decode_args(num_q_rows, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  need = std::max(need, tq::plan_prefill_mq(a, current_device_sms(), false).workspace_bytes);
  return need;
}

tq_status tq_paged_prefill(const void* q, tq_dtype q_dtype, int num_q_rows, int num_q_heads, int num_kv_heads,
                           int head_dim, const uint8_t* k_pages, int k_bits, const uint8_t* v_pages, int v_bits,
                           int64_t num_blocks, int block_size, const int32_t* block_table, int num_seqs,
                           int max_blocks_per_seq, const int32_t* q_seq, const int32_t* q_len, const float* signs,
                           const float* k_centroids, const float* v_centroids, float scale, void* out,
                           tq_dtype out_dtype, void* workspace, size_t workspace_bytes, int32_t* status_dev,
                           void* stream) {
  if (num_seqs < 0) return fail(TQ_ERR_INVALID_ARG, "tq_paged_prefill: num_seqs < 0");
  if (num_q_rows > 0 && (!q_seq || !q_len || !aligned(q_seq, 4) || !aligned(q_len, 4)))
    return fail(TQ_ERR_INVALID_ARG, "tq_paged_prefill: q_seq and q_len must be non-null, 4-byte aligned");
  return decode_impl("tq_paged_prefill", q, q_dtype, num_q_rows, num_q_heads, num_kv_heads, head_dim, k_pages,
                     k_bits, v_pages, v_bits, num_blocks, block_size, block_table, max_blocks_per_seq, q_len, signs,
                     k_centroids, v_centroids, scale, out, out_dtype, workspace, workspace_bytes, status_dev, stream,
                     q_seq, num_seqs);
}

tq_status tq_quantize_queries_int8(const void* q, tq_dtype q_dtype, int64_t num_q_rows, int num_q_heads, int head_dim,
                                   int8_t* q_codes, float* q_scales, void* stream) {
  const char* name = "tq_quantize_queries_int8";
  if (num_q_rows < 0 || num_q_heads < 1) return fail(TQ_ERR_INVALID_ARG, "%s: invalid sizes", name);
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  if (!dtype_ok(q_dtype)) return fail(TQ_ERR_INVALID_ARG, "%s: unknown dtype %d", name, (int)q_dtype);
  if (num_q_rows > 0 && (!q || !q_codes || !q_scales)) return fail(TQ_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (num_q_rows > 0 && (!aligned(q, dtype_size(q_dtype)) || !aligned(q_scales, 4)))
    return fail(TQ_ERR_INVALID_ARG, "%s: misaligned pointer", name);
  return check_cuda(tq::launch_quantize_queries(q, (int)q_dtype, num_q_rows * num_q_heads, head_dim, q_codes, q_scales,
                                                static_cast<cudaStream_t>(stream)),
                    name);
}

tq_status tq_paged_prefill_int8q(const int8_t* q_codes, const float* q_scales, int num_q_rows, int num_q_heads,
                                 int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                                 const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                                 const int32_t* block_table, int num_seqs, int max_blocks_per_seq, const int32_t* q_seq,
                                 const int32_t* q_len, const float* signs, const float* k_centroids,
                                 const float* v_centroids, float scale, void* out, tq_dtype out_dtype, void* workspace,
                                 size_t workspace_bytes, int32_t* status_dev, void* stream) {
  const char* name = "tq_paged_prefill_int8q";
  if (num_seqs < 0) return fail(TQ_ERR_INVALID_ARG, "%s: num_seqs < 0", name);
  if (num_q_rows > 0 && (!q_seq || !q_len || !aligned(q_seq, 4) || !aligned(q_len, 4)))
    return fail(TQ_ERR_INVALID_ARG, "%s: q_seq and q_len must be non-null, 4-byte aligned", name);
  if (num_q_rows > 0 && !q_scales) return fail(TQ_ERR_INVALID_ARG, "%s: q_scales is NULL", name);
  // a non-null scale array marks the int8 codes (an empty batch needs none)
  static const float kNoRows = 0.f;
  return decode_impl(name, q_codes, (tq_dtype)tq::kI8, num_q_rows, num_q_heads, num_kv_heads, head_dim, k_pages,
                     k_bits, v_pages, v_bits, num_blocks, block_size, block_table, max_blocks_per_seq, q_len, signs,
                     k_centroids, v_centroids, scale, out, out_dtype, workspace, workspace_bytes, status_dev, stream,
                     q_seq, num_seqs, q_scales ? q_scales : &kNoRows);
}

tq_status tq_paged_decode_static(const void* q, tq_dtype q_dtype, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                                 const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                                 const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, const float* signs, const float* k_centroids,
                                 const float* v_centroids, float scale, void* out, tq_dtype out_dtype,
                                 int32_t* status_dev, void* stream) {
  // Same work as tq_paged_decode, with the split-K partials in the library's fixed
  // device array instead of a caller-provided workspace.  Nothing is allocated.
  void* scratch = nullptr;
  size_t capacity = 0;
  const cudaError_t err = tq::static_decode_scratch(&scratch, &capacity);
  if (err != cudaSuccess)
    return fail(TQ_ERR_CUDA, "tq_paged_decode_static: scratch address lookup failed: %s", cudaGetErrorString(err));
  tq_status st = decode_shape_check(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  if (st != TQ_OK) return st;
  tq::DecodeArgs shape = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  const size_t need = decode_workspace_any_bits(shape, current_device_sms());
  if (need > capacity)
    return fail(TQ_ERR_INVALID_ARG,
                "tq_paged_decode_static: these shapes need %zu bytes of scratch, more than the fixed %zu bytes; "
                "use tq_paged_decode with a caller workspace", need, capacity);
  return tq_paged_decode(q, q_dtype, batch, num_q_heads, num_kv_heads, head_dim, k_pages, k_bits, v_pages, v_bits,
                         num_blocks, block_size, block_table, max_blocks_per_seq, seq_lens, signs, k_centroids,
                         v_centroids, scale, out, out_dtype, scratch, capacity, status_dev, stream);
}

// ---------------------------------------------------------------- product-quantised keys

int64_t tq_prod_row_bytes(int head_dim, int bits) {
  if (!pow2_dim_ok(head_dim) || !bits_ok(bits)) return -1;
  return ((int64_t)head_dim * (bits - 1) + 7) / 8 + (head_dim + 7) / 8 + 8;
}

tq_status tq_build_qjl_matrix(int head_dim, uint64_t seed, float* s_host) {
  if (!s_host) return fail(TQ_ERR_INVALID_ARG, "tq_build_qjl_matrix: s_host is NULL");
  if (!pow2_dim_ok(head_dim)) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: must be a power of two in [16, 256]", head_dim);
  // splitmix64 (Steele, Lea & Flood 2014), outputs in pairs through Box-Muller (1958)
  uint64_t state = seed;
  auto next = [&state]() {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  };
  const int64_t n = (int64_t)head_dim * head_dim;  // even
  for (int64_t k = 0; k < n; k += 2) {
    const uint64_t z1 = next(), z2 = next();
    const double u1 = (double)((z1 >> 11) + 1) * 0x1p-53;  // (0, 1]
    const double u2 = (double)(z2 >> 11) * 0x1p-53;        // [0, 1)
    const double rad = std::sqrt(-2.0 * std::log(u1));
    s_host[k] = (float)(rad * std::cos(2.0 * M_PI * u2));
    s_host[k + 1] = (float)(rad * std::sin(2.0 * M_PI * u2));
  }
  return ok();
}

tq_status tq_write_kv_prod(const void* raw, tq_dtype raw_dtype, int64_t num_tokens, int num_kv_heads,
                           int head_dim, int bits, const int64_t* slots, uint8_t* pages, int64_t num_blocks,
                           int block_size, const float* signs, const float* mse_centroids,
                           const float* qjl_matrix, int32_t* status_dev, void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 0 || block_size < 1)
    return fail(TQ_ERR_INVALID_ARG, "tq_write_kv_prod: invalid sizes (tokens=%lld, kv_heads=%d, blocks=%lld, block_size=%d)",
                (long long)num_tokens, num_kv_heads, (long long)num_blocks, block_size);
  if (!tq::prod_supported(head_dim, bits))
    return fail(TQ_ERR_UNSUPPORTED, "tq_write_kv_prod: head_dim %d / bits %d: needs head_dim 64 or 128 and bits 3..5",
                head_dim, bits);
  if (!dtype_ok(raw_dtype)) return fail(TQ_ERR_INVALID_ARG, "tq_write_kv_prod: unknown raw dtype %d", (int)raw_dtype);
  if (num_tokens > 0 && (!raw || !slots || !pages || !signs || !mse_centroids || !qjl_matrix))
    return fail(TQ_ERR_INVALID_ARG, "tq_write_kv_prod: null pointer argument");
  if (num_tokens > 0 && (!aligned(raw, 16) || !aligned(pages, 16) || !aligned(slots, 8) || !aligned(signs, 4) ||
                         !aligned(mse_centroids, 4) || !aligned(qjl_matrix, 4) || !aligned(status_dev, 4)))
    return fail(TQ_ERR_INVALID_ARG, "tq_write_kv_prod: raw and pages must be 16-byte aligned, slots 8-byte aligned");
  tq::WriteArgs a{raw, (int)raw_dtype, num_tokens, num_kv_heads, head_dim, bits, slots, pages,
                  num_blocks, block_size, signs, mse_centroids, status_dev};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!status_dev)
    return write_with_own_status("tq_write_kv_prod", s, [&](int32_t* st) {
      a.status = st;
      return tq::launch_write_prod(a, qjl_matrix, s, current_device_sms());
    });
  return check_cuda(tq::launch_write_prod(a, qjl_matrix, s, current_device_sms()), "tq_write_kv_prod launch");
}

size_t tq_paged_decode_prod_workspace(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                      int max_blocks_per_seq, int block_size) {
  if (decode_shape_check(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size) != TQ_OK)
    return 0;
  tq::DecodeArgs a = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  a.k_bits = a.v_bits = 0;  // the SIMT split plan
  return tq::prod_decode_workspace(a, tq::plan_decode(a, current_device_sms()));
}

tq_status tq_paged_decode_prod(const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int num_kv_heads,
                               int head_dim, const uint8_t* k_pages, int k_bits, const uint8_t* v_pages,
                               int v_bits, int64_t num_blocks, int block_size, const int32_t* block_table,
                               int max_blocks_per_seq, const int32_t* seq_lens, const float* signs,
                               const float* k_mse_centroids, const float* v_centroids, const float* qjl_matrix,
                               float scale, void* out, tq_dtype out_dtype, void* workspace,
                               size_t workspace_bytes, int32_t* status_dev, void* stream) {
  const char* name = "tq_paged_decode_prod";
  tq_status st = decode_shape_check(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  if (st != TQ_OK) return st;
  if (!tq::prod_supported(head_dim, k_bits) || !bits_ok(v_bits))
    return fail(TQ_ERR_UNSUPPORTED, "%s: head_dim %d, k_bits %d, v_bits %d: needs head_dim 64 or 128, k_bits 3..5, "
                "v_bits 2..5", name, head_dim, k_bits, v_bits);
  if (!dtype_ok(q_dtype) || !dtype_ok(out_dtype)) return fail(TQ_ERR_INVALID_ARG, "%s: unknown dtype", name);
  if (num_blocks < 0) return fail(TQ_ERR_INVALID_ARG, "%s: num_blocks < 0", name);
  if (batch > 0 && (!q || !k_pages || !v_pages || !seq_lens || !signs || !k_mse_centroids || !v_centroids ||
                    !qjl_matrix || !out || (max_blocks_per_seq > 0 && !block_table)))
    return fail(TQ_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (batch > 0 && (!aligned(q, dtype_size(q_dtype)) || !aligned(out, dtype_size(out_dtype)) ||
                    !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(block_table, 4) ||
                    !aligned(seq_lens, 4) || !aligned(qjl_matrix, 4)))
    return fail(TQ_ERR_INVALID_ARG, "%s: misaligned pointer (pages need 16-byte alignment)", name);
  tq::DecodeArgs a = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  const tq::DecodePlan plan = tq::plan_decode(a, current_device_sms());  // SIMT split plan (k_bits 0)
  const size_t need = tq::prod_decode_workspace(a, plan);
  if (batch > 0 && (workspace_bytes < need || !workspace || !aligned(workspace, 16)))
    return fail(TQ_ERR_INVALID_ARG, "%s: workspace must be >= %zu bytes and 16-byte aligned (got %zu)", name, need,
                workspace_bytes);
  a.q = q;
  a.q_dtype = (int)q_dtype;
  a.k_pages = k_pages;
  a.k_bits = k_bits;
  a.v_pages = v_pages;
  a.v_bits = v_bits;
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.signs = signs;
  a.k_centroids = k_mse_centroids;
  a.v_centroids = v_centroids;
  a.scale = scale;
  a.out = out;
  a.out_dtype = (int)out_dtype;
  a.workspace = workspace;
  a.status = status_dev;
  // centroid scales of the tensor-core form's fp16 tables (the SIMT form reads fp32 centroids)
  a.k_alpha = fp16_scale_for(head_dim, k_bits - 1);
  a.v_alpha = fp16_scale_for(head_dim, v_bits);
  return check_cuda(tq::launch_decode_prod(a, qjl_matrix, plan, static_cast<cudaStream_t>(stream)), name);
}

}  // extern "C"

// ---------------------------------------------------------------- recipe modes

namespace {

// (high-group bits, low-group bits) of a recipe; false for an unknown one.
bool recipe_bits(int recipe, int* hi, int* lo) {
  if (recipe == TQ_RECIPE_TURBOQUANT25) {
    *hi = 3;
    *lo = 2;
    return true;
  }
  if (recipe == TQ_RECIPE_TURBOQUANT35) {
    *hi = 4;
    *lo = 3;
    return true;
  }
  return false;
}

tq_status recipe_codec_check(const char* name, int recipe, int head_dim, tq::RecipeArgs* rc) {
  int hi = 0, lo = 0;
  if (!recipe_bits(recipe, &hi, &lo)) return fail(TQ_ERR_INVALID_ARG, "%s: unknown recipe %d", name, recipe);
  if (!tq::recipe_supported(head_dim))
    return fail(TQ_ERR_UNSUPPORTED, "%s: head_dim %d: the recipe kernels take 64 or 128", name, head_dim);
  rc->bits_hi = hi;
  rc->bits_lo = lo;
  return ok();
}

}  // namespace

extern "C" {

int64_t tq_recipe_row_bytes(int recipe, int head_dim) {
  int hi = 0, lo = 0;
  if (!recipe_bits(recipe, &hi, &lo) || !tq::recipe_supported(head_dim)) return -1;
  return tq::recipe_row_bytes(head_dim, hi, lo);
}

tq_status tq_recipe_channel_order(int recipe, int head_dim, int num_kv_heads, const int32_t* high_host,
                                  int32_t* order_host) {
  int hi = 0, lo = 0;
  if (!recipe_bits(recipe, &hi, &lo)) return fail(TQ_ERR_INVALID_ARG, "tq_recipe_channel_order: unknown recipe %d", recipe);
  if (head_dim < 4 || head_dim % 2 || head_dim > 4096)
    return fail(TQ_ERR_INVALID_ARG, "tq_recipe_channel_order: head_dim %d cannot be split in two groups", head_dim);
  if (num_kv_heads < 1 || !high_host || !order_host)
    return fail(TQ_ERR_INVALID_ARG, "tq_recipe_channel_order: num_kv_heads < 1 or a NULL array");
  const int n = head_dim / 2;
  std::vector<char> used(head_dim);
  for (int h = 0; h < num_kv_heads; ++h) {
    const int32_t* row = high_host + (int64_t)h * n;
    std::fill(used.begin(), used.end(), 0);
    for (int k = 0; k < n; ++k) {
      if (row[k] < 0 || row[k] >= head_dim)
        return fail(TQ_ERR_INVALID_ARG, "tq_recipe_channel_order: kv head %d: high-group index %d outside [0, %d)", h,
                    (int)row[k], head_dim);
      if (k > 0 && row[k] <= row[k - 1])
        return fail(TQ_ERR_INVALID_ARG, "tq_recipe_channel_order: kv head %d: high-group indices must be sorted and unique",
                    h);
      used[row[k]] = 1;
    }
    int32_t* out = order_host + (int64_t)h * head_dim;
    std::copy(row, row + n, out);
    int w = n;
    for (int c = 0; c < head_dim; ++c)
      if (!used[c]) out[w++] = c;
  }
  return ok();
}

tq_status tq_recipe_calibrate(int recipe, int head_dim, int num_kv_heads, const float* samples_host,
                              int64_t num_samples, int32_t* high_host) {
  int hi = 0, lo = 0;
  if (!recipe_bits(recipe, &hi, &lo)) return fail(TQ_ERR_INVALID_ARG, "tq_recipe_calibrate: unknown recipe %d", recipe);
  if (head_dim < 4 || head_dim % 2 || head_dim > 4096 || num_kv_heads < 1 || num_samples < 0 || !high_host ||
      (num_samples > 0 && !samples_host))
    return fail(TQ_ERR_INVALID_ARG, "tq_recipe_calibrate: invalid sizes or a NULL array");
  const int n = head_dim / 2;
  std::vector<double> energy((size_t)num_kv_heads * head_dim, 0.0);
  for (int64_t t = 0; t < num_samples; ++t)
    for (int h = 0; h < num_kv_heads; ++h)
      for (int c = 0; c < head_dim; ++c) {
        const double x = samples_host[(t * num_kv_heads + h) * head_dim + c];
        energy[(size_t)h * head_dim + c] += x * x;
      }
  std::vector<int> chans(head_dim);
  for (int h = 0; h < num_kv_heads; ++h) {
    const double* e = energy.data() + (size_t)h * head_dim;
    for (int c = 0; c < head_dim; ++c) chans[c] = c;
    // largest energy first, ties to the lower channel
    std::stable_sort(chans.begin(), chans.end(), [e](int a, int b) { return e[a] > e[b]; });
    std::sort(chans.begin(), chans.begin() + n);
    std::copy(chans.begin(), chans.begin() + n, high_host + (int64_t)h * n);
  }
  return ok();
}

tq_status tq_write_kv_recipe(const void* raw, tq_dtype raw_dtype, int64_t num_tokens, int num_kv_heads, int head_dim,
                             int recipe, const int64_t* slots, uint8_t* pages, int64_t num_blocks, int block_size,
                             const int32_t* channel_order, const float* group_signs, const float* mse_high,
                             const float* mse_low, const float* qjl_matrix, int32_t* status_dev, void* stream) {
  const char* name = "tq_write_kv_recipe";
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 0 || block_size < 1)
    return fail(TQ_ERR_INVALID_ARG, "%s: invalid sizes (tokens=%lld, kv_heads=%d, blocks=%lld, block_size=%d)", name,
                (long long)num_tokens, num_kv_heads, (long long)num_blocks, block_size);
  tq::RecipeArgs rc{};
  tq_status st = recipe_codec_check(name, recipe, head_dim, &rc);
  if (st != TQ_OK) return st;
  if (!dtype_ok(raw_dtype)) return fail(TQ_ERR_INVALID_ARG, "%s: unknown raw dtype %d", name, (int)raw_dtype);
  if (num_tokens > 0 && (!raw || !slots || !pages || !channel_order || !group_signs || !mse_high || !mse_low ||
                         !qjl_matrix))
    return fail(TQ_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (num_tokens > 0 && (!aligned(raw, dtype_size(raw_dtype)) || !aligned(pages, 16) || !aligned(slots, 8) ||
                         !aligned(channel_order, 4) || !aligned(group_signs, 4) || !aligned(mse_high, 4) ||
                         !aligned(mse_low, 4) || !aligned(qjl_matrix, 4) || !aligned(status_dev, 4)))
    return fail(TQ_ERR_INVALID_ARG, "%s: misaligned pointer (pages need 16 bytes, slots 8)", name);
  rc.order = channel_order;
  rc.mse_hi = mse_high;
  rc.mse_lo = mse_low;
  rc.smat = qjl_matrix;
  tq::WriteArgs a{raw, (int)raw_dtype, num_tokens, num_kv_heads, head_dim, 0, slots, pages,
                  num_blocks, block_size, group_signs, nullptr, status_dev};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!status_dev)
    return write_with_own_status(name, s, [&](int32_t* w) {
      a.status = w;
      return tq::launch_write_recipe(a, rc, s, current_device_sms());
    });
  return check_cuda(tq::launch_write_recipe(a, rc, s, current_device_sms()), name);
}

size_t tq_paged_decode_recipe_workspace(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int block_size) {
  if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 0 || block_size < 1 ||
      num_q_heads % num_kv_heads || !tq::recipe_supported(head_dim))
    return 0;
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return 0;
  tq::DecodeArgs a = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  a.k_bits = a.v_bits = 0;  // the SIMT split plan
  return tq::recipe_decode_workspace(a, tq::plan_decode(a, current_device_sms()));
}

tq_status tq_paged_decode_recipe(const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, const uint8_t* k_pages, const uint8_t* v_pages, int recipe,
                                 int64_t num_blocks, int block_size, const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* channel_order, const float* group_signs,
                                 const float* mse_high, const float* mse_low, const float* qjl_matrix, float scale,
                                 void* out, tq_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, void* stream) {
  const char* name = "tq_paged_decode_recipe";
  tq::RecipeArgs rc{};
  tq_status st = recipe_codec_check(name, recipe, head_dim, &rc);
  if (st != TQ_OK) return st;
  st = decode_shape_check(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  if (st != TQ_OK) return st;
  if (!dtype_ok(q_dtype) || !dtype_ok(out_dtype)) return fail(TQ_ERR_INVALID_ARG, "%s: unknown dtype", name);
  if (num_blocks < 0) return fail(TQ_ERR_INVALID_ARG, "%s: num_blocks < 0", name);
  if (batch > 0 && (!q || !k_pages || !v_pages || !seq_lens || !channel_order || !group_signs || !mse_high ||
                    !mse_low || !qjl_matrix || !out || (max_blocks_per_seq > 0 && !block_table)))
    return fail(TQ_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (batch > 0 && (!aligned(q, dtype_size(q_dtype)) || !aligned(out, dtype_size(out_dtype)) ||
                    !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(block_table, 4) ||
                    !aligned(seq_lens, 4) || !aligned(channel_order, 4) || !aligned(qjl_matrix, 4)))
    return fail(TQ_ERR_INVALID_ARG, "%s: misaligned pointer (pages need 16-byte alignment)", name);
  tq::DecodeArgs a = make_decode_args(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size);
  const tq::DecodePlan plan = tq::plan_decode(a, current_device_sms());  // SIMT split plan (k_bits 0)
  const size_t need = tq::recipe_decode_workspace(a, plan);
  if (batch > 0 && (workspace_bytes < need || !workspace || !aligned(workspace, 16)))
    return fail(TQ_ERR_INVALID_ARG, "%s: workspace must be >= %zu bytes and 16-byte aligned (got %zu)", name, need,
                workspace_bytes);
  rc.order = channel_order;
  rc.mse_hi = mse_high;
  rc.mse_lo = mse_low;
  rc.smat = qjl_matrix;
  a.q = q;
  a.q_dtype = (int)q_dtype;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.k_bits = a.v_bits = 0;
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.signs = group_signs;
  a.scale = scale;
  a.out = out;
  a.out_dtype = (int)out_dtype;
  a.workspace = workspace;
  a.status = status_dev;
  a.v_alpha = a.k_alpha = 1.0f;
  return check_cuda(tq::launch_decode_recipe(a, rc, plan, static_cast<cudaStream_t>(stream)), name);
}

}  // extern "C"
