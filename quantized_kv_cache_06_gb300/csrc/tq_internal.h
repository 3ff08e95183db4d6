// Internal declarations shared by the host API (tq_api.cpp) and the kernels
// (tq_write.cu, tq_decode.cu).  Not part of the public C ABI (include/tq.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tq {

// Status codes written to the device status word; same values as tq_status.
enum : int32_t {
  kOk = 0,
  kInvalidArg = 1,
  kUnsupported = 2,
  kSlotOutOfRange = 3,
  kBlockOutOfRange = 4,
  kTimeout = 6,
};

// kI8: int8 query codes with one fp32 scale per (query row, q head) (the INT8-query
// prefill); queries only.
enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2, kI8 = 3 };

// Tries of one bounded mbarrier wait before it gives up and reports kTimeout (seconds at
// most with the hardware's own suspend time per try), and the number the next launches
// use: the default unless a failure-path test set another with tq_set_wait_limit.
constexpr uint32_t kDefaultWaitTries = 1u << 22;
uint32_t wait_tries();

// Process-wide count of kernel launches the library has enqueued (tq_launch_count): every
// launch site adds its launches once the launch call has returned without error.
void count_launches(int n);

struct WriteArgs {
  const void* raw;
  int dtype;
  int64_t num_tokens;
  int num_kv_heads;
  int head_dim;
  int bits;
  const int64_t* slots;
  uint8_t* pages;
  int64_t num_blocks;
  int block_size;
  const float* signs;
  const float* centroids;
  int32_t* status;
};

// Enqueues: status <- 0, slot validation, row write.  Returns the first launch error.
cudaError_t launch_write(const WriteArgs& a, cudaStream_t stream);

// Device address (current device) of the library's own status word, used by the writes
// called without one (tq_write.cu).
cudaError_t internal_write_status(int32_t** ptr);

// Tensor-core writer (tq_write_tc.cu): fp16 / bf16 rows, head_dim 64, 128 or 256, 2 to 5 bits.
bool write_tc_supported(const WriteArgs& a);
cudaError_t launch_write_tc(const WriteArgs& a, cudaStream_t stream, int grid);

// Multi-query attention (tq_prefill_mq.cu): windows of query rows against 32-token tiles
// dequantised once into shared memory, split-K over tokens.  Mixed prefill/decode takes
// windows of 64 / G rows; a plain decode of shapes without a tensor-core decode
// instantiation takes one row (sequence) per window.
struct MqPlan {
  int nsplit;           // token splits per sequence
  int split_len;        // tokens per split
  int windows;          // CTAs per (split, kv head)
  int rows_per_window;  // query rows per CTA
  size_t workspace_bytes;
};
struct DecodePlan {
  int kernel;            // which decode kernel runs (see tq_decode.cu)
  int num_splits;        // split-K factor per sequence
  int blocks_per_split;  // KV blocks per split
  size_t workspace_bytes;
  MqPlan mq;             // kernel 3: the multi-query kernel, one sequence per window
};

struct DecodeArgs {
  const void* q;
  int q_dtype;
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  const uint8_t* k_pages;
  int k_bits;
  const uint8_t* v_pages;
  int v_bits;
  int64_t num_blocks;
  int block_size;
  const int32_t* block_table;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  const float* signs;
  const float* k_centroids;
  const float* v_centroids;
  float scale;
  void* out;
  int out_dtype;
  void* workspace;
  int32_t* status;  // may be null
  float v_alpha;    // fp16 scale of the V centroids (tensor-core decode); 1 when unknown
  float k_alpha;    // fp16 scale of the K centroids (tensor-core decode); 1 when unknown
  // Mixed prefill/decode: row b of the batch reads block-table row bt_rows[b] (null: row b).
  // A row outside [0, bt_num_rows) reports kInvalidArg and reads nothing.
  const int32_t* bt_rows;
  int bt_num_rows;
  // q_dtype == kI8: scale of query (row, q head) r at q_scale[r] (null otherwise).
  const float* q_scale;
};

#ifdef __CUDACC__
// Block-table row of batch row b (-1 when the row map points outside the table).
__device__ __forceinline__ int block_table_row(const DecodeArgs& a, int b) {
  if (!a.bt_rows) return b;
  const int r = __ldg(a.bt_rows + b);
  return (r >= 0 && r < a.bt_num_rows) ? r : -1;
}
#endif

// head_dim 16 (tq_small.cu): rows of 8 to 14 bytes, taken byte by byte.  The writer runs
// after the slot validation; the decode handles row maps (prefill) and int8 queries.
struct DequantArgs;
cudaError_t launch_write_d16(const WriteArgs& a, cudaStream_t stream);
cudaError_t launch_decode_d16(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_dequant_d16(const DequantArgs& a, cudaStream_t stream);
cudaError_t launch_quantize_d16(const void* q, int q_dtype, int64_t rows, int8_t* codes, float* scales,
                                cudaStream_t stream);

// Int8 query codes -> codes and scales (tq_query.cu): one warp per (row, q head) of
// rows = num_q_rows * num_q_heads, D = head_dim.
cudaError_t launch_quantize_queries(const void* q, int q_dtype, int64_t rows, int head_dim, int8_t* codes,
                                    float* scales, cudaStream_t stream);

// Tensor-core decode (tq_decode_tc.cu): whether the shapes/bits in `a` have an
// instantiation, its warps per kv head, and its launch.
bool tc_decode_supported(const DecodeArgs& a);
int tc_partials_per_sequence_split();
cudaError_t launch_decode_tc(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);
// Its product-quantised key form (tq_decode_tc_p.cu): a.k_bits is the total key width,
// p_all the projection p = S q~ per (sequence, q head); p.num_splits CTAs.
bool tc_prod_decode_supported(const DecodeArgs& a);
cudaError_t launch_tc_prod(const DecodeArgs& a, const DecodePlan& p, const float* p_all, cudaStream_t stream);
// SM count of the current device (tq_write.cu).
int device_sms();

bool prefill_mq_supported(const DecodeArgs& a);
MqPlan plan_prefill_mq(const DecodeArgs& a, int num_sms, bool one_row_per_window);
// Enqueues status reset, the multi-query kernel and the split combine.
cudaError_t launch_prefill_mq(const DecodeArgs& a, const MqPlan& p, cudaStream_t stream);

// Split combine of the SIMT decode (tq_decode.cu): for each of `rows` rows merges
// `nsplit` partials acc [rows][nsplit][head_dim], ml [rows][nsplit][2] (running max in
// log2 units, sum), divides by the sum, applies R^T and writes out[rows][head_dim].
cudaError_t launch_combine_splits(const float* acc, const float* ml, int rows, int nsplit, int head_dim,
                                  const float* signs, void* out, int out_dtype, cudaStream_t stream);

// Split plan for the shapes in `a` on a device with `num_sms` SMs.
DecodePlan plan_decode(const DecodeArgs& a, int num_sms);

// Enqueues the decode for plan `p`.  Returns the first launch error.
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, cudaStream_t stream);

}  // namespace tq

namespace tq {

// Dense readback of packed rows (tq_dequant.cu).
struct DequantArgs {
  const uint8_t* pages;
  int bits;
  int64_t num_blocks;
  int block_size;
  int num_kv_heads;
  int head_dim;
  const int64_t* slots;
  int64_t num_tokens;
  const float* signs;
  const float* centroids;
  void* out;
  int out_dtype;
  int32_t* status;  // may be null
};

bool dequant_supported(const DequantArgs& a);
// Enqueues the readback (status must already be reset by the caller).
cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t stream, int num_sms);

// Fixed device scratch for tq_paged_decode_static: a file-scope __device__ array in
// tq_decode.cu.  Returns its device address on the current device (looked up once
// per device with cudaGetSymbolAddress) and its capacity in bytes.
cudaError_t static_decode_scratch(void** ptr, size_t* capacity);

}  // namespace tq
