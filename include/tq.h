/*
 * tq.h -- C ABI of the GB300 TurboQuant packed-KV library (libtq_gb300.so).
 *
 * The library implements the two data-parallel steps of TurboQuant's packed KV
 * cache as hand-written CUDA kernels for sm_103a:
 *
 *   tq_write_kv      rotate, quantise, bit-pack and scatter K or V rows into uint8
 *                    pages ("vLLM Usage": TQ Byte Layout, Slot Mapping, TQ Packed
 *                    Page Contract; "Architecture": PackedPageCache).
 *   tq_paged_decode  single-query attention that reads those pages through a block
 *                    table without materialising dense K/V ("Architecture":
 *                    Diagnostic vs Serving Paths, direct-QK and packed-V).
 *
 * plus the host-side set-up the contract call needs (rotation signs, Lloyd-Max
 * codebook, row size), and the calls that widen the path over the same pages:
 *
 *   tq_paged_decode_static  the decode without a caller workspace (fixed scratch).
 *   tq_paged_prefill        mixed prefill/decode: query rows of one sequence share each
 *                           dequantised key/value tile ("vLLM Usage", Runtime Dispatch);
 *                           tq_paged_prefill_int8q takes int8 query codes and scales
 *                           (tq_quantize_queries_int8 makes them).
 *   tq_dequant_rows         dense readback of packed rows ("vLLM Reference Audit",
 *                           tq4_decompress).
 *   tq_write_kv_prod,       product-quantised ("QJL residual") key rows and the decode
 *   tq_paged_decode_prod    over them ("vLLM Reference Audit", MSE and QJL codecs).
 *   tq_write_kv_recipe,     the recipe cache modes turboquant25 / turboquant35: grouped
 *   tq_paged_decode_recipe  product-quantised K and V rows ("vLLM Usage", Cache Dtypes;
 *                           "Architecture", vLLM Runtime Mapping), with the metadata
 *                           helpers tq_recipe_channel_order and tq_recipe_calibrate.
 *
 * Conventions shared by every entry point:
 *   - Every buffer is owned by the caller.  "device" pointers must point to memory of
 *     the current CUDA device; "host" pointers to ordinary host memory.  The library
 *     never allocates or frees device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Device work is enqueued on it and the call returns without synchronising.
 *   - Every call returns a tq_status.  On a non-OK return, tq_last_error() gives a
 *     message for the calling thread.  Argument errors are detected on the host
 *     before anything is enqueued.  Errors that depend on device data (slots, block
 *     ids, sequence lengths) are reported through `status_dev`, a device int32 the
 *     caller reads after the stream reaches it: 0 = OK, otherwise a tq_status code
 *     (the largest one when several kinds occur).  No kernel traps or asserts.
 *   - Geometry: head_dim D is a power of two in [16, 256]; bits b in {2, 3, 4, 5};
 *     row_bytes RB(D, b) = ceil(D*b/8) + 4.  A page tensor is
 *     uint8[num_blocks][block_size][num_kv_heads][RB], contiguous, no padding, one
 *     tensor per component (K and V are independent and may use different bits).
 *   - Row layout (reading of "TQ Byte Layout"): index j of a row occupies bits
 *     [j*b, (j+1)*b) of the index bytes, LSB first (stream bit k = bit k%8 of byte
 *     k/8); bytes [RB-4, RB) hold the row's L2 norm as a little-endian fp32.
 *   - Rotation: R = H_D diag(s) / sqrt(D) with H_D the Sylvester Hadamard matrix
 *     (sign flip, then normalised Walsh-Hadamard transform; RHT in "TQ Packed Page
 *     Contract").
 */
#ifndef TQ_GB300_H
#define TQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tq_status {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,        /* null pointer, negative size, inconsistent shapes */
  TQ_ERR_UNSUPPORTED = 2,        /* valid but outside what the kernels handle (D, bits, GQA group) */
  TQ_ERR_SLOT_OUT_OF_RANGE = 3,  /* a write slot >= num_blocks * block_size */
  TQ_ERR_BLOCK_OUT_OF_RANGE = 4, /* a block-table entry read by decode lies outside [0, num_blocks) */
  TQ_ERR_CUDA = 5,               /* a CUDA runtime call failed (message in tq_last_error) */
  TQ_ERR_TIMEOUT = 6             /* a device-side wait gave up after its iteration limit; the
                                    output of that call is incomplete (an internal error: no
                                    valid input produces it) */
} tq_status;

typedef enum tq_dtype { TQ_F32 = 0, TQ_F16 = 1, TQ_BF16 = 2 } tq_dtype;

/* Message for the last non-OK status returned on the calling thread ("" if none).
 * The pointer stays valid until the next library call on that thread. */
const char* tq_last_error(void);

/* Failure-path testing hook (the pages have no counterpart).  Every device-side wait of
 * the tensor-core decode is bounded: after a number of tries it gives up, the kernel
 * records TQ_ERR_TIMEOUT in status_dev and returns (its copies in flight drained first),
 * so a wait that cannot end never hangs the GPU.  This sets the number of tries of the
 * pipeline waits of launches made after the call: `tries` >= 0 sets it (0: every such
 * wait gives up at once, so a decode with at least one block reports TQ_ERR_TIMEOUT and
 * leaves its output incomplete), `tries` < 0 restores the default.  Returns the previous
 * value.  Process-wide; meant for tests that check the timeout is reported and that the
 * next call with the default is correct, not for production use. */
int64_t tq_set_wait_limit(int64_t tries);

/* Number of kernel launches the library has enqueued in this process, all devices and
 * streams together (each launch counted once its launch call returned without error).
 * For measurement: the difference over a timed region is the number of the library's own
 * kernels that region ran. */
uint64_t tq_launch_count(void);

/* Row size in bytes for one component, one token and one KV head: ceil(D*b/8) + 4
 * ("vLLM Usage", TQ Byte Layout).  Returns -1 when head_dim or bits is unsupported. */
int64_t tq_row_bytes(int head_dim, int bits);

/* Lloyd-Max codebooks exist for bits 1..5 (tq_codebook); rows and kernels take 2..5, the
 * 1-bit codebook serves the MSE part of 2-bit recipe groups. */

/* RHT signs for build_rotation(dim, RHT, seed) ("vLLM Usage", TQ Packed Page Contract).
 * Writes head_dim values in {-1.0f, +1.0f} to signs_host[0..D): sign i is -1 when the
 * top bit of the i-th output of splitmix64 seeded with `seed` is set (a reading: the
 * pages fix only the mode and the seed).  Host only; errors: TQ_ERR_INVALID_ARG
 * (null), TQ_ERR_UNSUPPORTED (head_dim). */
tq_status tq_build_rotation(int head_dim, uint64_t seed, float* signs_host);

/* Lloyd-Max codebook for one coordinate of a uniformly random unit vector in R^D
 * (get_codebook_tensors(dim, bits) in "TQ Packed Page Contract"; Lloyd-Max / Beta in
 * "vLLM Reference Audit", Feature Checklist).  Density on [-1, 1]:
 * f_D(x) = Gamma(D/2) / (sqrt(pi) Gamma((D-1)/2)) (1 - x^2)^((D-3)/2).
 * centroids_host[0 .. 2^b) receives the ascending fp32 centroids (fp64 fixed point,
 * rounded once); boundaries_host[0 .. 2^b - 1), if not NULL, receives the decision
 * points the writer uses: the midpoint of neighbouring fp32 centroids, rounded to
 * fp32.  Host only; results are cached per (D, b).  Errors: TQ_ERR_INVALID_ARG,
 * TQ_ERR_UNSUPPORTED. */
tq_status tq_codebook(int head_dim, int bits, float* centroids_host, float* boundaries_host);

/* Packed-KV row writer (write_tq4_kv in "TQ Packed Page Contract").
 *
 *   raw        device, raw_dtype[num_tokens][num_kv_heads][head_dim], contiguous.
 *   slots      device, int64[num_tokens], flat slots: row (t, h) goes to
 *              pages[slots[t] / block_size][slots[t] % block_size][h][:].
 *              Negative slots are skipped ("Slot Mapping").
 *   pages      device, uint8[num_blocks][block_size][num_kv_heads][RB(D, bits)].
 *   signs      device, float[head_dim] from tq_build_rotation.
 *   centroids  device, float[2^bits] ascending, from tq_codebook.
 *   status_dev device int32 or NULL.  If not NULL: set to 0 at the start of the call,
 *              then to TQ_ERR_SLOT_OUT_OF_RANGE if any slot >= num_blocks * block_size
 *              -- in that case NO row is written (validation runs before the write) --
 *              and the call stays asynchronous (it can be captured in a CUDA graph; the
 *              caller reads the word later).  If NULL ("Slot Mapping": a slot outside
 *              the allocated pages raises): the call uses a status word of the library
 *              (one per device, shared by such calls, which the library serialises),
 *              synchronises `stream` and returns TQ_ERR_SLOT_OUT_OF_RANGE itself when a
 *              slot was out of range (nothing written) or TQ_OK.  That form cannot be
 *              captured in a CUDA graph (its synchronisation fails with TQ_ERR_CUDA).
 *
 * Each row x is encoded as: nu = ||x||_2 (fp32), u = x / nu (0 if nu == 0),
 * y = R u (fp32, in-register FWHT), index_j = #{k : boundary_k < y_j} (the nearest
 * centroid, ties to the lower index), packed LSB-first, norm appended.  Rows of any
 * finite scale are encoded the same way (a row whose fp32 sum of squares would leave
 * [2^-100, 2^100] is first scaled by an exact power of two).  A row with a NaN or an
 * infinite coordinate is stored as a zero row's indices with a non-finite norm.  Rows
 * of skipped tokens keep their previous bytes.  Duplicate non-negative slots: which
 * token's row survives is unspecified.  Asynchronous unless status_dev is NULL; errors
 * detected on the host: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA. */
tq_status tq_write_kv(const void* raw, tq_dtype raw_dtype, int64_t num_tokens, int num_kv_heads,
                      int head_dim, int bits, const int64_t* slots, uint8_t* pages,
                      int64_t num_blocks, int block_size, const float* signs,
                      const float* centroids, int32_t* status_dev, void* stream);

/* Bytes of device workspace tq_paged_decode needs for these shapes on the current
 * device (split-K partials).  0 when the arguments are invalid. */
size_t tq_paged_decode_workspace(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size);

/* Paged decode attention over packed pages (decode_tq4_paged in "TQ Packed Page
 * Contract"; "Architecture", Diagnostic vs Serving Paths).
 *
 *   q            device, q_dtype[batch][num_q_heads][head_dim].
 *   k_pages      device, uint8[num_blocks][block_size][num_kv_heads][RB(D, k_bits)].
 *   v_pages      device, uint8[num_blocks][block_size][num_kv_heads][RB(D, v_bits)].
 *   block_table  device, int32[batch][max_blocks_per_seq]: token t of sequence b is
 *                row (t % block_size) of block block_table[b][t / block_size].
 *   seq_lens     device, int32[batch]; 0 gives a zero output row.
 *   signs        device, float[head_dim]; k_centroids / v_centroids device,
 *                float[2^k_bits] / float[2^v_bits].
 *   scale        softmax scale; <= 0 selects 1/sqrt(head_dim).
 *   out          device, out_dtype[batch][num_q_heads][head_dim].
 *   workspace    device, >= tq_paged_decode_workspace(...) bytes, 16-byte aligned.
 *   status_dev   device int32 or NULL.  If not NULL it is set to 0 at the start of
 *                the call, then to TQ_ERR_BLOCK_OUT_OF_RANGE if a block id read lies
 *                outside [0, num_blocks) (its tokens are left out of the softmax),
 *                or TQ_ERR_INVALID_ARG if a seq_len is negative or exceeds
 *                max_blocks_per_seq * block_size (it is clamped).
 *
 * q head h attends with kv head h / (num_q_heads / num_kv_heads).  Scores are
 * scale * nu_k * <R q, c_k[idx]> computed from the packed indices; values are
 * accumulated in rotated space, sum p nu_v c_v[idx_v], with an online softmax, and
 * one inverse rotation R^T is applied per output row.  Asynchronous; host-detected
 * errors: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA. */
tq_status tq_paged_decode(const void* q, tq_dtype q_dtype, int batch, int num_q_heads,
                          int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                          const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, const float* signs, const float* k_centroids,
                          const float* v_centroids, float scale, void* out, tq_dtype out_dtype,
                          void* workspace, size_t workspace_bytes, int32_t* status_dev,
                          void* stream);

/* Mixed prefill/decode attention over the packed cache ("vLLM Usage", Runtime Dispatch:
 * "cache plus mixed prefill/decode" reads the packed cache).
 *
 * Query row i (0 <= i < num_q_rows) is one token of sequence q_seq[i] that sees the first
 * q_len[i] tokens of that sequence (causal: its position + 1; the cache already holds the
 * new tokens, written by tq_write_kv).  Row i is computed exactly as tq_paged_decode would
 * compute a one-query sequence with block-table row block_table[q_seq[i]] and length
 * q_len[i]; a decode batch is the case of one row per sequence at its full length.
 *
 *   q            device, q_dtype [num_q_rows][num_q_heads][head_dim]
 *   block_table  device int32 [num_seqs][max_blocks_per_seq]
 *   q_seq, q_len device int32 [num_q_rows]
 *   out          device, out_dtype [num_q_rows][num_q_heads][head_dim]
 *   workspace    device, >= tq_paged_prefill_workspace(num_q_rows, ...) bytes, 16-byte aligned
 * Other arguments, the status word and the errors are those of tq_paged_decode; a q_seq
 * entry outside [0, num_seqs) gives a zero row and TQ_ERR_INVALID_ARG in status_dev.
 * For head_dim 64, 128 or 256 with 2/4-bit (or equal 3/5-bit) K and V, up to 64 / G
 * consecutive rows of one sequence share every dequantised 32-token key/value tile, so a
 * prefill chunk reads the cache once: keep the rows of a chunk next to each other in
 * q_seq (rows of several sequences in one window are taken one sequence after the other).
 * Other shapes run the decode kernels row by row. */
size_t tq_paged_prefill_workspace(int num_q_rows, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int block_size);
tq_status tq_paged_prefill(const void* q, tq_dtype q_dtype, int num_q_rows, int num_q_heads, int num_kv_heads,
                           int head_dim, const uint8_t* k_pages, int k_bits, const uint8_t* v_pages, int v_bits,
                           int64_t num_blocks, int block_size, const int32_t* block_table, int num_seqs,
                           int max_blocks_per_seq, const int32_t* q_seq, const int32_t* q_len, const float* signs,
                           const float* k_centroids, const float* v_centroids, float scale, void* out,
                           tq_dtype out_dtype, void* workspace, size_t workspace_bytes, int32_t* status_dev,
                           void* stream);

/* INT8-query prefill ("vLLM Usage", Runtime Dispatch: cache plus the INT8 prefill gate
 * takes the int8 query path; "vLLM Reference Audit", File Map: INT8-Q prefill, int8 query
 * scale over packed pages).  The pages give no quantiser; the reading: one symmetric scale
 * per (query row, q head), s = amax / 127, code = round-half-even(q / s) in [-127, 127],
 * both divisions correctly rounded fp32; a zero row has s = 0 and codes 0.
 *
 * tq_quantize_queries_int8: q device q_dtype [num_q_rows][num_q_heads][head_dim] ->
 *   q_codes device int8 [num_q_rows][num_q_heads][head_dim] and q_scales device float
 *   [num_q_rows][num_q_heads].  Asynchronous; errors TQ_ERR_INVALID_ARG / UNSUPPORTED.
 * tq_paged_prefill_int8q: tq_paged_prefill with int8 query codes and their scales in place
 *   of q / q_dtype: row i attends with the query q_scales[i][h] * q_codes[i][h][:] (the
 *   kernels take the codes and scales as they are; out_dtype gives the output type).  The
 *   workspace is tq_paged_prefill_workspace's. */
tq_status tq_quantize_queries_int8(const void* q, tq_dtype q_dtype, int64_t num_q_rows, int num_q_heads, int head_dim,
                                   int8_t* q_codes, float* q_scales, void* stream);
tq_status tq_paged_prefill_int8q(const int8_t* q_codes, const float* q_scales, int num_q_rows, int num_q_heads,
                                 int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                                 const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                                 const int32_t* block_table, int num_seqs, int max_blocks_per_seq, const int32_t* q_seq,
                                 const int32_t* q_len, const float* signs, const float* k_centroids,
                                 const float* v_centroids, float scale, void* out, tq_dtype out_dtype, void* workspace,
                                 size_t workspace_bytes, int32_t* status_dev, void* stream);

/* Dense readback of packed rows: the inverse addressing of tq_write_kv ("vLLM Reference
 * Audit", file map: tq4_decompress, the TQ4 unpack kernel for diagnostic readback of
 * packed index bytes and norms; "Architecture", Diagnostic vs Serving Paths: dense
 * reconstruction for layout and distortion checks).
 *
 * For token t (0 <= t < num_tokens) and kv head h, with s = slots[t]:
 *   s >= 0:  out[t][h][:] = nu * R^T c[idx], the row pages[s / block_size][s % block_size][h]
 *            unpacked (LSB-first b-bit indices idx, fp32 norm nu in its last 4 bytes), with
 *            R^T = diag(signs) H_D / sqrt(D) and c = `centroids`;
 *   s < 0:   out[t][h][:] = 0;
 *   s >= num_blocks * block_size: out[t][h][:] = 0 and TQ_ERR_SLOT_OUT_OF_RANGE in status_dev.
 * A sequence's rows are read back by passing its slots (token i of the sequence sits at
 * block_table[i / block_size] * block_size + i % block_size, "vLLM Usage", Slot Mapping).
 *
 *   pages      device, uint8 [num_blocks][block_size][num_kv_heads][RB(head_dim, bits)],
 *              16-byte aligned
 *   slots      device, int64 [num_tokens], 8-byte aligned
 *   signs      device, fp32 [head_dim] (tq_build_rotation); centroids device, fp32 [2^bits]
 *              (tq_codebook) -- the ones the rows were written with
 *   out        device, out_dtype [num_tokens][num_kv_heads][head_dim], 16-byte aligned;
 *              computed in fp32, rounded once to out_dtype
 *   status_dev device int32 or NULL; reset to 0 by the call, then set as above
 *
 * head_dim must be 32, 64, 128 or 256 and bits 2..5 (TQ_ERR_UNSUPPORTED otherwise).
 * Reads RB bytes and writes head_dim values per row; no workspace, graph-capturable. */
tq_status tq_dequant_rows(const uint8_t* pages, int bits, int64_t num_blocks, int block_size, int num_kv_heads,
                          int head_dim, const int64_t* slots, int64_t num_tokens, const float* signs,
                          const float* centroids, void* out, tq_dtype out_dtype, int32_t* status_dev,
                          void* stream);

/* Allocation-free variant of tq_paged_decode.  The TurboQuant pages have no
 * counterpart: it exists for callers that cannot call cudaMalloc -- a plugin whose
 * host framework owns all device memory, a deployment held to a fixed memory
 * budget, or a latency-critical loop that must not hit cudaMalloc/cudaFree (which
 * can synchronise the device).
 *
 * Arguments, semantics and errors are those of tq_paged_decode, without `workspace`
 * and `workspace_bytes`: the split-K partials live in a fixed 16 MiB device array
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  The caller still passes every input and output.  Shapes whose
 * partials exceed 16 MiB (tq_paged_decode_workspace(...) > 16 MiB) are rejected
 * with TQ_ERR_INVALID_ARG and a message naming the size.
 *
 * The first call on each device looks the array's device address up (with that
 * device current); make that first call before any stream capture.  All calls share
 * the one array and it keeps the last call's contents (the decode overwrites every
 * partial it reads, so nothing needs clearing); calls whose work overlaps on the
 * GPU -- on different streams, or from different host threads -- race on it, so
 * serialise them.  Calls no cudaMalloc, cudaFree or allocating routine. */
tq_status tq_paged_decode_static(const void* q, tq_dtype q_dtype, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, const uint8_t* k_pages, int k_bits,
                                 const uint8_t* v_pages, int v_bits, int64_t num_blocks, int block_size,
                                 const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, const float* signs, const float* k_centroids,
                                 const float* v_centroids, float scale, void* out, tq_dtype out_dtype,
                                 int32_t* status_dev, void* stream);

/* ---------------------------------------------------------------------------------
 * Product-quantised ("QJL residual") key rows ("vLLM Reference Audit": File Map, the
 * quantizer's "MSE and QJL codecs" with indices, norms and signs, TurboQuantMSE /
 * TurboQuantProd; Feature Checklist, "QJL residual").  The pages name the codec but not
 * its arithmetic or layout; the readings below follow the product quantiser that
 * TurboQuantProd names: a (b-1)-bit MSE row plus a one-bit Johnson-Lindenstrauss sketch
 * of its residual, which makes the score an unbiased estimate of <q, k>.
 *
 * Key row at b bits (b in {2..5} for the layout): the (b-1)-bit MSE indices of y = R x/nu
 * (LSB-first, as in the MSE rows), then D sign bits z_i = [(S r)_i >= 0] with r = y -
 * c[idx] the rotated residual (bit i = bit i%8 of byte i/8), then nu = ||x|| and gamma =
 * ||r|| as little-endian fp32: RBP(D, b) = D (b-1)/8 + D/8 + 8.  S is a D x D matrix of
 * N(0, 1) numbers (tq_build_qjl_matrix).  Values keep the MSE rows of tq_write_kv.
 * --------------------------------------------------------------------------------- */

/* RBP(head_dim, bits); -1 when head_dim is not a power of two in [16, 256] or bits is
 * outside 2..5. */
int64_t tq_prod_row_bytes(int head_dim, int bits);

/* The sketch matrix S, row-major fp32 [head_dim][head_dim], written to s_host: entry
 * (i, j) is normal number i*D + j of the stream seeded with `seed` -- splitmix64 outputs
 * taken in pairs (z1, z2), u1 = ((z1 >> 11) + 1) 2^-53, u2 = (z2 >> 11) 2^-53, and the
 * Box-Muller pair sqrt(-2 ln u1) (cos 2 pi u2, sin 2 pi u2) in that order, computed in
 * fp64 and rounded once (a reading: the pages fix no generator).  Host only; errors:
 * TQ_ERR_INVALID_ARG (null), TQ_ERR_UNSUPPORTED (head_dim). */
tq_status tq_build_qjl_matrix(int head_dim, uint64_t seed, float* s_host);

/* Key writer for product-quantised rows: tq_write_kv's contract (raw, slots, pages,
 * status_dev -- NULL included -- and its errors) with rows of RBP(D, bits) bytes.
 *   mse_centroids  device, float[2^(bits-1)] from tq_codebook(head_dim, bits - 1)
 *   qjl_matrix     device, float[head_dim][head_dim] from tq_build_qjl_matrix
 * Per row (fp32): nu, y and the indices exactly as tq_write_kv at bits - 1; r = y -
 * c[idx]; gamma = ||r||; z_i = [sum_j S[i][j] r_j >= 0].  head_dim 64 or 128 and bits
 * 3..5 (TQ_ERR_UNSUPPORTED otherwise). */
tq_status tq_write_kv_prod(const void* raw, tq_dtype raw_dtype, int64_t num_tokens, int num_kv_heads,
                           int head_dim, int bits, const int64_t* slots, uint8_t* pages, int64_t num_blocks,
                           int block_size, const float* signs, const float* mse_centroids,
                           const float* qjl_matrix, int32_t* status_dev, void* stream);

/* Workspace bytes of tq_paged_decode_prod for these shapes (split-K partials and the
 * projected queries S R q); 0 when the arguments are invalid. */
size_t tq_paged_decode_prod_workspace(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                      int max_blocks_per_seq, int block_size);

/* Paged decode with product-quantised keys (k_bits = b in 3..5, rows of RBP(D, b)
 * bytes, k_mse_centroids float[2^(b-1)]) and MSE value rows (v_bits 2..5, RB(D, v_bits),
 * v_centroids float[2^v_bits]).  Every other argument, the status word and the errors
 * are those of tq_paged_decode.  The score of key row (idx, z, nu, gamma) is
 *   scale * nu * (<R q, c[idx]> + gamma sqrt(pi/2) / D * <S R q, 2z - 1>);
 * S R q is computed once per (sequence, q head) into the workspace.  head_dim 64 or 128
 * (TQ_ERR_UNSUPPORTED otherwise). */
tq_status tq_paged_decode_prod(const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int num_kv_heads,
                               int head_dim, const uint8_t* k_pages, int k_bits, const uint8_t* v_pages,
                               int v_bits, int64_t num_blocks, int block_size, const int32_t* block_table,
                               int max_blocks_per_seq, const int32_t* seq_lens, const float* signs,
                               const float* k_mse_centroids, const float* v_centroids, const float* qjl_matrix,
                               float scale, void* out, tq_dtype out_dtype, void* workspace,
                               size_t workspace_bytes, int32_t* status_dev, void* stream);

/* ---------------------------------------------------------------- recipe cache modes
 *
 * turboquant25 / turboquant35 ("vLLM Usage": Cache Dtypes -- recipe modes require
 * metadata; Metadata Validation Rules; Page Geometry -- recipe row-byte overrides;
 * "Architecture", vLLM Runtime Mapping: channels selected by energy, grouped MSE+QJL rows).
 * The pages give no numbers; the readings: the recipe name is the mean bits per channel.
 * A row's D channels form a high and a low group of d = D/2 channels each, coded at 3 and 2
 * bits (turboquant25) or 4 and 3 bits (turboquant35).  Each group is a product-quantised
 * vector of dimension d (tq_write_kv_prod's codec at head_dim d: (b-1)-bit MSE indices of
 * R_d x_g/||x_g||, d sign bits of S_d r, fp32 nu and gamma), R_d the RHT of dimension d and
 * seed 42 (tq_build_rotation(d, 42)), S_d = tq_build_qjl_matrix(d, 43), the MSE codebooks
 * tq_codebook(d, b - 1).  The row holds the high group's bytes, then the low group's.  K and
 * V both use recipe rows.  head_dim 64 or 128. */
typedef enum tq_recipe { TQ_RECIPE_TURBOQUANT25 = 25, TQ_RECIPE_TURBOQUANT35 = 35 } tq_recipe;

/* Bytes of one recipe row (56 / 72 at head_dim 128 for turboquant25 / 35); -1 when the recipe
 * or head_dim is unsupported. */
int64_t tq_recipe_row_bytes(int recipe, int head_dim);

/* The metadata check ("Metadata Validation Rules": sorted unique high-group indices, inside
 * the head, as many as the recipe expects -- D/2, fixed by the array shape) and the channel
 * order the kernels take.
 *   high_host   host int32[num_kv_heads][head_dim / 2]: each kv head's high-group channels.
 *   order_host  host int32[num_kv_heads][head_dim]: the high group, then the low group (the
 *               other channels, ascending).
 * Errors: TQ_ERR_INVALID_ARG naming the broken rule (an index outside [0, head_dim), not
 * sorted or repeated), an unknown recipe or an odd head_dim. */
tq_status tq_recipe_channel_order(int recipe, int head_dim, int num_kv_heads, const int32_t* high_host,
                                  int32_t* order_host);

/* Calibration ("Architecture": channels selected by energy): per kv head, the head_dim / 2
 * channels of largest energy sum_t x[t][h][c]^2 (fp64 sums; ties to the lower channel),
 * ascending.
 *   samples_host  host float[num_samples][num_kv_heads][head_dim]
 *   high_host     host int32[num_kv_heads][head_dim / 2], written. */
tq_status tq_recipe_calibrate(int recipe, int head_dim, int num_kv_heads, const float* samples_host,
                              int64_t num_samples, int32_t* high_host);

/* Recipe row writer: tq_write_kv's contract (raw, slots -- negative skipped, out of range an
 * error with nothing written --, pages of RB = tq_recipe_row_bytes, status_dev NULL or not)
 * for K or V.
 *   channel_order  device int32[num_kv_heads][head_dim] from tq_recipe_channel_order
 *   group_signs    device float[head_dim / 2] = tq_build_rotation(head_dim / 2, 42)
 *   mse_high       device float[2^(b_high - 1)] = tq_codebook(head_dim / 2, b_high - 1)
 *   mse_low        device float[2^(b_low - 1)]
 *   qjl_matrix     device float[head_dim / 2][head_dim / 2] = tq_build_qjl_matrix(head_dim / 2, 43)
 * Per group (fp32): the gathered channels x_g, nu = ||x_g||, y = R_d x_g / nu, the nearest
 * centroid indices, r = y - c[idx], gamma = ||r||, z_i = [(S_d r)_i >= 0]. */
tq_status tq_write_kv_recipe(const void* raw, tq_dtype raw_dtype, int64_t num_tokens, int num_kv_heads, int head_dim,
                             int recipe, const int64_t* slots, uint8_t* pages, int64_t num_blocks, int block_size,
                             const int32_t* channel_order, const float* group_signs, const float* mse_high,
                             const float* mse_low, const float* qjl_matrix, int32_t* status_dev, void* stream);

/* Workspace bytes of tq_paged_decode_recipe (split partials with two accumulators per group,
 * and the projected queries); 0 when the arguments are invalid. */
size_t tq_paged_decode_recipe_workspace(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int block_size);

/* Paged decode over recipe K and V pages (both of tq_recipe_row_bytes(recipe, head_dim)
 * bytes per row).  Every other argument, the status word and the errors are those of
 * tq_paged_decode; the codec arguments are those of tq_write_kv_recipe.  The score of key
 * row k is scale * sum_g nu_g (<R_d q_g, c_g[idx]> + gamma_g sqrt(pi/2)/d <S_d R_d q_g, 2z - 1>)
 * with q_g the query's channels of group g; the value of row v is, per group,
 * nu_g R_d^T (c_g[idx] + gamma_g sqrt(pi/2)/d S_d^T (2z - 1)) put back at the group's
 * channels. */
tq_status tq_paged_decode_recipe(const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, const uint8_t* k_pages, const uint8_t* v_pages, int recipe,
                                 int64_t num_blocks, int block_size, const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* channel_order, const float* group_signs,
                                 const float* mse_high, const float* mse_low, const float* qjl_matrix, float scale,
                                 void* out, tq_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_GB300_H */
