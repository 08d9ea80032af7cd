/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention computed directly on
 * the compressed latent KV cache by matrix absorption, on one NVIDIA GB300
 * (sm_103a).
 *
 * The method is the one described on the page "MLA matrix absorption in
 * ik_llama.cpp" (czykbl.com/news/93068):
 *   sec. 3  K absorption: the K up-projection is folded into the query,
 *           q_lat[h] = wk_b[h]^T q_nope[h]                       (128 -> 512)
 *   sec. 5  move elision: scores are split into a RoPE part and a latent
 *           part, s = q_pe . k_pe + q_lat . c_kv, with no concatenation
 *   sec. 8.1 FlashMLA: causal online softmax over the latent cache
 *   sec. 4  V absorption: the weighted sum stays in latent space,
 *           o_lat = P c_kv, and W^UV is applied late, o[h] = wv_b[h] o_lat[h]
 *   sec. 8.1 MLA with a Q8_0-quantised latent cache.
 * Dimensions follow the DeepSeek GGUF metadata quoted on the page
 * "ik_llama.cpp PR #394 mainline DeepSeek GGUF support" (czykbl.com/news/94940),
 * sec. 2.1: kv_lora_rank 512, rope 64, nope 128, v 128, key_length 576.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked "device" are device memory of the current CUDA device,
 *   allocated, owned and freed by the caller.  No entry point allocates
 *   device or host memory, and none keeps a pointer after it returns.
 * - bf16 buffers are raw bfloat16 bit patterns (uint16_t); fp16 likewise.
 * - Inputs taken from the model (queries, cache, weights) are bf16.  The two
 *   intermediates of the path, q_lat and o_lat, are fp16: the attention
 *   contractions run on fp16 tensor-core operands (bf16 cache rows are
 *   converted on load, exactly for values inside the fp16 range), because
 *   rounding q_lat, P and o_lat to bf16 alone would cost about 2.8e-3 mean
 *   relative error of o, against about 0.6e-3 with fp16.
 * - fp16 range.  Where a bf16 value (cache row, q_pe) or an fp32 result
 *   (q_lat) becomes an fp16 operand, a magnitude of 65536 or more (bf16
 *   values between 65504 and 65536 do not exist), an infinity or a NaN is
 *   recorded as MLA_ERR_RANGE in the device error word; for a q8_0 cache the
 *   check is a block scale of 516 or more (127 x 516 > 65504).  A row whose
 *   partial score (before the softmax scale) exceeds 65504 in magnitude is
 *   recorded the same way when it makes the row maximum infinite or NaN.  The
 *   affected outputs are not defined; the others are computed as usual.
 * - Every device pointer must be 16-byte aligned (MLA_ERR_MISALIGNED).
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Work is enqueued asynchronously on it; host arguments are
 *   validated before anything is enqueued, and a validation error returns
 *   at once with nothing launched.
 * - Return value: MLA_OK or a negative mla_status.  Nothing aborts, traps or
 *   prints.  A launch error reported by the CUDA runtime maps to MLA_ERR_CUDA.
 * - The device address of the error word (and of the fixed scratch of
 *   mla_attn_decode_static) is looked up on a device's first call and kept
 *   for the life of the process: after cudaDeviceReset() on a device, do not
 *   call the library on that device again in the same process.
 * - Kernels that wait on asynchronous copies or tensor-core work bound every
 *   wait (0.5 s of the GPU's global timer).  A wait that runs out records
 *   MLA_ERR_TIMEOUT in a per-device error word, abandons its tile and
 *   returns; mla_get_device_error() reads and clears it.  While the word
 *   holds a timeout, any wait that does not complete at once gives up too, so
 *   a failing launch (and any launch after it, until the word is read) ends
 *   quickly.  The other device-side errors (MLA_ERR_RANGE, a skipped
 *   request) only record themselves: later launches run as usual.
 * - Dims other than kv_lora_rank 512, qk_rope 64, qk_nope 128, v_head 128,
 *   or n_head not a multiple of 16 in [16, 128], return MLA_ERR_UNSUPPORTED.
 *
 * Cache layouts
 * -------------
 * bf16 latent cache `kv`: row-major [n_rows][576] bf16.  Columns 0..511 hold
 *   c_kv (the latent), 512..575 hold k_pe (the RoPE key, shared by all
 *   heads): 1152 bytes per cached token, the "1.15 KB" of the method page,
 *   sec. 7.  Row j of a prefill cache holds position j.
 * q8_0 latent cache: the same 576 values per row, quantised in 18 blocks of
 *   32 (the Q8_0 cache of sec. 8.1; 18 x 34 = 612 bytes per row):
 *     kv_q  int8 [n_rows][576]   codes, row-major;
 *     kv_d  fp16 [18][n_rows]    block scales, block-major (scale of row j,
 *                                block b at kv_d[b * n_rows + j]).
 *   Element i of block b of row j is x = kv_d[b][j] * kv_q[j][32 b + i].
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mla_dims {
  int32_t n_head;        /* H: heads; a multiple of 16 in [16, 128]            */
  int32_t kv_lora_rank;  /* must be 512 (latent width)                         */
  int32_t qk_rope;       /* must be 64  (RoPE part of keys and queries)        */
  int32_t qk_nope;       /* must be 128 (non-RoPE query part per head)         */
  int32_t v_head;        /* must be 128 (value width per head)                 */
  float scale;           /* softmax scale on q.k, e.g. 1/sqrt(128 + 64)        */
} mla_dims;

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, bad positions */
  MLA_ERR_UNSUPPORTED = -2,  /* dims outside the supported set                 */
  MLA_ERR_MISALIGNED = -3,   /* a device pointer is not 16-byte aligned        */
  MLA_ERR_WORKSPACE = -4,    /* workspace missing or smaller than required     */
  MLA_ERR_CUDA = -5,         /* the CUDA runtime reported an error             */
  MLA_ERR_TIMEOUT = -6,      /* a device-side bounded wait ran out             */
  MLA_ERR_RANGE = -7         /* a value fp16 cannot hold met an fp16 operand   */
} mla_status;

/* Step 1, K absorption (method page sec. 3 and the q_nope2 line of sec. 4):
 *   q_lat[t][h][c] = sum_d q_nope[t][h][d] * wk_b[h][d][c]
 * q_nope  device bf16 [T][H][128]
 * wk_b    device bf16 [H][128][512]   (K up-projection, per head)
 * q_lat   device fp16 [T][H][512]     output, fp32 accumulation, rounded once
 * T >= 1.                                                                     */
int mla_absorb_q(const mla_dims* dims, const void* q_nope, const void* wk_b,
                 void* q_lat, int32_t T, void* stream);

/* Bytes of device workspace mla_attn_prefill / mla_attn_prefill_q8_0 need for
 * a cache of n_kv rows: an fp16 copy of the rows a prefill reads (1152 bytes
 * a row, rounded up to 256).  Returns 0 for invalid arguments.               */
size_t mla_prefill_workspace_size(const mla_dims* dims, int32_t n_kv);

/* Steps 2-4 for a causal prefill chunk (method page sec. 4, 5, 8.1):
 *   s[t][h][j] = scale * (q_pe[t][h] . k_pe[j] + q_lat[t][h] . c_kv[j])
 *   visible iff j <= q_pos0 + t   (query t sits at position q_pos0 + t)
 *   o_lat[t][h] = sum_j softmax_j(s[t][h]) * c_kv[j]
 * q_lat   device fp16 [T][H][512]
 * q_pe    device bf16 [T][H][64]
 * kv      device bf16 [n_kv][576]    latent cache (layout above)
 * workspace device, ws_bytes >= mla_prefill_workspace_size(dims, n_kv): the
 *         call first writes the rows it reads there as fp16 (every query
 *         tile reads every visible row, so they are converted once, not once
 *         per tile); its contents need not be kept between calls.
 * o_lat   device fp16 [T][H][512]    output
 * lse     device fp32 [T][H] or NULL; natural-log sum_j exp(s[t][h][j])
 * Requires T >= 1, q_pos0 >= 0 and q_pos0 + T <= n_kv.  Rows past
 * q_pos0 + T - 1 are never read.  MLA_ERR_WORKSPACE if the workspace is
 * missing or too small.                                                       */
int mla_attn_prefill(const mla_dims* dims, const void* q_lat, const void* q_pe,
                     const void* kv, int32_t n_kv, int32_t T, int32_t q_pos0,
                     void* workspace, size_t ws_bytes, void* o_lat, float* lse,
                     void* stream);

/* As mla_attn_prefill over a q8_0 latent cache (method page sec. 8.1):
 * kv_q device int8 [n_kv][576], kv_d device fp16 [18][n_kv].  Each block is
 * dequantised as fp16 scale x int8 code before it enters the scores and the
 * latent weighted sum.                                                        */
int mla_attn_prefill_q8_0(const mla_dims* dims, const void* q_lat, const void* q_pe,
                          const int8_t* kv_q, const uint16_t* kv_d, int32_t n_kv,
                          int32_t T, int32_t q_pos0, void* workspace, size_t ws_bytes,
                          void* o_lat, float* lse, void* stream);

/* Bytes of device workspace mla_attn_prefill_materialized needs for a chunk
 * of T queries at positions q_pos0.. with head_chunk heads decompressed at a
 * time (0 = all n_head): for one head chunk the fp16 keys (nope part) and
 * values (512 bytes a row and head), and for a q8_0 cache an fp16 copy of its
 * rows (1152 bytes a row), for the q_pos0 + T rows a chunk reads.  The size
 * serves either cache type.  Returns 0 for invalid arguments.                 */
size_t mla_prefill_materialized_workspace_size(const mla_dims* dims, int32_t T, int32_t q_pos0,
                                               int32_t head_chunk);

/* The materialised prefill ("pp_opt", method page sec. 8.4): for a long chunk
 * the keys and values of every visible row are decompressed from the latent
 * cache per head, once per call, and standard causal attention runs on them:
 *   k[j][h] = [ wk_b[h] c_kv[j] (128) | k_pe[j] (64) ],  v[j][h] = wv_b[h]^T c_kv[j]
 *   q[t][h] = [ q_nope[t][h] | q_pe[t][h] ]
 *   o[t][h] = sum_j softmax_j(scale * q[t][h] . k[j][h]) v[j][h],  j <= q_pos0 + t
 * (the un-absorbed definition of the method page, sec. 1, computed directly:
 * 640 FLOPs per visible pair and head instead of the absorbed 2176, plus the
 * decompression).  No late decompression follows: o is the per-head output.
 * q_nope device bf16 [T][H][128]; q_pe device bf16 [T][H][64]
 * kv     device bf16 [n_kv][576] latent cache; wk_b bf16 [H][128][512];
 *        wv_b bf16 [H][512][128]
 * head_chunk  heads decompressed at a time (0 = all): bounds the workspace the
 *        way ik_llama.cpp's -amb option bounds its attention buffers
 * workspace device, ws_bytes >= mla_prefill_materialized_workspace_size(...)
 * o      device fp32 [T][H][128] output;  lse fp32 [T][H] or NULL
 * Requires T >= 1, q_pos0 >= 0, q_pos0 + T <= n_kv; rows past q_pos0 + T - 1
 * are never read.  The nope parts of keys and queries, the values and the
 * probabilities are fp16 tensor-core operands, the RoPE parts the bf16 values
 * as given (fp32 accumulation); the fp16 range rules above apply.             */
int mla_attn_prefill_materialized(const mla_dims* dims, const void* q_nope, const void* q_pe,
                                  const void* kv, const void* wk_b, const void* wv_b, int32_t n_kv,
                                  int32_t T, int32_t q_pos0, int32_t head_chunk, void* workspace,
                                  size_t ws_bytes, float* o, float* lse, void* stream);

/* As mla_attn_prefill_materialized over a q8_0 latent cache (kv_q int8
 * [n_kv][576], kv_d fp16 [18][n_kv]; method page sec. 8.1 and 8.4): the rows
 * read are first dequantised to fp16 (scale x code, the values every q8_0
 * entry point uses), then decompressed with the weights converted to fp16.   */
int mla_attn_prefill_materialized_q8_0(const mla_dims* dims, const void* q_nope, const void* q_pe,
                                       const int8_t* kv_q, const uint16_t* kv_d, const void* wk_b,
                                       const void* wv_b, int32_t n_kv, int32_t T, int32_t q_pos0,
                                       int32_t head_chunk, void* workspace, size_t ws_bytes, float* o,
                                       float* lse, void* stream);

/* Bytes of device workspace mla_attn_decode / mla_attn_decode_q8_0 need for
 * B sequences (split-KV partial results): the keys of all sequences are split
 * evenly over G = (SM count / 2) clusters, which makes at most B + G - 1
 * pieces of H x 2056 bytes each.  max_len only bounds the lengths.  Returns 0
 * for invalid arguments.  The value depends only on the arguments and the
 * current device.                                                             */
size_t mla_decode_workspace_size(const mla_dims* dims, int32_t B, int32_t max_len);

/* Steps 2-4 for one new token per sequence (decode), with split-KV and a
 * log-sum-exp combine of the partial results:
 *   sequence b's cache rows are kv[seq_start[b] .. seq_start[b] + seq_len[b]),
 *   its query sits at position seq_len[b] - 1 and sees all of them.
 * q_lat      device fp16 [B][H][512];  q_pe device bf16 [B][H][64]
 * kv         device bf16 [n_rows][576] (rows of all sequences)
 * seq_start  device int64 [B]  first row of each sequence
 * seq_len    device int32 [B]  1 <= seq_len[b] <= max_len, rows inside kv
 * workspace  device, ws_bytes >= mla_decode_workspace_size(dims, B, max_len)
 * o_lat      device fp16 [B][H][512]  output
 * n_rows is the row count of kv (the q8_0 scale stride, and the bound of the
 * rows a sequence may name).  seq_start/seq_len are read on the device only:
 * a sequence with seq_len[b] < 1, seq_len[b] > max_len, seq_start[b] < 0 or
 * seq_start[b] + seq_len[b] > n_rows is skipped (no row of it is read and its
 * o_lat rows are left as they were) and recorded as MLA_ERR_INVALID_ARG in
 * the device error word; the other sequences are computed as usual.           */
int mla_attn_decode(const mla_dims* dims, const void* q_lat, const void* q_pe,
                    const void* kv, int64_t n_rows, const int64_t* seq_start,
                    const int32_t* seq_len, int32_t B, int32_t max_len,
                    void* workspace, size_t ws_bytes, void* o_lat, void* stream);

/* As mla_attn_decode over a q8_0 cache: kv_q int8 [n_rows][576], kv_d fp16
 * [18][n_rows].                                                               */
int mla_attn_decode_q8_0(const mla_dims* dims, const void* q_lat, const void* q_pe,
                         const int8_t* kv_q, const uint16_t* kv_d, int64_t n_rows,
                         const int64_t* seq_start, const int32_t* seq_len, int32_t B,
                         int32_t max_len, void* workspace, size_t ws_bytes,
                         void* o_lat, void* stream);

/* Split-KV decode exactly as mla_attn_decode (bf16 cache), for callers that
 * cannot allocate device memory: a plugin running inside a host engine that
 * owns every device allocation and forbids cudaMalloc, or a caller with no
 * allocator from which to take the decode workspace.  The pages have no
 * counterpart to this entry point; it exists only for such callers.
 * It takes no workspace: the split-KV partial results go to one fixed 32 MiB
 * device array inside the library, which every GPU that loads the library
 * holds until the process exits.  The entry point allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 * Limit: mla_decode_workspace_size(dims, B, max_len) must not exceed
 *   33554432 bytes (32 MiB); larger requests return MLA_ERR_WORKSPACE with
 *   nothing launched.  On GB300 (G = 76) at 128 heads: B = 8 needs 21.8 MB,
 *   B = 52 fits, B = 53 does not.
 * Sharing: every call uses the same array.  Calls whose work overlaps on the
 *   GPU (different streams without ordering, several host threads) race on it
 *   and corrupt each other's results; order them on one stream or with
 *   events.  Nothing in the array needs to start at zero: each call writes
 *   every partial it later reads, so the previous call's contents do no harm.
 * Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * Arguments, layouts and errors are otherwise those of mla_attn_decode.       */
int mla_attn_decode_static(const mla_dims* dims, const void* q_lat, const void* q_pe,
                           const void* kv, int64_t n_rows, const int64_t* seq_start,
                           const int32_t* seq_len, int32_t B, int32_t max_len,
                           void* o_lat, void* stream);

/* Step 5, late decompression (method page sec. 4, the wv_b line):
 *   o[t][h][e] = sum_c o_lat[t][h][c] * wv_b[h][c][e]
 * o_lat device fp16 [T][H][512]; wv_b device bf16 [H][512][128];
 * o     device fp32 [T][H][128] output.  T >= 1.                              */
int mla_late_decompress(const mla_dims* dims, const void* o_lat, const void* wv_b,
                        float* o, int32_t T, void* stream);

/* As mla_late_decompress, with o rounded once to fp16 (the type the output
 * projection below takes; bf16 would cost about 1.6e-3 mean relative error
 * of u by itself): o device fp16 [T][H][128].                                  */
int mla_late_decompress_f16(const mla_dims* dims, const void* o_lat, const void* wv_b,
                            void* o, int32_t T, void* stream);

/* Weight preparation, once per model load: dst = fp16(src) for n bf16 values
 * (n a multiple of 8), e.g. the output projection's w_o.  Exact for values in
 * fp16's normal range; a value fp16 cannot hold records MLA_ERR_RANGE.        */
int mla_convert_bf16_to_f16(const void* src, void* dst, int64_t n, void* stream);

/* The step after the path, the attention output projection (method page
 * sec. 4: the heads' outputs, flattened to H * 128, times wo -- the einsum
 * hdD,bhqd->bqD; the V up-projection stays a separate, earlier step):
 *   u[t][n] = sum_h sum_e o[t][h][e] * w_o[h][e][n]
 * o    device fp16 [T][H][128]   (mla_late_decompress_f16's output)
 * w_o  device fp16 [H][128][D]   (row-major [H*128][D]; the model's bf16
 *                                 weight converted once, mla_convert_bf16_to_f16)
 * u    device fp32 [T][D]        output, fp16 x fp16 products, fp32 accumulation
 * T >= 1; D (the hidden size) a multiple of 64, at most 1<<20
 * (MLA_ERR_UNSUPPORTED otherwise).  A dense GEMM on the tensor cores.         */
int mla_output_project(const mla_dims* dims, const void* o, const void* w_o, float* u,
                       int32_t T, int32_t D, void* stream);

/* Quantise n bf16 cache rows [n][576] to the q8_0 layout above (the producer
 * of the sec. 8.1 cache).  Per block: amax = max |x|, d = amax / 127 (fp32),
 * q = round-half-away-from-zero(x / d) clamped to [-127, 127] (0 when
 * amax = 0), stored scale fp16(d).  kv_d is [18][ld_d] with ld_d >= n: row
 * j's scales go to kv_d[b * ld_d + j].                                        */
int mla_quantize_q8_0(const void* kv, int8_t* kv_q, uint16_t* kv_d, int64_t n,
                      int64_t ld_d, void* stream);

/* The step before the path: write the cache rows of n new tokens (pages:
 * "MLA matrix absorption in ik_llama.cpp" sec. 3 -- the RoPE part of a key is
 * rotated by position and kept apart from the latent part; "llama.cpp KV
 * Cache 与注意力机制" sec. 2.2-2.3 -- new tokens go to the cache slots found
 * for them, keys rotated by ggml_rope_ext over n_rot = 64 dims; freq_base and
 * freq_scale as in the context log of "ik_llama.cpp discussion #586").
 * Row slot[j] of the cache receives [c_kv[j] (512, as given) | RoPE(k_pe[j],
 * pos[j]) (64)], RoPE pairing dims (2i, 2i+1) and turning pair i by
 * pos * freq_scale * freq_base^(-2i/64).
 * c_kv  device bf16 [n][512]; k_pe device bf16 [n][64] (not yet rotated);
 * pos   device int32 [n] positions (>= 0); slot device int64 [n] cache rows.
 * kv    device bf16 [n_rows][576] cache, or NULL; kv_q / kv_d the q8_0 cache
 *       (int8 [n_rows][576], fp16 [18][ld_d], ld_d >= n_rows) or both NULL;
 *       at least one cache.  The q8_0 row is the quantisation (as
 *       mla_quantize_q8_0) of the bf16 row.
 * A slot outside [0, n_rows) or a negative position is skipped on the
 * device and recorded as MLA_ERR_INVALID_ARG in the device error word.
 * The angles use freq_base and freq_scale as the floats given (the type ggml
 * keeps them in); the fraction of a turn is exact fixed-point arithmetic
 * (error < 2^-23 rad at any position), sine, cosine and the rotation are
 * fp32, with one rounding to bf16.
 * Host errors: n < 1, freq_base <= 1 or freq_scale <= 0 (MLA_ERR_INVALID_ARG),
 * pointers as above (MLA_ERR_MISALIGNED for kv_d only when odd).             */
int mla_rope_append(const void* c_kv, const void* k_pe, const int32_t* pos, const int64_t* slot,
                    int32_t n, float freq_base, float freq_scale, void* kv, int8_t* kv_q,
                    uint16_t* kv_d, int64_t ld_d, int64_t n_rows, void* stream);

/* Synchronise `stream`, then return and clear the current device's error
 * word: MLA_OK, or the first device-side error recorded since the last call
 * (MLA_ERR_TIMEOUT from a bounded wait, MLA_ERR_INVALID_ARG from the slot
 * check of mla_rope_append or the sequence check of the decodes,
 * MLA_ERR_RANGE from an fp16 conversion).  MLA_ERR_CUDA if the
 * synchronisation itself fails.                                               */
int mla_get_device_error(void* stream);

/* Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier phase nothing completes, giving up after `limit_us` microseconds
 * (1 <= limit_us <= 1<<20).  It records MLA_ERR_TIMEOUT in the device error word exactly as
 * a kernel's real waits do, and returns normally.  No counterpart on the
 * pages: it exists so that tests can check failure reporting without
 * hanging or faulting a GPU.                                                  */
int mla_selftest_wait_timeout(int32_t limit_us, void* stream);

/* Static description of a status code (never NULL).                           */
const char* mla_status_string(int status);

/* Library version string, e.g. "mla-gb300 0.1 sm_103a".                      */
const char* mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
