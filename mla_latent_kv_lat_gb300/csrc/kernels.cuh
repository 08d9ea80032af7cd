// Internal kernel interfaces of libmla (not part of the C ABI).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {

// Split-KV decode, evenly over G clusters by cost.  A valid sequence of len
// rows costs its 64-key tiles plus `piece_cost` more, the start of a piece
// (its queries' load, the previous piece's output, the pipeline's refill)
// counted in tiles; in sequence order these costs form one run of T units,
// sequence b's start-up units first and then its tiles, and cluster c takes
// units [c*T/G, (c+1)*T/G).  Where a cluster's range meets a sequence's tiles
// is a piece; it produces one partial result, in slot b + c (pieces are
// ordered by sequence, then cluster, and each starts at a sequence or cluster
// boundary).  Every cluster does the same cost (to one unit): a cluster whose
// range holds more pieces gets fewer tiles.
constexpr int kDecodeTile = 64;
MLA_DEVINL int64_t decode_seq_tiles(int32_t len) { return (static_cast<int64_t>(len) + kDecodeTile - 1) / kDecodeTile; }
MLA_DEVINL int64_t decode_seq_cost(int32_t len, int piece_cost) {
  return len > 0 ? decode_seq_tiles(len) + piece_cost : 0;
}
MLA_DEVINL int64_t decode_cluster_lo(int64_t T, int G, int c) { return T * c / G; }
// Sequence b's length if its rows [seq_start, seq_start + len) are a valid
// request (1 <= len <= max_len, inside the n_rows rows of the cache), else 0:
// the attention and combine kernels both skip such a sequence.
MLA_DEVINL int32_t decode_valid_len(const int64_t* seq_start, const int32_t* seq_len, int b, int32_t max_len,
                                    int64_t n_rows) {
  const int32_t len = seq_len[b];
  const int64_t s = seq_start[b];
  return (len >= 1 && len <= max_len && s >= 0 && s <= n_rows - len) ? len : 0;
}

struct CombineArgs {
  const float* ws_o;
  const float* ws_ml;
  const int64_t* seq_start;
  const int32_t* seq_len;
  void* o_lat;
  int64_t n_rows;
  int* err;
  int B, n_head, n_clusters, max_len;
  int piece_cost;           // the attention kernel's (see decode_seq_cost)
};

// C[t][h][n] = sum_k A[t][h][k] * W[h][k][n]  (absorb: bf16 A, K=128, N=512,
// fp16 out; late decompression: fp16 A, K=512, N=128, fp32 or fp16 out).
// W is bf16.
struct HeadGemmArgs {
  const void* a;            // bf16 or fp16 [T][H][K]
  const void* w;            // bf16 [H][K][N]
  void* c;                  // fp16 or fp32 [T][H][N]
  int T, H, K, N;
  int out_f32;
  int a_f16;
  int out_f16;
};

// Arguments of the tensor-core latent attention (prefill or decode partials).
struct AttnTcArgs {
  const void* q_lat;        // fp16 [rows][H][512]
  const void* q_pe;         // bf16 [rows][H][64]
  const void* kv;           // decode: bf16 [n_rows][576]; prefill: the fp16 [n_rows][576] staging copy
  const int8_t* kv_q;       // int8 [n_rows][576]
  const uint16_t* kv_d;     // fp16 [18][ld_d]
  int64_t ld_d;
  int64_t n_rows;           // rows of the cache arrays the kernel may address
  int n_head;
  float scale_log2;         // softmax scale * log2(e)
  // prefill
  int q_pos0;
  int64_t n_qrows;          // T * H
  void* o_lat;              // fp16 [T][H][512]
  float* lse;               // fp32 [T][H] or null
  // decode
  const int64_t* seq_start;
  const int32_t* seq_len;
  int n_seq;                // B
  int max_len;              // longest valid sequence (longer ones are skipped)
  int piece_cost;           // start-up cost of a piece in tiles (see decode_seq_cost)
  float* ws_o;              // fp32 [B + G - 1][H][512] partial o_lat per piece, normalised by its own sum
  float* ws_ml;             // fp32 [B + G - 1][H][2]   running max (log2 units) and sum
  int* err;
  uint32_t wait_us;
  int n_items;              // set by launch_attn_tc
};

// 3-D tiled tensor map of 16-bit elements with 128-byte swizzle, or 64-byte
// with swizzle_bytes = 64 (zero fill outside).
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                         int swizzle_bytes = 128);

// Prefill: n_items row tiles of 128.  Decode: n_items = number of clusters G
// (the pieces are found on the device).
cudaError_t launch_attn_tc(const AttnTcArgs& a, bool q8, bool decode, int n_items, cudaStream_t stream);
// Clusters a decode launch uses (one per SM pair); its workspace holds B + G - 1 pieces.
int decode_clusters();
int attn_tc_rows_per_item();

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t stream);
// Cache rows [0, rows) as fp16 [rows][576] in `out` (bf16 cache when kv is
// not null, else the q8_0 arrays kv_q / kv_d with scale row stride ld_d).
// Records MLA_ERR_RANGE in *err when a value is too large for fp16 (see
// bf16x2_absmax_overflows / f16_scale_overflows).
cudaError_t launch_stage_cache_f16(const void* kv, const int8_t* kv_q, const uint16_t* kv_d, int64_t ld_d,
                                   int64_t rows, void* out, int* err, cudaStream_t stream);
cudaError_t launch_head_gemm_tc(const HeadGemmArgs& g, int* err, uint32_t wait_us, cudaStream_t stream);
// Materialised prefill (pp_opt): decompress the visible rows into per-head
// fp16 keys/values, hc heads at a time, then 192/128 causal flash attention.
struct PpArgs {
  const void* q_nope;       // bf16 [T][H][128]
  const void* q_pe;         // bf16 [T][H][64]
  const void* kv;           // bf16 [>= q_pos0 + T][576], or null for a q8_0 cache:
  const int8_t* kv_q;       //   int8 [n][576] codes
  const uint16_t* kv_d;     //   fp16 [18][ld_d] scales
  int64_t ld_d;
  const void* wk_b;         // bf16 [H][128][512]
  const void* wv_b;         // bf16 [H][512][128]
  void* workspace;          // pp_workspace_bytes(H, T, q_pos0, hc)
  float* o;                 // fp32 [T][H][128]
  float* lse;               // fp32 [T][H] or null
  int T, H, q_pos0, hc;
  float scale_log2;
  int* err;
  uint32_t wait_us;
};
size_t pp_workspace_bytes(int H, int32_t T, int32_t q_pos0, int hc, bool q8);
cudaError_t launch_pp_prefill(const PpArgs& p, cudaStream_t stream);

// u[M][N] (fp32) = a[M][K] (fp16) . w_o[K][N] (fp16); K a multiple of 64, N of 64.
cudaError_t launch_wo_gemm_tc(const void* a, const void* w_o, float* u, int M, int K, int N, int* err,
                              uint32_t wait_us, cudaStream_t stream);
int device_sm_count();
// dst[i] = fp16(src[i]) for n bf16 values (records MLA_ERR_RANGE past fp16).
cudaError_t launch_bf16_to_f16(const void* src, void* dst, int64_t n, int* err, cudaStream_t stream);
cudaError_t launch_quantize_q8_0(const void* kv, int8_t* kv_q, uint16_t* kv_d, int64_t n, int64_t ld_d,
                                 cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(uint32_t wait_us, int* err, cudaStream_t stream);

}  // namespace mla
