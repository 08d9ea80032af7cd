// The C ABI of libmla (declared in include/mla.h): argument validation,
// launch planning and the per-device error word.  Every step of the path runs
// in the kernels launched from here; there is no host or fallback compute.
#include <stdint.h>

#include <math.h>

#include <mutex>

#include "append.cuh"
#include "kernels.cuh"

namespace mla {
namespace {

__device__ int g_device_error;   // first device-side error since the last read

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

// Device address of the current device's error word (looked up once per
// device, with that device current; several host threads may make their
// first call at once).
cudaError_t error_word(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_err_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const mla_dims* d) {
  if (d == nullptr) return MLA_ERR_INVALID_ARG;
  if (d->kv_lora_rank != kLatent || d->qk_rope != kRope || d->qk_nope != kNope || d->v_head != kVHead)
    return MLA_ERR_UNSUPPORTED;
  if (d->n_head < 16 || d->n_head > 128 || d->n_head % 16 != 0) return MLA_ERR_UNSUPPORTED;
  if (!(d->scale > 0.f) || !(d->scale < 1e30f)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (p == nullptr) return MLA_ERR_INVALID_ARG;
    if (!aligned16(p)) return MLA_ERR_MISALIGNED;
  }
  return MLA_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

constexpr float kLog2eF = 1.4426950408889634f;

// Decode workspace: one partial per piece (a cluster's tile range meeting a
// sequence), at most B + G - 1 of them.
size_t decode_ws_bytes(int H, int32_t B) {
  const size_t slots = static_cast<size_t>(B + decode_clusters() - 1) * H;
  return slots * kLatent * sizeof(float) + slots * 2 * sizeof(float);
}

size_t prefill_ws_bytes(int32_t n_kv) {
  // fp16 staging copy of the cache rows, rounded up to whole 256-byte lines
  return (static_cast<size_t>(n_kv) * kRow * 2 + 255) & ~static_cast<size_t>(255);
}

int prefill_common(const mla_dims* dims, const void* q_lat, const void* q_pe, const void* kv,
                   const int8_t* kv_q, const uint16_t* kv_d, int32_t n_kv, int32_t T, int32_t q_pos0,
                   void* workspace, size_t ws_bytes, void* o_lat, float* lse, void* stream, bool q8) {
  int s = check_dims(dims);
  if (s != MLA_OK) return s;
  s = q8 ? check_ptrs({q_lat, q_pe, kv_q, kv_d, o_lat}) : check_ptrs({q_lat, q_pe, kv, o_lat});
  if (s != MLA_OK) return s;
  if (lse != nullptr && !aligned16(lse)) return MLA_ERR_MISALIGNED;
  if (T < 1 || q_pos0 < 0 || n_kv < 1) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(q_pos0) + T > n_kv) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < prefill_ws_bytes(n_kv)) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_MISALIGNED;
  int* err = nullptr;
  cudaError_t e = error_word(&err);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  const int64_t rows = static_cast<int64_t>(q_pos0) + T;     // rows past the last query are never read
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = launch_stage_cache_f16(q8 ? nullptr : kv, kv_q, kv_d, n_kv, rows, workspace, err, st);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  AttnTcArgs a = {};
  a.q_lat = q_lat;
  a.q_pe = q_pe;
  a.kv = workspace;
  a.ld_d = n_kv;
  a.n_rows = rows;
  a.n_head = dims->n_head;
  a.scale_log2 = dims->scale * kLog2eF;
  a.q_pos0 = q_pos0;
  a.n_qrows = static_cast<int64_t>(T) * dims->n_head;
  a.o_lat = o_lat;
  a.lse = lse;
  a.err = err;
  a.wait_us = kDefaultWaitUs;
  const int64_t items = (a.n_qrows + attn_tc_rows_per_item() - 1) / attn_tc_rows_per_item();
  if (items > (1 << 30)) return MLA_ERR_UNSUPPORTED;
  return to_status(launch_attn_tc(a, false, false, static_cast<int>(items), st));
}

int decode_common(const mla_dims* dims, const void* q_lat, const void* q_pe, const void* kv, const int8_t* kv_q,
                  const uint16_t* kv_d, int64_t n_rows, const int64_t* seq_start, const int32_t* seq_len,
                  int32_t B, int32_t max_len, void* workspace, size_t ws_bytes, void* o_lat, void* stream,
                  bool q8) {
  int s = check_dims(dims);
  if (s != MLA_OK) return s;
  s = q8 ? check_ptrs({q_lat, q_pe, kv_q, kv_d, o_lat}) : check_ptrs({q_lat, q_pe, kv, o_lat});
  if (s != MLA_OK) return s;
  if (seq_start == nullptr || seq_len == nullptr) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seq_start) & 7u) || (reinterpret_cast<uintptr_t>(seq_len) & 3u))
    return MLA_ERR_MISALIGNED;
  if (B < 1 || max_len < 1 || n_rows < 1) return MLA_ERR_INVALID_ARG;
  if (n_rows > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (B > 65535) return MLA_ERR_UNSUPPORTED;
  const size_t need = decode_ws_bytes(dims->n_head, B);
  if (workspace == nullptr || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_MISALIGNED;
  int* err = nullptr;
  cudaError_t e = error_word(&err);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  const int G = decode_clusters();
  const size_t slots = static_cast<size_t>(B + G - 1) * dims->n_head;
  AttnTcArgs a = {};
  a.q_lat = q_lat;
  a.q_pe = q_pe;
  a.kv = kv;
  a.kv_q = kv_q;
  a.kv_d = kv_d;
  a.ld_d = n_rows;
  a.n_rows = n_rows;
  a.n_head = dims->n_head;
  a.scale_log2 = dims->scale * kLog2eF;
  a.seq_start = seq_start;
  a.seq_len = seq_len;
  a.n_seq = B;
  a.max_len = max_len;
  // A piece's start-up (its queries' load, the previous piece's output, the
  // refill) measured ~7 us per piece at B=32: ~5 bf16 tiles or ~3 q8_0 tiles.
  a.piece_cost = q8 ? 3 : 5;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_ml = a.ws_o + slots * kLatent;
  a.err = err;
  a.wait_us = kDefaultWaitUs;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = launch_attn_tc(a, q8, true, G, st);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  CombineArgs c = {};
  c.ws_o = a.ws_o;
  c.ws_ml = a.ws_ml;
  c.seq_start = seq_start;
  c.seq_len = seq_len;
  c.n_rows = n_rows;
  c.max_len = max_len;
  c.err = err;
  c.o_lat = o_lat;
  c.B = B;
  c.n_head = dims->n_head;
  c.n_clusters = G;
  c.piece_cost = a.piece_cost;
  return to_status(launch_combine(c, st));
}

int head_gemm(const mla_dims* dims, const void* a, const void* w, void* c, int32_t T, int K, int N, bool f32,
              void* stream, bool out_f16 = false) {
  int s = check_dims(dims);
  if (s != MLA_OK) return s;
  s = check_ptrs({a, w, c});
  if (s != MLA_OK) return s;
  if (T < 1) return MLA_ERR_INVALID_ARG;
  int* err = nullptr;
  if (error_word(&err) != cudaSuccess) return MLA_ERR_CUDA;
  HeadGemmArgs g = {a, w, c, T, dims->n_head, K, N, f32 ? 1 : 0, (f32 || out_f16) ? 1 : 0, out_f16 ? 1 : 0};
  return to_status(launch_head_gemm_tc(g, err, kDefaultWaitUs, static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int mla_absorb_q(const mla_dims* dims, const void* q_nope, const void* wk_b, void* q_lat, int32_t T,
                 void* stream) {
  return head_gemm(dims, q_nope, wk_b, q_lat, T, kNope, kLatent, false, stream);
}

int mla_late_decompress(const mla_dims* dims, const void* o_lat, const void* wv_b, float* o, int32_t T,
                        void* stream) {
  return head_gemm(dims, o_lat, wv_b, o, T, kLatent, kVHead, true, stream);
}

int mla_late_decompress_f16(const mla_dims* dims, const void* o_lat, const void* wv_b, void* o, int32_t T,
                            void* stream) {
  return head_gemm(dims, o_lat, wv_b, o, T, kLatent, kVHead, false, stream, true);
}

size_t mla_prefill_materialized_workspace_size(const mla_dims* dims, int32_t T, int32_t q_pos0, int32_t head_chunk) {
  if (check_dims(dims) != MLA_OK || T < 1 || q_pos0 < 0 || head_chunk < 0 || head_chunk > dims->n_head) return 0;
  if (static_cast<int64_t>(q_pos0) + T > INT32_MAX) return 0;
  // enough for either cache type (a q8_0 cache adds the fp16 staging copy)
  return pp_workspace_bytes(dims->n_head, T, q_pos0, head_chunk == 0 ? dims->n_head : head_chunk, true);
}

int materialized_common(const mla_dims* dims, const void* q_nope, const void* q_pe, const void* kv,
                        const int8_t* kv_q, const uint16_t* kv_d, const void* wk_b, const void* wv_b, int32_t n_kv,
                        int32_t T, int32_t q_pos0, int32_t head_chunk, void* workspace, size_t ws_bytes, float* o,
                        float* lse, void* stream) {
  const bool q8 = kv == nullptr;
  int s = check_dims(dims);
  if (s != MLA_OK) return s;
  s = q8 ? check_ptrs({q_nope, q_pe, kv_q, kv_d, wk_b, wv_b, o}) : check_ptrs({q_nope, q_pe, kv, wk_b, wv_b, o});
  if (s != MLA_OK) return s;
  if (lse != nullptr && !aligned16(lse)) return MLA_ERR_MISALIGNED;
  if (T < 1 || q_pos0 < 0 || n_kv < 1 || head_chunk < 0 || head_chunk > dims->n_head) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(q_pos0) + T > n_kv) return MLA_ERR_INVALID_ARG;
  const int hc = head_chunk == 0 ? dims->n_head : head_chunk;
  if (workspace == nullptr || ws_bytes < pp_workspace_bytes(dims->n_head, T, q_pos0, hc, q8)) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_MISALIGNED;
  PpArgs p = {};
  p.q_nope = q_nope;
  p.q_pe = q_pe;
  p.kv = q8 ? nullptr : kv;
  p.kv_q = kv_q;
  p.kv_d = kv_d;
  p.ld_d = n_kv;
  p.wk_b = wk_b;
  p.wv_b = wv_b;
  p.workspace = workspace;
  p.o = o;
  p.lse = lse;
  p.T = T;
  p.H = dims->n_head;
  p.q_pos0 = q_pos0;
  p.hc = hc;
  p.scale_log2 = dims->scale * kLog2eF;
  p.wait_us = kDefaultWaitUs;
  if (error_word(&p.err) != cudaSuccess) return MLA_ERR_CUDA;
  return to_status(launch_pp_prefill(p, static_cast<cudaStream_t>(stream)));
}

int mla_attn_prefill_materialized(const mla_dims* dims, const void* q_nope, const void* q_pe, const void* kv,
                                  const void* wk_b, const void* wv_b, int32_t n_kv, int32_t T, int32_t q_pos0,
                                  int32_t head_chunk, void* workspace, size_t ws_bytes, float* o, float* lse,
                                  void* stream) {
  if (kv == nullptr) return MLA_ERR_INVALID_ARG;
  return materialized_common(dims, q_nope, q_pe, kv, nullptr, nullptr, wk_b, wv_b, n_kv, T, q_pos0, head_chunk,
                             workspace, ws_bytes, o, lse, stream);
}

int mla_attn_prefill_materialized_q8_0(const mla_dims* dims, const void* q_nope, const void* q_pe,
                                       const int8_t* kv_q, const uint16_t* kv_d, const void* wk_b, const void* wv_b,
                                       int32_t n_kv, int32_t T, int32_t q_pos0, int32_t head_chunk, void* workspace,
                                       size_t ws_bytes, float* o, float* lse, void* stream) {
  if (kv_q == nullptr || kv_d == nullptr) return MLA_ERR_INVALID_ARG;
  return materialized_common(dims, q_nope, q_pe, nullptr, kv_q, kv_d, wk_b, wv_b, n_kv, T, q_pos0, head_chunk,
                             workspace, ws_bytes, o, lse, stream);
}

int mla_output_project(const mla_dims* dims, const void* o, const void* w_o, float* u, int32_t T, int32_t D,
                       void* stream) {
  int s = check_dims(dims);
  if (s != MLA_OK) return s;
  s = check_ptrs({o, w_o, u});
  if (s != MLA_OK) return s;
  if (T < 1 || D < 64) return MLA_ERR_INVALID_ARG;
  if (D % 64 != 0 || D > (1 << 20)) return MLA_ERR_UNSUPPORTED;
  int* err = nullptr;
  if (error_word(&err) != cudaSuccess) return MLA_ERR_CUDA;
  return to_status(launch_wo_gemm_tc(o, w_o, u, T, dims->n_head * kVHead, D, err, kDefaultWaitUs,
                                     static_cast<cudaStream_t>(stream)));
}

size_t mla_prefill_workspace_size(const mla_dims* dims, int32_t n_kv) {
  if (check_dims(dims) != MLA_OK || n_kv < 1) return 0;
  return prefill_ws_bytes(n_kv);
}

int mla_attn_prefill(const mla_dims* dims, const void* q_lat, const void* q_pe, const void* kv, int32_t n_kv,
                     int32_t T, int32_t q_pos0, void* workspace, size_t ws_bytes, void* o_lat, float* lse,
                     void* stream) {
  return prefill_common(dims, q_lat, q_pe, kv, nullptr, nullptr, n_kv, T, q_pos0, workspace, ws_bytes, o_lat, lse,
                        stream, false);
}

int mla_attn_prefill_q8_0(const mla_dims* dims, const void* q_lat, const void* q_pe, const int8_t* kv_q,
                          const uint16_t* kv_d, int32_t n_kv, int32_t T, int32_t q_pos0, void* workspace,
                          size_t ws_bytes, void* o_lat, float* lse, void* stream) {
  return prefill_common(dims, q_lat, q_pe, nullptr, kv_q, kv_d, n_kv, T, q_pos0, workspace, ws_bytes, o_lat, lse,
                        stream, true);
}

size_t mla_decode_workspace_size(const mla_dims* dims, int32_t B, int32_t max_len) {
  if (check_dims(dims) != MLA_OK || B < 1 || max_len < 1) return 0;
  return decode_ws_bytes(dims->n_head, B);
}

int mla_attn_decode(const mla_dims* dims, const void* q_lat, const void* q_pe, const void* kv, int64_t n_rows,
                    const int64_t* seq_start, const int32_t* seq_len, int32_t B, int32_t max_len, void* workspace,
                    size_t ws_bytes, void* o_lat, void* stream) {
  return decode_common(dims, q_lat, q_pe, kv, nullptr, nullptr, n_rows, seq_start, seq_len, B, max_len, workspace,
                       ws_bytes, o_lat, stream, false);
}

int mla_attn_decode_q8_0(const mla_dims* dims, const void* q_lat, const void* q_pe, const int8_t* kv_q,
                         const uint16_t* kv_d, int64_t n_rows, const int64_t* seq_start, const int32_t* seq_len,
                         int32_t B, int32_t max_len, void* workspace, size_t ws_bytes, void* o_lat, void* stream) {
  return decode_common(dims, q_lat, q_pe, nullptr, kv_q, kv_d, n_rows, seq_start, seq_len, B, max_len, workspace,
                       ws_bytes, o_lat, stream, true);
}

int mla_convert_bf16_to_f16(const void* src, void* dst, int64_t n, void* stream) {
  int s = check_ptrs({src, dst});
  if (s != MLA_OK) return s;
  if (n < 1 || n % 8 != 0) return MLA_ERR_INVALID_ARG;
  int* err = nullptr;
  if (error_word(&err) != cudaSuccess) return MLA_ERR_CUDA;
  return to_status(launch_bf16_to_f16(src, dst, n, err, static_cast<cudaStream_t>(stream)));
}

int mla_quantize_q8_0(const void* kv, int8_t* kv_q, uint16_t* kv_d, int64_t n, int64_t ld_d, void* stream) {
  int s = check_ptrs({kv, kv_q});
  if (s != MLA_OK) return s;
  if (kv_d == nullptr) return MLA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(kv_d) & 1u) return MLA_ERR_MISALIGNED;
  if (n < 1 || ld_d < n) return MLA_ERR_INVALID_ARG;
  if ((n * kQ8Blocks + 7) / 8 > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  return to_status(launch_quantize_q8_0(kv, kv_q, kv_d, n, ld_d, static_cast<cudaStream_t>(stream)));
}

int mla_rope_append(const void* c_kv, const void* k_pe, const int32_t* pos, const int64_t* slot, int32_t n,
                    float freq_base, float freq_scale, void* kv, int8_t* kv_q, uint16_t* kv_d, int64_t ld_d,
                    int64_t n_rows, void* stream) {
  int s = check_ptrs({c_kv, k_pe, pos, slot});
  if (s != MLA_OK) return s;
  if (n < 1 || n_rows < 1) return MLA_ERR_INVALID_ARG;
  if (!(freq_base > 1.f) || !(freq_scale > 0.f) || !isfinite(freq_base) || !isfinite(freq_scale))
    return MLA_ERR_INVALID_ARG;
  if (kv == nullptr && kv_q == nullptr) return MLA_ERR_INVALID_ARG;
  if ((kv_q == nullptr) != (kv_d == nullptr)) return MLA_ERR_INVALID_ARG;
  if (kv != nullptr && !aligned16(kv)) return MLA_ERR_MISALIGNED;
  if (kv_q != nullptr) {
    if (!aligned16(kv_q)) return MLA_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(kv_d) & 1u) return MLA_ERR_MISALIGNED;
    if (ld_d < n_rows) return MLA_ERR_INVALID_ARG;
  }
  RopeAppendArgs a = {};
  a.c_kv = static_cast<const uint16_t*>(c_kv);
  a.k_pe = static_cast<const uint16_t*>(k_pe);
  a.pos = pos;
  a.slot = slot;
  a.n = n;
  a.kv = static_cast<uint16_t*>(kv);
  a.kv_q = kv_q;
  a.kv_d = kv_d;
  a.ld_d = ld_d;
  a.n_rows = n_rows;
  if (error_word(&a.err) != cudaSuccess) return MLA_ERR_CUDA;
  // turns per position of pair i, frac(t_i) as 0.64 fixed point: two exact
  // 32-bit halves of the double's fraction
  const double kTwoPi = 6.283185307179586;
  for (int i = 0; i < kRope / 2; ++i) {
    double t = static_cast<double>(freq_scale) * pow(static_cast<double>(freq_base), -2.0 * i / kRope) / kTwoPi;
    t -= floor(t);
    const double hi = floor(ldexp(t, 32));
    const double lo = nearbyint(ldexp(ldexp(t, 32) - hi, 32));
    a.turn[i] = (static_cast<uint64_t>(hi) << 32) + static_cast<uint64_t>(lo);
  }
  return to_status(launch_rope_append(a, static_cast<cudaStream_t>(stream)));
}

int mla_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  int* err = nullptr;
  if (error_word(&err) != cudaSuccess) return MLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return v;
}

int mla_selftest_wait_timeout(int32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > (1 << 20)) return MLA_ERR_INVALID_ARG;
  int* err = nullptr;
  if (error_word(&err) != cudaSuccess) return MLA_ERR_CUDA;
  return to_status(launch_wait_timeout_selftest(static_cast<uint32_t>(limit_us), err,
                                                static_cast<cudaStream_t>(stream)));
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported dims or size";
    case MLA_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_TIMEOUT: return "device-side bounded wait timed out";
    case MLA_ERR_RANGE: return "value outside the fp16 range met an fp16 operand";
    default: return "unknown status";
  }
}

const char* mla_version(void) { return "mla-gb300 0.1 sm_103a"; }

}  // extern "C"
