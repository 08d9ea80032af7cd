// mla_attn_decode_static: the split-KV decode for callers that cannot
// allocate device memory.
//
// Some callers run inside a host that owns every device allocation and does
// not let plugins call cudaMalloc (an inference engine's custom-operator
// interface with a fixed memory plan, for example), or have no allocator of
// their own to obtain the decode workspace from.  This entry point needs no
// workspace argument: its split-KV partial results live in one file-scope
// device array of fixed size, which every GPU that loads this library holds
// until the process exits.
#include <mutex>

#include "kernels.cuh"

namespace {

// Maximum scratch: 32 MiB.  A decode needs (B + G - 1) * H * 2056 bytes of it
// (G = SM count / 2 clusters; per piece and head, fp32 partial sums of 512
// latent values plus a running max and sum), e.g. B = 8 sequences at 128
// heads on GB300 (G = 76) use 21.8 MB.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device, with that device current, and cached for the life of
// the process (after a cudaDeviceReset of that device the cached address is
// stale: the header tells callers not to use the library on it again).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_attn_decode_static(const mla_dims* dims, const void* q_lat, const void* q_pe, const void* kv,
                                      int64_t n_rows, const int64_t* seq_start, const int32_t* seq_len, int32_t B,
                                      int32_t max_len, void* o_lat, void* stream) {
  const size_t need = mla_decode_workspace_size(dims, B, max_len);
  // Arguments no workspace can serve: mla_attn_decode's own checks give the
  // status (they run before its workspace check, so nothing is launched).
  if (need == 0)
    return mla_attn_decode(dims, q_lat, q_pe, kv, n_rows, seq_start, seq_len, B, max_len, nullptr, 0, o_lat, stream);
  if (need > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int s = scratch_for_current_device(&scratch);
  if (s != MLA_OK) return s;
  return mla_attn_decode(dims, q_lat, q_pe, kv, n_rows, seq_start, seq_len, B, max_len, scratch,
                         kStaticScratchBytes, o_lat, stream);
}
