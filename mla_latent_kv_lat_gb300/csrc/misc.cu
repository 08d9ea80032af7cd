// The split-KV combine of the decode partials, the q8_0 cache quantiser and
// the bounded-wait self-test.
#include "kernels.cuh"

namespace mla {

namespace {

// One warp per (row, block of 32): amax, d = amax/127, codes = round(x/d).
// The rounding and scale rules are those of the q8_0 cache format (method
// page sec. 8.1; block size from the cache size in discussion #586).
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const uint16_t* kv, int8_t* kv_q, __half* kv_d,
                                                            int64_t n, int64_t ld_d) {
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= n * kQ8Blocks) return;
  const int64_t row = wid / kQ8Blocks;
  const int blk = static_cast<int>(wid % kQ8Blocks);
  const int64_t idx = row * kRow + blk * kQ8Block + lane;
  const float x = bf16_to_f32(kv[idx]);
  const float amax = warp_max(fabsf(x));
  const float d = amax / 127.0f;
  int q = 0;
  if (amax > 0.f) {
    q = static_cast<int>(roundf(x / d));
    q = max(-127, min(127, q));
  }
  kv_q[idx] = static_cast<int8_t>(q);
  if (lane == 0) kv_d[static_cast<int64_t>(blk) * ld_d + row] = __float2half_rn(d);
}

__global__ void wait_timeout_selftest_kernel(uint32_t wait_us, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: phase 0 never completes.
  if (threadIdx.x == 0) (void)mbar_wait_bounded(&bar, 0, wait_us, err);
  __syncthreads();
}

}  // namespace

cudaError_t launch_quantize_q8_0(const void* kv, int8_t* kv_q, uint16_t* kv_d, int64_t n, int64_t ld_d,
                                 cudaStream_t stream) {
  const int64_t warps = n * kQ8Blocks;
  const int64_t blocks = (warps + 7) / 8;
  quantize_q8_0_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(kv), kv_q, reinterpret_cast<__half*>(kv_d), n, ld_d);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint32_t wait_us, int* err, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(wait_us, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Split-KV combine: merge the per-split partials of each (sequence, head) --
// o_s normalised by its own sum l_s, running max m_s in log2 units -- by
// log-sum-exp, and write o_lat in fp16.
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(128) combine_kernel(CombineArgs c) {
  const int b = blockIdx.x / c.n_head, h = blockIdx.x % c.n_head;
  const int64_t len = c.seq_len[b];
  const int ns = static_cast<int>(min(static_cast<int64_t>(c.n_split), (len + c.chunk - 1) / c.chunk));
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) {
    const int64_t slot = (static_cast<int64_t>(b) * c.n_split + s) * c.n_head + h;
    M = fmaxf(M, c.ws_ml[2 * slot]);
  }
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int col = threadIdx.x * 4;
  for (int s = 0; s < ns; ++s) {
    const int64_t slot = (static_cast<int64_t>(b) * c.n_split + s) * c.n_head + h;
    // partials are normalised by their own sum l_s: weight 2^(m_s - M) * l_s
    const float w = exp2f(c.ws_ml[2 * slot] - M) * c.ws_ml[2 * slot + 1];
    L += w;
    const float4 o = *reinterpret_cast<const float4*>(c.ws_o + slot * kLatent + col);
    acc.x = fmaf(w, o.x, acc.x);
    acc.y = fmaf(w, o.y, acc.y);
    acc.z = fmaf(w, o.z, acc.z);
    acc.w = fmaf(w, o.w, acc.w);
  }
  const float inv = 1.f / L;
  uint16_t* out = static_cast<uint16_t*>(c.o_lat) + (static_cast<int64_t>(b) * c.n_head + h) * kLatent + col;
  uint2 pk;
  pk.x = pack_f16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_f16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out) = pk;
}
}  // namespace

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t stream) {
  combine_kernel<<<c.B * c.n_head, 128, 0, stream>>>(c);
  return cudaGetLastError();
}


}  // namespace mla
