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
  // This sequence's tiles [Sb, Eb) in the run of all sequences' tiles, and
  // the clusters whose ranges meet it (one piece each, slot b + cluster).
  int64_t T = 0, Sb = 0;
  for (int q = 0; q < c.B; ++q) {
    const int64_t t = decode_seq_tiles(c.seq_len[q]);
    if (q < b) Sb += t;
    T += t;
  }
  const int64_t Eb = Sb + decode_seq_tiles(c.seq_len[b]);
  const int G = c.n_clusters;
  int c0 = static_cast<int>(min(static_cast<int64_t>(G - 1), Sb * G / max(T, static_cast<int64_t>(1))));
  while (c0 > 0 && decode_cluster_lo(T, G, c0) > Sb) --c0;
  while (c0 + 1 < G && decode_cluster_lo(T, G, c0 + 1) <= Sb) ++c0;
  float M = -INFINITY;
  for (int cl = c0; cl < G && decode_cluster_lo(T, G, cl) < Eb; ++cl) {
    if (decode_cluster_lo(T, G, cl + 1) <= decode_cluster_lo(T, G, cl)) continue;   // empty range
    const int64_t slot = static_cast<int64_t>(b + cl) * c.n_head + h;
    M = fmaxf(M, c.ws_ml[2 * slot]);
  }
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int col = threadIdx.x * 4;
  for (int cl = c0; cl < G && decode_cluster_lo(T, G, cl) < Eb; ++cl) {
    if (decode_cluster_lo(T, G, cl + 1) <= decode_cluster_lo(T, G, cl)) continue;
    const int64_t slot = static_cast<int64_t>(b + cl) * c.n_head + h;
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

// ---------------------------------------------------------------------------
// Prefill operand staging: the cache rows a prefill reads, as fp16 [rows][576]
// (latent and RoPE parts), the type the latent tensor-core products take.
// Every query tile of a prefill reads every visible cache row, so converting
// once here replaces one conversion per tile inside the attention kernel.
// bf16 -> fp16 is exact over fp16's normal range (|x| in [2^-14, 65504]);
// q8_0 codes become fp16(scale x code), the value the decode kernel forms.
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(256) cache_bf16_to_f16_kernel(const uint4* kv, uint4* out, int64_t n_units) {
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(kv + u);
    uint4 o;
    float2 f;
    f = bf16x2_to_f32(v.x); o.x = pack_f16x2(f.x, f.y);
    f = bf16x2_to_f32(v.y); o.y = pack_f16x2(f.x, f.y);
    f = bf16x2_to_f32(v.z); o.z = pack_f16x2(f.x, f.y);
    f = bf16x2_to_f32(v.w); o.w = pack_f16x2(f.x, f.y);
    out[u] = o;
  }
}

// One thread per 16 codes (half a q8_0 block): 36 per row.
__global__ void __launch_bounds__(256) cache_q8_0_to_f16_kernel(const int8_t* kv_q, const __half* kv_d, int64_t ld_d,
                                                                 uint4* out, int64_t rows) {
  const int64_t n_units = rows * (kRow / 16);
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = u / (kRow / 16);
    const int c = static_cast<int>(u % (kRow / 16));
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(kv_q + row * kRow) + c);
    const float d = __half2float(__ldg(kv_d + static_cast<int64_t>(c >> 1) * ld_d + row));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a0 = static_cast<float>(static_cast<int8_t>(w[k] & 0xFF));
      const float a1 = static_cast<float>(static_cast<int8_t>((w[k] >> 8) & 0xFF));
      const float a2 = static_cast<float>(static_cast<int8_t>((w[k] >> 16) & 0xFF));
      const float a3 = static_cast<float>(static_cast<int8_t>(w[k] >> 24));
      h[2 * k] = pack_f16x2(a0 * d, a1 * d);
      h[2 * k + 1] = pack_f16x2(a2 * d, a3 * d);
    }
    out[2 * u] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * u + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

unsigned stage_blocks(int64_t n_units) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  return static_cast<unsigned>(max(static_cast<int64_t>(1), min(cap, (n_units + 255) / 256)));
}
}  // namespace

cudaError_t launch_stage_cache_f16(const void* kv, const int8_t* kv_q, const uint16_t* kv_d, int64_t ld_d,
                                   int64_t rows, void* out, cudaStream_t stream) {
  if (kv != nullptr) {
    const int64_t n_units = rows * (kRow / 8);
    cache_bf16_to_f16_kernel<<<stage_blocks(n_units), 256, 0, stream>>>(static_cast<const uint4*>(kv),
                                                                         static_cast<uint4*>(out), n_units);
  } else {
    const int64_t n_units = rows * (kRow / 16);
    cache_q8_0_to_f16_kernel<<<stage_blocks(n_units), 256, 0, stream>>>(
        kv_q, reinterpret_cast<const __half*>(kv_d), ld_d, static_cast<uint4*>(out), rows);
  }
  return cudaGetLastError();
}


}  // namespace mla
