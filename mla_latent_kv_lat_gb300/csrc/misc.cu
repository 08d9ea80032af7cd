// Per-head projections on CUDA cores (absorb and late decompression), the
// q8_0 cache quantiser, and the bounded-wait self-test.
#include "kernels.cuh"

namespace mla {

namespace {

// C[t][h][n] = sum_k A[t][h][k] W[h][k][n]; 64 x 64 output tile per CTA,
// 4 x 4 per thread, K staged 32 at a time.  ("MLA matrix absorption in
// ik_llama.cpp", sec. 3 for wk_b and sec. 4 for wv_b.)
__global__ void __launch_bounds__(256) head_gemm_simt_kernel(HeadGemmArgs g) {
  __shared__ __align__(16) float As[32][64 + 4];
  __shared__ __align__(16) float Ws[32][64 + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int n0 = blockIdx.x * 64, t0 = blockIdx.y * 64, h = blockIdx.z;
  const uint16_t* A = static_cast<const uint16_t*>(g.a);
  const uint16_t* Wt = static_cast<const uint16_t*>(g.w) + static_cast<int64_t>(h) * g.K * g.N;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += 32) {
    {
      const int t = tid >> 2, kc = (tid & 3) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t0 + t < g.T)
        v = *reinterpret_cast<const uint4*>(A + (static_cast<int64_t>(t0 + t) * g.H + h) * g.K + k0 + kc);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = g.a_f16 ? f16x2_to_f32(w[e]) : bf16x2_to_f32(w[e]);
        As[kc + 2 * e][t] = f.x;
        As[kc + 2 * e + 1][t] = f.y;
      }
    }
    {
      const int k = tid >> 3, nc = (tid & 7) * 8;
      const uint4 v = *reinterpret_cast<const uint4*>(Wt + static_cast<int64_t>(k0 + k) * g.N + n0 + nc);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = bf16x2_to_f32(w[e]);
        Ws[k][nc + 2 * e] = f.x;
        Ws[k][nc + 2 * e + 1] = f.y;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float4 a4 = *reinterpret_cast<const float4*>(&As[k][ty * 4]);
      const float4 w4 = *reinterpret_cast<const float4*>(&Ws[k][tx * 4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w}, wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= g.T) continue;
    const int64_t base = (static_cast<int64_t>(t) * g.H + h) * g.N + n0 + tx * 4;
    if (g.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(g.c) + base) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    } else {
      uint2 pk;
      pk.x = pack_f16x2(acc[i][0], acc[i][1]);
      pk.y = pack_f16x2(acc[i][2], acc[i][3]);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(g.c) + base) = pk;
    }
  }
}

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

__global__ void wait_timeout_selftest_kernel(uint32_t polls, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: phase 0 never completes.
  if (threadIdx.x == 0) (void)mbar_wait_bounded(&bar, 0, polls, err);
  __syncthreads();
}

}  // namespace

cudaError_t launch_head_gemm_simt(const HeadGemmArgs& g, cudaStream_t stream) {
  dim3 grid(g.N / 64, (g.T + 63) / 64, g.H);
  head_gemm_simt_kernel<<<grid, 256, 0, stream>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_quantize_q8_0(const void* kv, int8_t* kv_q, uint16_t* kv_d, int64_t n, int64_t ld_d,
                                 cudaStream_t stream) {
  const int64_t warps = n * kQ8Blocks;
  const int64_t blocks = (warps + 7) / 8;
  quantize_q8_0_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(kv), kv_q, reinterpret_cast<__half*>(kv_d), n, ld_d);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint32_t polls, int* err, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(polls, err);
  return cudaGetLastError();
}

}  // namespace mla
