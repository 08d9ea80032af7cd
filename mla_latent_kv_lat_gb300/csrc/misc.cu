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
// Split-KV combine: merge the per-piece partials of each (sequence, head) --
// o_s normalised by its own sum l_s, running max m_s in log2 units -- by
// log-sum-exp, and write o_lat in fp16.  One warp per (sequence, head), eight
// heads per block; a lane holds 16 of the 512 columns (four 16-byte pieces,
// 128 columns apart, so that each load instruction covers 512 contiguous
// bytes), and the loads of up to four partials are in flight at once.
// Launched as a programmatic dependent of the attention kernel: the block
// sets up (the sequence's tile range) while the attention kernel drains, and
// waits for its completion before the first read of the workspace.
// ---------------------------------------------------------------------------
namespace {
constexpr int kCombHeads = 8;

__global__ void __launch_bounds__(32 * kCombHeads) combine_kernel(CombineArgs c) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This sequence's costs [Sb, Eb) in the run of all sequences' costs; its
  // tiles are [Sb + piece_cost, Eb).
  __shared__ long long red[2][kCombHeads];
  long long tb = 0, tt = 0;
  for (int q = threadIdx.x; q < c.B; q += blockDim.x) {
    const long long t = decode_seq_cost(decode_valid_len(c.seq_start, c.seq_len, q, c.max_len, c.n_rows),
                                        c.piece_cost);
    tt += t;
    if (q < b) tb += t;
  }
  tb = warp_sum_i64(tb);
  tt = warp_sum_i64(tt);
  if (lane == 0) {
    red[0][warp] = tb;
    red[1][warp] = tt;
  }
  __syncthreads();
  int64_t Sb = 0, T = 0;
#pragma unroll
  for (int w = 0; w < kCombHeads; ++w) {
    Sb += red[0][w];
    T += red[1][w];
  }
  const int32_t len_b = decode_valid_len(c.seq_start, c.seq_len, b, c.max_len, c.n_rows);
  if (len_b == 0) {                  // an invalid request: skipped by the attention kernel too
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(c.err, MLA_ERR_INVALID_ARG);
    return;
  }
  const int64_t Eb = Sb + decode_seq_cost(len_b, c.piece_cost);
  const int64_t Rb = Sb + c.piece_cost;                // the first of its tiles
  const int G = c.n_clusters;
  // The clusters' range starts lo(x) = T x / G, x = 0..G, once per block (a
  // 64-bit division each: computed on the fly they made this kernel
  // instruction-bound).
  extern __shared__ long long s_lo[];
  for (int x = threadIdx.x; x <= G; x += blockDim.x) s_lo[x] = decode_cluster_lo(T, G, x);
  __syncthreads();
  auto lo = [&](int x) { return s_lo[x]; };
  // The first cluster whose range meets the tiles [Rb, Eb): ranges are
  // [lo(c), lo(c+1)); every later one that meets them has lo(c) < Eb.
  int c0 = static_cast<int>(min(static_cast<int64_t>(G - 1), Rb * G / max(T, static_cast<int64_t>(1))));
  while (c0 > 0 && lo(c0) > Rb) --c0;
  while (c0 + 1 < G && lo(c0 + 1) <= Rb) ++c0;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the attention kernel's partials are complete
  const int h = blockIdx.y * kCombHeads + warp;
  if (h >= c.n_head) return;
  // Pass 1: the largest running max over the pieces (a lane per piece).
  float M = -INFINITY;
  for (int x = c0 + lane; x < G && lo(x) < Eb; x += 32) {
    if (lo(x + 1) <= lo(x)) continue;   // empty range
    M = fmaxf(M, c.ws_ml[2 * ((static_cast<int64_t>(b) + x) * c.n_head + h)]);
  }
  M = warp_max(M);
  // Pass 2: weights 2^(m_s - M) * l_s and the weighted partials.
  float L = 0.f;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  int cl = c0;
  while (cl < G && lo(cl) < Eb) {
    // the next (up to) four non-empty pieces
    int64_t slot[4];
    bool has[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      while (cl < G && lo(cl) < Eb && lo(cl + 1) <= lo(cl)) ++cl;     // empty range
      has[j] = cl < G && lo(cl) < Eb;
      slot[j] = (static_cast<int64_t>(b) + cl) * c.n_head + h;
      if (has[j]) ++cl;
    }
    float4 v[4][4];
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w[j] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) v[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (has[j]) {
        const float4* src = reinterpret_cast<const float4*>(c.ws_o + slot[j] * kLatent) + lane;
#pragma unroll
        for (int k = 0; k < 4; ++k) v[j][k] = src[32 * k];
        w[j] = exp2f(c.ws_ml[2 * slot[j]] - M) * c.ws_ml[2 * slot[j] + 1];
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      L += w[j];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x = fmaf(w[j], v[j][k].x, acc[k].x);
        acc[k].y = fmaf(w[j], v[j][k].y, acc[k].y);
        acc[k].z = fmaf(w[j], v[j][k].z, acc[k].z);
        acc[k].w = fmaf(w[j], v[j][k].w, acc[k].w);
      }
    }
  }
  const float inv = 1.f / L;
  uint2* out = reinterpret_cast<uint2*>(static_cast<uint16_t*>(c.o_lat) +
                                        (static_cast<int64_t>(b) * c.n_head + h) * kLatent) + lane;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint2 pk;
    pk.x = pack_f16x2(acc[k].x * inv, acc[k].y * inv);
    pk.y = pack_f16x2(acc[k].z * inv, acc[k].w * inv);
    out[32 * k] = pk;
  }
}
}  // namespace

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c.B), static_cast<unsigned>((c.n_head + kCombHeads - 1) / kCombHeads));
  cfg.blockDim = dim3(32 * kCombHeads);
  cfg.dynamicSmemBytes = static_cast<size_t>(c.n_clusters + 1) * sizeof(long long);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, c);
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
__global__ void __launch_bounds__(256) cache_bf16_to_f16_kernel(const uint4* kv, uint4* out, int64_t n_units,
                                                                 int* err) {
  uint32_t run = 0;                  // |x| bit patterns seen (fp16 range check)
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(kv + u);
    run = bf16x2_absmax(bf16x2_absmax(run, v.x), v.y);
    run = bf16x2_absmax(bf16x2_absmax(run, v.z), v.w);
    uint4 o;
    float2 f;
    f = bf16x2_to_f32(v.x); o.x = pack_f16x2(f.x, f.y);
    f = bf16x2_to_f32(v.y); o.y = pack_f16x2(f.x, f.y);
    f = bf16x2_to_f32(v.z); o.z = pack_f16x2(f.x, f.y);
    f = bf16x2_to_f32(v.w); o.w = pack_f16x2(f.x, f.y);
    out[u] = o;
  }
  if (bf16x2_absmax_overflows(run)) record_error(err, MLA_ERR_RANGE);
}

// One thread per 16 codes (half a q8_0 block): 36 per row.
__global__ void __launch_bounds__(256) cache_q8_0_to_f16_kernel(const int8_t* kv_q, const __half* kv_d, int64_t ld_d,
                                                                 uint4* out, int64_t rows, int* err) {
  const int64_t n_units = rows * (kRow / 16);
  uint32_t dmax = 0;                 // largest |scale| bit pattern seen (fp16 range check)
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = u / (kRow / 16);
    const int c = static_cast<int>(u % (kRow / 16));
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(kv_q + row * kRow) + c);
    const uint32_t ds = __half_as_ushort(__ldg(kv_d + static_cast<int64_t>(c >> 1) * ld_d + row));
    dmax = max(dmax, ds & 0x7FFFu);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) i8x4_to_f16x4(w[k], ds | (ds << 16), h[2 * k], h[2 * k + 1]);
    out[2 * u] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * u + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
  if (f16_scale_overflows(dmax)) record_error(err, MLA_ERR_RANGE);
}

unsigned stage_blocks(int64_t n_units) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  return static_cast<unsigned>(max(static_cast<int64_t>(1), min(cap, (n_units + 255) / 256)));
}
}  // namespace

cudaError_t launch_bf16_to_f16(const void* src, void* dst, int64_t n, int* err, cudaStream_t stream) {
  const int64_t n_units = n / 8;
  cache_bf16_to_f16_kernel<<<stage_blocks(n_units), 256, 0, stream>>>(static_cast<const uint4*>(src),
                                                                       static_cast<uint4*>(dst), n_units, err);
  return cudaGetLastError();
}

cudaError_t launch_stage_cache_f16(const void* kv, const int8_t* kv_q, const uint16_t* kv_d, int64_t ld_d,
                                   int64_t rows, void* out, int* err, cudaStream_t stream) {
  if (kv != nullptr) {
    const int64_t n_units = rows * (kRow / 8);
    cache_bf16_to_f16_kernel<<<stage_blocks(n_units), 256, 0, stream>>>(static_cast<const uint4*>(kv),
                                                                         static_cast<uint4*>(out), n_units, err);
  } else {
    const int64_t n_units = rows * (kRow / 16);
    cache_q8_0_to_f16_kernel<<<stage_blocks(n_units), 256, 0, stream>>>(
        kv_q, reinterpret_cast<const __half*>(kv_d), ld_d, static_cast<uint4*>(out), rows, err);
  }
  return cudaGetLastError();
}


}  // namespace mla
