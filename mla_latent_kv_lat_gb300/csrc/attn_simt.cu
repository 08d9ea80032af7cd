// Latent-space attention on CUDA cores: split scores (RoPE part + latent part),
// causal online softmax and the weighted sum over the latent cache, for one
// query token and a group of 16 heads per CTA.  ("MLA matrix absorption in
// ik_llama.cpp", sec. 4 and 5.)  This is the plain CUDA-core path; it serves
// prefill and the split-KV decode partials for any supported head count.
#include "kernels.cuh"

namespace mla {

namespace {

constexpr int kG = 16;          // heads (query rows) per CTA
constexpr int kBK = 32;         // keys per tile
constexpr int kKS = kRow + 1;   // padded fp32 row stride of the key tile
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct SimtSmem {
  float q[kG * kRow];        // scaled queries: [q_lat | q_pe] * scale * log2(e)
  float k[kBK * kKS];        // key tile, dequantised to fp32
  float p[kG * kBK];         // probabilities of the tile
  float alpha[kG];           // per-row rescale of the running sum
  float m[kG];
  float l[kG];
};

// Load `rows` cache rows starting at `row0` into the fp32 key tile; rows at or
// past `row_end` are zero-filled (their scores are masked anyway).
template <bool kQ8>
MLA_DEVINL void load_key_tile(float* ks, const AttnArgs& a, int64_t row0, int64_t row_end) {
  if constexpr (!kQ8) {
    const uint16_t* kv = static_cast<const uint16_t*>(a.kv);
    for (int idx = threadIdx.x; idx < kBK * (kRow / 8); idx += kThreads) {
      const int key = idx / (kRow / 8), ch = idx % (kRow / 8);
      const int64_t row = row0 + key;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < row_end) v = *reinterpret_cast<const uint4*>(kv + row * kRow + ch * 8);
      float* dst = ks + key * kKS + ch * 8;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = bf16x2_to_f32(w[e]);
        dst[2 * e] = f.x;
        dst[2 * e + 1] = f.y;
      }
    }
  } else {
    const int8_t* kq = a.kv_q;
    const __half* kd = reinterpret_cast<const __half*>(a.kv_d);
    for (int idx = threadIdx.x; idx < kBK * (kRow / 16); idx += kThreads) {
      const int key = idx / (kRow / 16), ch = idx % (kRow / 16);
      const int64_t row = row0 + key;
      float* dst = ks + key * kKS + ch * 16;
      if (row < row_end) {
        const int4 v = *reinterpret_cast<const int4*>(kq + row * kRow + ch * 16);
        const float d = __half2float(kd[static_cast<int64_t>(ch / 2) * a.ld_d + row]);
        const int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int8_t q = static_cast<int8_t>((w[e / 4] >> (8 * (e % 4))) & 0xFF);
          dst[e] = d * static_cast<float>(q);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[e] = 0.f;
      }
    }
  }
}

template <bool kQ8>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.n_head;
  const int h0 = blockIdx.y * kG;

  // Work item: which query row block, which key range.
  int64_t q_row;          // index of the query token (prefill t, decode b)
  int64_t kbeg, kend;     // cache rows [kbeg, kend)
  int64_t part = -1;      // decode: partial slot index
  if (a.decode) {
    const int b = blockIdx.x / a.n_split, s = blockIdx.x % a.n_split;
    const int64_t len = a.seq_len[b];
    const int64_t lo = static_cast<int64_t>(s) * a.chunk;
    if (lo >= len) return;                      // this split is past the sequence
    kbeg = a.seq_start[b] + lo;
    kend = a.seq_start[b] + min(len, lo + a.chunk);
    q_row = b;
    part = static_cast<int64_t>(b) * a.n_split + s;
  } else {
    q_row = blockIdx.x;
    kbeg = 0;
    kend = static_cast<int64_t>(a.q_pos0) + q_row + 1;
  }

  // Queries, pre-scaled so that scores come out in log2 units.
  const float qs = a.scale * kLog2e;
  const uint16_t* ql = static_cast<const uint16_t*>(a.q_lat);
  const uint16_t* qp = static_cast<const uint16_t*>(a.q_pe);
  for (int idx = tid; idx < kG * kRow; idx += kThreads) {
    const int r = idx / kRow, c = idx % kRow;
    const int64_t qi = q_row * H + h0 + r;
    const float v = c < kLatent ? f16_to_f32(ql[qi * kLatent + c]) : bf16_to_f32(qp[qi * kRope + (c - kLatent)]);
    sm.q[idx] = v * qs;
  }

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  const int pr = tid >> 4, pc = tid & 15;     // PV mapping: row, column phase

  for (int64_t k0 = kbeg; k0 < kend; k0 += kBK) {
    __syncthreads();
    load_key_tile<kQ8>(sm.k, a, k0, kend);
    __syncthreads();
    // Scores: warp w owns rows 2w, 2w+1; lane = key.
    const int r0 = 2 * warp;
    const float* kr = sm.k + lane * kKS;
    const float* q0 = sm.q + r0 * kRow;
    const float* q1 = q0 + kRow;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int c = 0; c < kRow; ++c) {
      const float kv = kr[c];
      s0 = fmaf(q0[c], kv, s0);
      s1 = fmaf(q1[c], kv, s1);
    }
    const bool valid = (k0 + lane) < kend;
    s0 = valid ? s0 : -INFINITY;
    s1 = valid ? s1 : -INFINITY;
    const float mn0 = fmaxf(m_run[0], warp_max(s0));
    const float mn1 = fmaxf(m_run[1], warp_max(s1));
    const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
    const float a0 = exp2f(m_run[0] - mn0), a1 = exp2f(m_run[1] - mn1);
    l_run[0] = l_run[0] * a0 + warp_sum(p0);
    l_run[1] = l_run[1] * a1 + warp_sum(p1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    sm.p[r0 * kBK + lane] = p0;
    sm.p[(r0 + 1) * kBK + lane] = p1;
    if (lane == 0) {
      sm.alpha[r0] = a0;
      sm.alpha[r0 + 1] = a1;
    }
    __syncthreads();
    // Weighted sum in latent space: 16 threads per row, strided columns.
    const float al = sm.alpha[pr];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] *= al;
    const int nk = static_cast<int>(min(static_cast<int64_t>(kBK), kend - k0));
    for (int key = 0; key < nk; ++key) {
      const float p = sm.p[pr * kBK + key];
      const float* vr = sm.k + key * kKS + pc;
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = fmaf(p, vr[16 * i], acc[i]);
    }
  }
  if (lane == 0) {
    sm.m[2 * warp] = m_run[0];
    sm.m[2 * warp + 1] = m_run[1];
    sm.l[2 * warp] = l_run[0];
    sm.l[2 * warp + 1] = l_run[1];
  }
  __syncthreads();
  const int64_t orow = q_row * H + h0 + pr;
  if (!a.decode) {
    const float inv = 1.f / sm.l[pr];
    uint16_t* o = static_cast<uint16_t*>(a.o_lat) + orow * kLatent;
#pragma unroll
    for (int i = 0; i < 32; ++i) o[pc + 16 * i] = f32_to_f16(acc[i] * inv);
    if (a.lse != nullptr && pc == 0) a.lse[orow] = (sm.m[pr] + log2f(sm.l[pr])) * kLn2;
  } else {
    const int64_t slot = part * H + h0 + pr;
    float* o = a.ws_o + slot * kLatent;
#pragma unroll
    for (int i = 0; i < 32; ++i) o[pc + 16 * i] = acc[i];
    if (pc == 0) {
      a.ws_ml[2 * slot] = sm.m[pr];
      a.ws_ml[2 * slot + 1] = sm.l[pr];
    }
  }
}

}  // namespace

size_t attn_simt_smem_bytes() { return sizeof(SimtSmem); }

cudaError_t launch_attn_simt(const AttnArgs& a, bool q8, int n_blocks_x, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem);
  dim3 grid(n_blocks_x, a.n_head / kG);
  if (q8) {
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attn_simt_kernel<true><<<grid, kThreads, smem, stream>>>(a);
  } else {
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attn_simt_kernel<false><<<grid, kThreads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Split-KV combine: merge the per-split (m, l, o) of each (sequence, head) by
// log-sum-exp and write o_lat in fp16.
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
    const float w = exp2f(c.ws_ml[2 * slot] - M);
    L += w * c.ws_ml[2 * slot + 1];
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
