// The step before the attention path: the rows of new tokens into the latent
// cache, bf16 and/or q8_0 (pages: "MLA matrix absorption in ik_llama.cpp"
// sec. 3 -- the RoPE part of a key is rotated by position, the latent part is
// not; "llama.cpp KV Cache 与注意力机制" sec. 2.2-2.3 -- slots and
// ggml_rope_ext over n_rot = 64 dims).  HBM-bound: 1164 bytes in and up to
// 1764 bytes out per token.
#include "append.cuh"
#include "kernels.cuh"

namespace mla {
namespace {

// Rotate this lane's 8 RoPE values (pairs 4 lane .. 4 lane + 3; dims (2i, 2i+1)
// form pair i) by pos * t_i turns.  The fraction of a turn is exact integer
// arithmetic (the low 64 bits of pos * turn[i]); its top 32 bits give the
// angle as a float in [0, 2) half-turns for sincospif (error < 2^-23 rad);
// the rotation is in fp32, rounded once to bf16.
MLA_DEVINL uint4 rope8(uint4 v, int32_t pos, const uint64_t* turn, int lane) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint64_t f = static_cast<uint64_t>(static_cast<uint32_t>(pos)) * turn[4 * lane + q];
    const float half_turns = static_cast<float>(static_cast<uint32_t>(f >> 32)) * 0x1p-31f;
    float sn, cs;
    sincospif(half_turns, &sn, &cs);
    const float2 x = bf16x2_to_f32(w[q]);
    w[q] = pack_bf16x2(x.x * cs - x.y * sn, x.x * sn + x.y * cs);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// This lane's 8 values v (16 bytes) at column col of cache row s: stored as
// bf16 and, four lanes making one q8_0 block, quantised by the rules of
// mla_quantize_q8_0.  Every lane of the warp calls it (the block maximum is
// shuffled); `active` lanes store.
MLA_DEVINL void store_pass(const RopeAppendArgs& a, uint4 v, bool active, int64_t s, int col, int lane) {
  if (active && a.kv != nullptr) *reinterpret_cast<uint4*>(a.kv + s * kRow + col) = v;
  if (a.kv_q == nullptr) return;
  float x[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = bf16x2_to_f32(w[q]);
    x[2 * q] = f.x;
    x[2 * q + 1] = f.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float d = amax / 127.0f;
  uint32_t c[2] = {0u, 0u};
  if (amax > 0.f) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int q = max(-127, min(127, static_cast<int>(roundf(x[e] / d))));
      c[e >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (e & 3));
    }
  }
  if (active) {
    *reinterpret_cast<uint2*>(a.kv_q + s * kRow + col) = make_uint2(c[0], c[1]);
    if ((lane & 3) == 0) a.kv_d[static_cast<int64_t>(col / kQ8Block) * a.ld_d + s] = __half_as_ushort(__float2half_rn(d));
  }
}

// One warp per group of four new tokens: the latent values token by token
// (two passes of 256 values, a lane holding 8), then the four tokens' RoPE
// values in one pass (8 lanes per token), so that no pass leaves lanes idle.
__global__ void __launch_bounds__(256) rope_append_kernel(RopeAppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t j0 = 4 * (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)); j0 < a.n;
       j0 += 4 * warps) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      const int64_t j = j0 + k;
      if (j >= a.n) break;
      const int64_t s = a.slot[j];
      const int32_t p = a.pos[j];
      if (s < 0 || s >= a.n_rows || p < 0) {
        if (lane == 0) record_error(a.err, MLA_ERR_INVALID_ARG);
        continue;
      }
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int col = 256 * h + 8 * lane;
        store_pass(a, __ldg(reinterpret_cast<const uint4*>(a.c_kv + j * kLatent + col)), true, s, col, lane);
      }
    }
    const int l8 = lane & 7;
    const int64_t j = j0 + (lane >> 3);
    bool ok = j < a.n;
    int64_t s = 0;
    int32_t p = 0;
    if (ok) {
      s = a.slot[j];
      p = a.pos[j];
      ok = s >= 0 && s < a.n_rows && p >= 0;
    }
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok) v = rope8(__ldg(reinterpret_cast<const uint4*>(a.k_pe + j * kRope + 8 * l8)), p, a.turn, l8);
    store_pass(a, v, ok, s, kLatent + 8 * l8, lane);
  }
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const unsigned blocks = static_cast<unsigned>(max(static_cast<int64_t>(1), min(cap, (a.n + 31) / 32)));
  rope_append_kernel<<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
