// The step before the attention path: new tokens' rows into the latent cache.
#pragma once
#include "common.cuh"

namespace mla {

struct RopeAppendArgs {
  const uint16_t* c_kv;   // bf16 [n][512]
  const uint16_t* k_pe;   // bf16 [n][64], not yet rotated
  const int32_t* pos;     // [n]
  const int64_t* slot;    // [n] cache rows
  int64_t n;
  uint16_t* kv;           // bf16 [n_rows][576] or null
  int8_t* kv_q;           // int8 [n_rows][576] or null
  uint16_t* kv_d;         // fp16 [18][ld_d] (with kv_q)
  int64_t ld_d;
  int64_t n_rows;
  int* err;
  // Pair i turns by pos * freq_scale * freq_base^(-2i/64) radians, i.e.
  // pos * t_i full turns; turn[i] = frac(t_i) as a 0.64 fixed-point number,
  // so that frac(pos * t_i) is the low 64 bits of the integer product.
  uint64_t turn[32];
};

cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream);

}  // namespace mla
