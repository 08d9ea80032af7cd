// Shared device helpers of libmla: status codes, the per-device error word,
// bounded mbarrier waits, bf16/fp16 conversion.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mla.h"

#define MLA_DEVINL __device__ __forceinline__

namespace mla {

constexpr int kLatent = 512;   // kv_lora_rank
constexpr int kRope = 64;      // qk_rope
constexpr int kRow = 576;      // latent + rope: one cache row
constexpr int kNope = 128;     // qk_nope
constexpr int kVHead = 128;    // v_head
constexpr int kQ8Block = 32;   // q8_0 block size
constexpr int kQ8Blocks = kRow / kQ8Block;   // 18 blocks per row

// Default number of polls before a bounded wait gives up.  A poll is one
// mbarrier.try_wait, which itself suspends for a hardware-defined time, so
// this bounds a stuck wait to well under a second on GB300.
constexpr uint32_t kDefaultWaitPolls = 1u << 22;

// Record the first device-side error; later errors keep the first one.
MLA_DEVINL void record_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

MLA_DEVINL float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two bf16 packed in one 32-bit word -> two floats.
MLA_DEVINL float2 bf16x2_to_f32(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

MLA_DEVINL float f16_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

MLA_DEVINL uint16_t f32_to_f16(float f) { return __half_as_ushort(__float2half_rn(f)); }

MLA_DEVINL uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

MLA_DEVINL float2 f16x2_to_f32(uint32_t w) {
  return __half22float2(*reinterpret_cast<__half2*>(&w));
}

MLA_DEVINL uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

MLA_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

MLA_DEVINL float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

MLA_DEVINL float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier primitives (PTX ISA, "mbarrier" instructions), shared::cta scope.
// ---------------------------------------------------------------------------
MLA_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MLA_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

MLA_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

MLA_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

MLA_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar` to complete.  Returns false (and
// records MLA_ERR_TIMEOUT) if it did not complete within `polls` polls.
MLA_DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t polls, int* err) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  record_error(err, MLA_ERR_TIMEOUT);
  return false;
}

}  // namespace mla
