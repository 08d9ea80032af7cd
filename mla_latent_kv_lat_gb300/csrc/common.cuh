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

// Time after which a bounded wait gives up, in microseconds of %globaltimer.
// Every wait inside a kernel normally completes within microseconds.
constexpr uint32_t kDefaultWaitUs = 500000;
// Longest time one try_wait may keep a waiting thread suspended.  The thread
// wakes as soon as the phase completes, so this only sets how often a stuck
// wait re-checks its time limit.
constexpr uint32_t kWaitSuspendNs = 20000;

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

// Four int8 codes (one 32-bit word) times the fp16 scale d2 (both halves):
// fp16(code x d) for each, as two fp16 pairs.  A biased byte c + 128 placed
// under the fp16 exponent of 1024 reads as 1024 + c + 128, so subtracting
// 1152 gives the code exactly; the product is then rounded once, the same
// result as rounding the exact product code x d to fp16.
MLA_DEVINL void i8x4_to_f16x4(uint32_t w, uint32_t d2, uint32_t& lo, uint32_t& hi) {
  const uint32_t b = w ^ 0x80808080u;
  const uint32_t h0 = __byte_perm(b, 0x64646464u, 0x4140), h1 = __byte_perm(b, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
  const __half2 d = *reinterpret_cast<const __half2*>(&d2);
  const __half2 r0 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&h0), bias), d);
  const __half2 r1 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&h1), bias), d);
  lo = *reinterpret_cast<const uint32_t*>(&r0);
  hi = *reinterpret_cast<const uint32_t*>(&r1);
}

// fp16 range checks.  A thread keeps a running maximum and records
// MLA_ERR_RANGE once, at the end of its work, if the maximum says a value fp16
// cannot hold went by.
//   bf16 words: the maximum of |x| bit patterns in each 16-bit half.  bf16 has
//   no value between 65504 (fp16's largest) and 65536 = 0x4780, so a half at or
//   above 0x4780 is too large for fp16, or an infinity or a NaN (0x7F80 and up).
MLA_DEVINL uint32_t bf16x2_absmax(uint32_t run, uint32_t w) { return __vmaxu2(run, w & 0x7FFF7FFFu); }
MLA_DEVINL bool bf16x2_absmax_overflows(uint32_t run) {
  return (run & 0xFFFFu) >= 0x4780u || (run >> 16) >= 0x4780u;
}
//   q8_0 block scales (fp16 bits): |d| >= 516 lets 127 x d pass 65504 (the
//   largest code of a block from the quantiser is +-127); 0x6008 = 516.
MLA_DEVINL bool f16_scale_overflows(uint32_t run_abs_bits) { return run_abs_bits >= 0x6008u; }
//   fp32 values about to be rounded to fp16: fp16(x) is infinite for
//   |x| >= 65520.  The running maximum keeps a NaN (max.NaN), and the negated
//   comparison flags it.
MLA_DEVINL float f32_absmax(float run, float x) {
  float r;
  asm("{\n\t.reg .f32 t;\n\tabs.f32 t, %2;\n\tmax.NaN.f32 %0, %1, t;\n\t}" : "=f"(r) : "f"(run), "f"(x));
  return r;
}
MLA_DEVINL bool f32_overflows_f16(float run_absmax) { return !(run_absmax < 65520.f); }

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

MLA_DEVINL long long warp_sum_i64(long long v) {
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

// Non-blocking check of phase `parity` (acquire at CTA scope when it returns
// true).  The result arrives like a load's, so a check issued early overlaps
// its latency with other work until the branch that consumes it.
MLA_DEVINL bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware suspend the thread for up to `ns`
// nanoseconds (or until the phase completes) instead of returning at once.
// A waiting warp then takes no issue slots from the warps doing the work.
MLA_DEVINL bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

MLA_DEVINL uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// The slow path shared by the bounded waits: keep trying (suspended between
// tries) until `done()` holds, `limit_us` microseconds have passed (records
// MLA_ERR_TIMEOUT) or another thread has already recorded a timeout, in which
// case the launch is failing anyway and this wait gives up at once, so that a
// failed launch ends quickly instead of each CTA timing out in turn.  While
// the error word holds a timeout (until the host reads it), a wait that does
// not complete at once gives up.  Other recorded errors (a value out of fp16
// range, a skipped request) leave the waits alone.
MLA_DEVINL bool timeout_recorded(const int* err) {
  return err != nullptr && *reinterpret_cast<const volatile int*>(err) == MLA_ERR_TIMEOUT;
}
template <typename Done>
MLA_DEVINL bool wait_slow(Done done, uint32_t limit_us, int* err) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (done()) return true;
    if (timeout_recorded(err)) return false;
    if (global_timer_ns() - t0 > static_cast<uint64_t>(limit_us) * 1000u) {
      record_error(err, MLA_ERR_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait for phase `parity` of `bar` to complete.  Returns false if it
// did not complete within `limit_us` microseconds (MLA_ERR_TIMEOUT recorded)
// or an error was already recorded.
MLA_DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit_us, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow([&] { return mbar_try_wait_suspend(bar, parity, kWaitSuspendNs); }, limit_us, err);
}

}  // namespace mla
