// Per-head projections on the 5th-generation tensor cores (tcgen05):
//   absorb            q_lat[t][h][:] = q_nope[t][h][:] . wk_b[h]   (K=128, N=512)
//   late decompress   o[t][h][:]     = o_lat[t][h][:]  . wv_b[h]   (K=512, N=128)
// ("MLA matrix absorption in ik_llama.cpp", sec. 3 and sec. 4.)
//
// One persistent CTA per (head, token group): the head's weight matrix stays
// in shared memory (MN-major, 128-byte swizzle), 128-token A tiles stream in
// through a 4-stage TMA ring (K-major, 128-byte swizzle), fp32 accumulators
// live in TMEM slots that four epilogue warps drain while the next tile's
// MMAs run.  Warp 0 issues TMA, warp 1 issues MMAs, warps 2-5 run the
// epilogue (and, for the late decompression, convert wv_b from bf16 to fp16
// so that both MMA operands are fp16).
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kStages = 4;
constexpr int kChunkBytes = 128 * 128;      // A K-chunk: 128 rows x 64 elements x 2 B
constexpr int kThreads = 192;

template <int K, int N, int NSUB>
struct GemmCfg {
  static constexpr int KC = K / 64;                 // A K-chunks per tile
  static constexpr int NS = N / NSUB;               // output sub-tiles per tile
  static constexpr int SLOTS = 512 / NSUB;          // accumulator slots in TMEM
  static constexpr int W_CHUNK = K * 128;           // one 64-column chunk of W: K rows x 128 B
  static constexpr int W_BYTES = (N / 64) * W_CHUNK;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + W_BYTES + kStages * kChunkBytes + BAR_BYTES;
};

struct TcGemmArgs {
  void* c;
  const uint16_t* w;     // bf16 [H][K][N], read directly when converting to fp16
  int T, H, tiles;
  int* err;
  uint32_t wait_us;
};

template <int K, int N, int NSUB, bool kAbsorb, bool kOutF16>
__global__ void __launch_bounds__(kThreads, 1)
    head_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                        TcGemmArgs g) {
  using C = GemmCfg<K, N, NSUB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sA = smem + C::W_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + kStages * kChunkBytes);
  uint64_t* a_full = bars;
  uint64_t* a_empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + C::SLOTS;
  uint64_t* w_full = acc_empty + C::SLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(w_full + 1);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, grp = blockIdx.y, G = gridDim.y;
  const int n_tiles = (g.tiles - grp + G - 1) / G;     // tiles grp, grp + G, ...

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int s = 0; s < C::SLOTS; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 128);
    }
    mbar_init(w_full, kAbsorb ? 1 : 128);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tmA);
      if constexpr (kAbsorb) {
        tc::prefetch_tmap(&tmW);
        mbar_arrive_expect_tx(w_full, C::W_BYTES);
        for (int c = 0; c < N / 64; ++c) tc::tma_load_3d(sW + c * C::W_CHUNK, &tmW, w_full, c * 64, 0, h);
      }
      for (int i = 0; i < n_tiles && !abort_flag; ++i) {
        const int tt = grp + i * G;
        for (int kc = 0; kc < C::KC; ++kc) {
          const int u = i * C::KC + kc, st = u % kStages;
          if (u >= kStages && !mbar_wait_bounded(&a_empty[st], ((u / kStages) - 1) & 1, g.wait_us, g.err)) {
            abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&a_full[st], kChunkBytes);
          tc::tma_load_3d(sA + st * kChunkBytes, &tmA, &a_full[st], kc * 64, h, tt * 128);
        }
      }
    }
  } else if (warp == 1) {
    {   // whole warp, converged; one lane issues (see mma_ss_warp)
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(w_full, 0, g.wait_us, g.err));
      tc::fence_after_sync();
      constexpr uint32_t idesc = tc::idesc_f16(128, NSUB, kAbsorb, false, true);
      for (int i = 0; ok && i < n_tiles; ++i) {
        for (int j = 0; ok && j < C::NS; ++j) {
          const int job = i * C::NS + j, slot = job % C::SLOTS;
          if (job >= C::SLOTS)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[slot], ((job / C::SLOTS) - 1) & 1, g.wait_us, g.err));
          tc::fence_after_sync();
          for (int kc = 0; ok && kc < C::KC; ++kc) {
            const int u = i * C::KC + kc, st = u % kStages;
            if (j == 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&a_full[st], (u / kStages) & 1, g.wait_us, g.err));
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t a0 = smem_u32(sA + st * kChunkBytes);
            const uint32_t b0 = smem_u32(sW + (j * NSUB / 64) * C::W_CHUNK);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const int k = kc * 64 + ks * 16;
              const uint64_t ad = tc::sdesc_sw128(a0 + ks * 32, 16, 1024);
              const uint64_t bd = tc::sdesc_sw128(b0 + (k / 16) * 2048, C::W_CHUNK, 1024);
              tc::mma_ss_warp(tmem + slot * NSUB, ad, bd, idesc, (kc | ks) != 0);
            }
            if (j == C::NS - 1) tc::mma_commit_warp(&a_empty[st]);
          }
          tc::mma_commit_warp(&acc_full[slot]);
        }
      }
      if (!ok) abort_flag = 1;
    }
  } else {
    const int q = warp & 3;                      // TMEM lane quadrant this warp may access
    const int et = threadIdx.x - 64;             // 0..127
    if constexpr (!kAbsorb) {
      // wv_b[h] (bf16 [K][N]) -> fp16, MN-major 128-byte-swizzled chunks of 64 columns.
      const uint16_t* w = g.w + static_cast<int64_t>(h) * K * N;
      for (int idx = et; idx < K * (N / 8); idx += 128) {
        const int k = idx / (N / 8), un = idx % (N / 8);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(w + static_cast<int64_t>(k) * N + un * 8));
        uint4 o;
        float2 f;
        f = bf16x2_to_f32(v.x); o.x = pack_f16x2(f.x, f.y);
        f = bf16x2_to_f32(v.y); o.y = pack_f16x2(f.x, f.y);
        f = bf16x2_to_f32(v.z); o.z = pack_f16x2(f.x, f.y);
        f = bf16x2_to_f32(v.w); o.w = pack_f16x2(f.x, f.y);
        const int c = un / 8, u = un % 8;
        *reinterpret_cast<uint4*>(sW + c * C::W_CHUNK + k * 128 + ((u ^ (k & 7)) << 4)) = o;
      }
      tc::fence_proxy_async();
      mbar_arrive(w_full);
    }
    bool ok = true;
    float amax = 0.f;                            // |q_lat| or |o| before its fp16 rounding
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int tt = grp + i * G;
      const int row = tt * 128 + q * 32 + lane;
      for (int j = 0; ok && j < C::NS; ++j) {
        const int job = i * C::NS + j, slot = job % C::SLOTS;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[slot], (job / C::SLOTS) & 1, g.wait_us, g.err));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int c0 = 0; c0 < NSUB; c0 += 32) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + slot * NSUB + c0, r);
          tc::tmem_ld_wait();
          if (row < g.T) {
            const int64_t base = (static_cast<int64_t>(row) * g.H + h) * N + j * NSUB + c0;
            if constexpr (kAbsorb) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.c) + base);
#pragma unroll
              for (int e = 0; e < 32; ++e) amax = f32_absmax(amax, __uint_as_float(r[e]));
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_f16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                o.y = pack_f16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                o.z = pack_f16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                o.w = pack_f16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                dst[v] = o;
              }
            } else if constexpr (kOutF16) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.c) + base);
#pragma unroll
              for (int e = 0; e < 32; ++e) amax = f32_absmax(amax, __uint_as_float(r[e]));
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_f16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                o.y = pack_f16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                o.z = pack_f16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                o.w = pack_f16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                dst[v] = o;
              }
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(g.c) + base);
#pragma unroll
              for (int v = 0; v < 8; ++v) dst[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
            }
          }
        }
        tc::fence_before_sync();
        mbar_arrive(&acc_empty[slot]);
      }
    }
    if ((kAbsorb || kOutF16) && f32_overflows_f16(amax)) record_error(g.err, MLA_ERR_RANGE);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

cudaError_t get_tmap_encoder(void** fn) {
  if (g_encode == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || p == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = reinterpret_cast<void*>(g_encode);
  return cudaSuccess;
}

// 3-D tiled tensor map, 16-bit elements, 128-byte (or 64-byte) swizzle, zero fill outside.
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                         int swizzle_bytes) {
  void* fn = nullptr;
  cudaError_t e = get_tmap_encoder(&fn);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)(
      map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
      dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int K, int N, int NSUB, bool kAbsorb, bool kOutF16>
static cudaError_t launch_tc(const HeadGemmArgs& g, int* err, uint32_t wait_us, cudaStream_t stream) {
  using C = GemmCfg<K, N, NSUB>;
  CUtensorMap tmA, tmW;
  const uint64_t H = static_cast<uint64_t>(g.H);
  cudaError_t e = make_tmap_3d(&tmA, g.a, kAbsorb, K, H, static_cast<uint64_t>(g.T), K * 2, H * K * 2, 64, 1, 128);
  if (e != cudaSuccess) return e;
  if (kAbsorb) {
    e = make_tmap_3d(&tmW, g.w, true, N, K, H, N * 2, static_cast<uint64_t>(K) * N * 2, 64, K, 1);
    if (e != cudaSuccess) return e;
  } else {
    tmW = tmA;   // unused
  }
  TcGemmArgs a;
  a.c = g.c;
  a.w = static_cast<const uint16_t*>(g.w);
  a.T = g.T;
  a.H = g.H;
  a.tiles = (g.T + 127) / 128;
  a.err = err;
  a.wait_us = wait_us;
  const int sms = device_sm_count();
  int G = sms / g.H;
  if (G < 1) G = 1;
  if (G > a.tiles) G = a.tiles;
  auto kern = head_gemm_tc_kernel<K, N, NSUB, kAbsorb, kOutF16>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(g.H, G), kThreads, C::SMEM, stream>>>(tmA, tmW, a);
  return cudaGetLastError();
}

cudaError_t launch_head_gemm_tc(const HeadGemmArgs& g, int* err, uint32_t wait_us, cudaStream_t stream) {
  if (g.K == kNope && g.N == kLatent && !g.out_f32 && !g.a_f16 && !g.out_f16)
    return launch_tc<kNope, kLatent, 256, true, false>(g, err, wait_us, stream);
  if (g.K == kLatent && g.N == kVHead && g.out_f32 && g.a_f16 && !g.out_f16)
    return launch_tc<kLatent, kVHead, 128, false, false>(g, err, wait_us, stream);
  if (g.K == kLatent && g.N == kVHead && !g.out_f32 && g.a_f16 && g.out_f16)
    return launch_tc<kLatent, kVHead, 128, false, true>(g, err, wait_us, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mla
