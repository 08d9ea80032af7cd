// The step after the path: the attention output projection
//   u[t][n] = sum_h sum_e o[t][h][e] * w_o[h][e][n]
// ("MLA matrix absorption in ik_llama.cpp", sec. 4: after late decompression
// the heads' 128-wide outputs are flattened to n_head * 128 and multiplied by
// wo, the einsum hdD,bhqd->bqD).  One dense GEMM, C[M][N] = A[M][K] B[K][N]
// with M = tokens, K = n_head * 128, N = the hidden size.
//
// Persistent CTAs, one per SM, walk 128 x 256 output tiles in groups of 16 row
// tiles (within a group M fastest): the ~152 tiles in flight then read about
// 16 row tiles of A and 10 column tiles of B, ~140 MB, which L2 holds.  Per tile, K moves
// in 64-wide steps through a 4-stage TMA ring (A: 128 x 64, K-major; B: 64 x
// 256, N-major, four 64-column boxes), 128-byte swizzled, on tcgen05 MMAs
// (M = 128, N = 256, K = 16, fp16 x fp16 -> fp32) into one of two TMEM
// accumulators, so the epilogue of one tile overlaps the MMAs of the next.
// Warp 0 issues the copies, warp 1 the MMAs, warps 2-5 drain the accumulators
// (one TMEM lane quadrant each) through a shared-memory slice, so that each
// store instruction writes four rows x 128 contiguous bytes of u.
#include "kernels.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;            // 16 KB
constexpr int kBBox = kBK * 64 * 2;               // 8 KB: 64 K-rows x 64 columns
constexpr int kBBytes = (kBN / 64) * kBBox;       // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStgBytes = 4 * 32 * 128;           // epilogue: 4 warps x 32 rows x 128 B
constexpr int kBarBytes = 256;
constexpr int kSmem = 1024 + kStages * kStageBytes + kStgBytes + kBarBytes;
constexpr int kThreads = 192;
static_assert(kSmem <= 232448, "shared memory");

struct WoArgs {
  float* u;
  int M, N, K;
  int m_tiles, n_tiles;
  int* err;
  uint32_t wait_us;
};

constexpr int kGroupM = 16;

// Output tile t -> (row, column) of its first element.
MLA_DEVINL void wo_tile(const WoArgs& g, int t, int& m0, int& n0) {
  const int per_group = kGroupM * g.n_tiles;
  const int grp = t / per_group, w = t % per_group;
  const int rows = min(kGroupM, g.m_tiles - grp * kGroupM);
  m0 = (grp * kGroupM + w % rows) * kBM;
  n0 = (w / rows) * kBN;
}

__global__ void __launch_bounds__(kThreads, 1)
    wo_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, WoArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sStage = sm;
  uint8_t* sStg = sm + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + kStgBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = g.m_tiles * g.n_tiles;
  const int kc_n = g.K / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
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
      tc::prefetch_tmap(&tmB);
      int u = 0;                                   // k-steps issued, across tiles
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        int m0, n0;
        wo_tile(g, t, m0, n0);
        for (int kc = 0; kc < kc_n; ++kc, ++u) {
          const int st = u % kStages;
          if (u >= kStages && !mbar_wait_bounded(&empty[st], ((u / kStages) - 1) & 1, g.wait_us, g.err)) {
            ok = false;
            break;
          }
          uint8_t* s = sStage + st * kStageBytes;
          mbar_arrive_expect_tx(&full[st], kStageBytes);
          tc::tma_load_3d(s, &tmA, &full[st], kc * kBK, m0, 0);
#pragma unroll
          for (int j = 0; j < kBN / 64; ++j) tc::tma_load_3d(s + kABytes + j * kBBox, &tmB, &full[st], n0 + 64 * j, kc * kBK, 0);
        }
      }
    }
  } else if (warp == 1) {
    // whole warp, converged; one elected lane issues (see mma_ss_warp)
    constexpr uint32_t idesc = tc::idesc_f16(kBM, kBN, false, false, true);   // fp16 x fp16
    bool ok = true;
    int u = 0, i = 0;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      if (i >= 2) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[buf], ((i >> 1) - 1) & 1, g.wait_us, g.err));
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t d = tmem + buf * kBN;
      for (int kc = 0; kc < kc_n; ++kc, ++u) {
        const int st = u % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (u / kStages) & 1, g.wait_us, g.err));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t a0 = smem_u32(sStage + st * kStageBytes);
        const uint32_t b0 = a0 + kABytes;
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)
          tc::mma_ss_warp(d, tc::sdesc_sw128(a0 + ks * 32, 16, 1024), tc::sdesc_sw128(b0 + ks * 2048, kBBox, 1024),
                          idesc, (kc | ks) != 0);
        tc::mma_commit_warp(&empty[st]);
      }
      if (ok) tc::mma_commit_warp(&acc_full[buf]);
    }
  } else {
    // epilogue: warp w serves TMEM lanes 32 (w % 4) .. +31 = tile rows
    const int q = warp & 3;
    uint8_t* stg = sStg + (warp - 2) * 4096;
    bool ok = true;
    int i = 0;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      int m0, n0;
      wo_tile(g, t, m0, n0);
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], (i >> 1) & 1, g.wait_us, g.err));
      if (!ok) break;
      tc::fence_after_sync();
      const int row0 = m0 + q * 32;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + c * 32, r);
        tc::tmem_ld_wait();
        const int col = n0 + c * 32;
        if (col >= g.N) continue;                  // past the last column (N is a multiple of 64)
        // row `lane`'s 32 values -> the warp's slice (16-byte units swizzled by row)
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((v ^ (lane & 7)) << 4)) =
              make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
        __syncwarp();
        // four rows x 128 contiguous bytes per store instruction
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int rr = (lane >> 3) + 4 * m, part = lane & 7;
          const uint4 x = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((part ^ (rr & 7)) << 4));
          if (row0 + rr < g.M)
            *reinterpret_cast<uint4*>(g.u + static_cast<int64_t>(row0 + rr) * g.N + col + part * 4) = x;
        }
        __syncwarp();
      }
      tc::fence_before_sync();
      mbar_arrive(&acc_empty[buf]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_wo_gemm_tc(const void* a, const void* w_o, float* u, int M, int K, int N, int* err,
                              uint32_t wait_us, cudaStream_t stream) {
  CUtensorMap tmA, tmB;
  // A = o [M][K] fp16 (K-major): 64 x 128 boxes; B = w_o [K][N] fp16 (N-major): 64 x 64 boxes.
  cudaError_t e = make_tmap_3d(&tmA, a, false, static_cast<uint64_t>(K), static_cast<uint64_t>(M), 1,
                               static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(K) * M * 2, kBK, kBM, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tmB, w_o, false, static_cast<uint64_t>(N), static_cast<uint64_t>(K), 1,
                   static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(N) * K * 2, 64, kBK, 1);
  if (e != cudaSuccess) return e;
  WoArgs g;
  g.u = u;
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + kBM - 1) / kBM;
  g.n_tiles = (N + kBN - 1) / kBN;
  g.err = err;
  g.wait_us = wait_us;
  const int tiles = g.m_tiles * g.n_tiles;
  const int grid = min(tiles, device_sm_count());
  e = cudaFuncSetAttribute(wo_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  wo_gemm_tc_kernel<<<grid, kThreads, kSmem, stream>>>(tmA, tmB, g);
  return cudaGetLastError();
}

}  // namespace mla
