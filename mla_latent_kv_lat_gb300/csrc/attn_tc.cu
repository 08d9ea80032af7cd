// Latent-space MLA attention on the 5th-generation tensor cores.
//
// What it computes ("MLA matrix absorption in ik_llama.cpp", sec. 4-5 and
// 8.1): for 128 query rows (query token x head pairs) and the latent cache,
//   s = scale * (q_lat . c_kv + q_pe . k_pe)     (split scores, no concat)
//   causal online softmax over the visible keys
//   o_lat = sum_j p_j c_kv[j]                    (weighted sum in latent space)
//
// How (one CTA pair = one 2-CTA cluster per 128 rows):
//   * The 512-wide fp32 output of 128 rows would fill all of a CTA's tensor
//     memory, leaving no room for scores, so the pair splits the latent
//     dimension: CTA r owns latent columns [256r, 256r+256) of the output and
//     of the score contraction; CTA 0 also owns the 64 RoPE dimensions.
//   * Each CTA computes its partial scores S_r = Q_r K_r^T on tcgen05 into
//     TMEM, scales and rounds them to fp16 and sends them to its peer with
//     st.async into distributed shared memory; both CTAs then hold the same
//     fp16 pair and form identical scores, maxima and probabilities, so their
//     output halves stay consistent without further exchange.
//   * P (fp16) goes to shared memory and O_r += P V_r runs on tcgen05 with V_r
//     read in place from the same cache tile (MN-major view).
//   * Cache tiles are loaded by four producer warps, converted to fp16 on the
//     way (bf16 cache: exact; q8_0 cache: fp16 scale x int8 code), and stored
//     in the 128-byte-swizzled layout the tensor core reads.
//   * Roles per CTA: warps 0-3 softmax / exchange / epilogue (thread = row),
//     warps 4-7 producer, warp 8 MMA issue.  Every wait is bounded.
#include "kernels.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kRows = 128;                   // query rows per cluster (MMA M)
constexpr int kBK = 64;                      // keys per tile
constexpr int kNChMax = 5;                   // 64-dim chunks per CTA (rank 0: 4 latent + rope)
constexpr int kKvChunk = kBK * 128;          // 8 KB: 64 keys x 64 fp16
constexpr int kKvStage = kNChMax * kKvChunk; // 40 KB
constexpr int kStages = 3;
constexpr int kQRopeBytes = kRows * 128;     // 16 KB: 128 rows x 64 fp16
constexpr int kPBytes = kRows * 128;         // 16 KB: 128 rows x 64 keys fp16
constexpr int kXBytes = kRows * kBK * 2;     // 16 KB: one exchange buffer
constexpr int kOffKv = kQRopeBytes;
constexpr int kOffP = kOffKv + kStages * kKvStage;
constexpr int kOffX = kOffP + kPBytes;
constexpr int kOffBar = kOffX + 2 * kXBytes;
constexpr int kSmem = 1024 + kOffBar + 256;
constexpr int kThreads = 288;
// TMEM columns: Q latent half (A operand, 256 fp16 = 128 cols), two fp32 score
// buffers of 64 columns, the fp32 output half (256 cols).
constexpr uint32_t kTmQ = 0, kTmS = 128, kTmO = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units: P stays <= 256, exact in fp16

struct Bars {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t x_full[2];
  uint64_t p_full;
  uint64_t pv_done;
  uint64_t q_ready;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

MLA_DEVINL bool wait_all(uint64_t* bar, uint32_t parity, const AttnTcArgs& a) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, a.polls, a.err));
}

// Store 8 halves (one 16-byte unit) to the swizzled K-major tile `base`
// (rows of 128 B): row `row`, unit `u` (elements 8u..8u+7).
MLA_DEVINL void st_unit(uint8_t* base, int row, int u, uint4 v) {
  *reinterpret_cast<uint4*>(base + row * 128 + ((u ^ (row & 7)) << 4)) = v;
}

MLA_DEVINL uint4 bf16x8_to_f16x8(uint4 v) {
  uint4 o;
  float2 f;
  f = bf16x2_to_f32(v.x); o.x = pack_f16x2(f.x, f.y);
  f = bf16x2_to_f32(v.y); o.y = pack_f16x2(f.x, f.y);
  f = bf16x2_to_f32(v.z); o.z = pack_f16x2(f.x, f.y);
  f = bf16x2_to_f32(v.w); o.w = pack_f16x2(f.x, f.y);
  return o;
}

MLA_DEVINL uint32_t i8x2_to_f16x2(uint32_t w, int sh, float d) {
  const float a = static_cast<float>(static_cast<int8_t>((w >> sh) & 0xFF));
  const float b = static_cast<float>(static_cast<int8_t>((w >> (sh + 8)) & 0xFF));
  return pack_f16x2(a * d, b * d);
}

template <bool kQ8, bool kDecode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQr = sm;
  uint8_t* sKV = sm + kOffKv;
  uint8_t* sP = sm + kOffP;
  uint8_t* sX = sm + kOffX;
  Bars& B = *reinterpret_cast<Bars*>(sm + kOffBar);

  const uint32_t rank = tc::cluster_ctarank(), peer = rank ^ 1u;
  const int nch = rank == 0 ? 5 : 4;          // 64-dim chunks of this CTA's score contraction
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.n_head;

  // ---- work item -----------------------------------------------------------
  const int n_items = gridDim.x >> 1;
  const int item = n_items - 1 - static_cast<int>(blockIdx.x >> 1);   // long prefill rows first
  int64_t key_base = 0;     // cache row of item key 0
  int kend = 0;             // keys [0, kend) of this item
  int nvalid = 0;           // valid query rows
  int64_t qrow0 = 0;        // flattened (token, head) index of row 0
  int64_t slot0 = 0;        // decode: partial slot of row 0
  if constexpr (kDecode) {
    const int b = item / a.n_split, s = item % a.n_split;
    const int len = a.seq_len[b];
    const int lo = s * a.chunk;
    if (lo >= len) return;                    // both CTAs of the pair leave together
    key_base = a.seq_start[b] + lo;
    kend = min(len - lo, a.chunk);
    nvalid = H;
    qrow0 = static_cast<int64_t>(b) * H;
    slot0 = static_cast<int64_t>(item) * H;
  } else {
    const int64_t rho0 = static_cast<int64_t>(item) * kRows;
    nvalid = static_cast<int>(min(static_cast<int64_t>(kRows), a.n_qrows - rho0));
    kend = a.q_pos0 + static_cast<int>((rho0 + nvalid - 1) / H) + 1;
    qrow0 = rho0;
  }
  const int n_tiles = (kend + kBK - 1) / kBK;

  // ---- setup -----------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&B.kv_full[i], 128);
      mbar_init(&B.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_free[i], 128);
      mbar_init(&B.x_full[i], 1);
    }
    mbar_init(&B.p_full, 128);
    mbar_init(&B.pv_done, 1);
    mbar_init(&B.q_ready, 128);
    B.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(&B.tmem, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  tc::cluster_sync();                 // peer barriers initialised before any remote arrival
  tc::fence_after_sync();
  const uint32_t tmem = B.tmem;

  if (warp < 4) {
    // ======================= softmax / exchange / epilogue =====================
    const int i = threadIdx.x;        // query row of this thread == TMEM lane
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    const bool rvalid = i < nvalid;
    const int64_t qrow = qrow0 + i;
    int lim;                          // last visible key index (item-relative)
    if constexpr (kDecode) {
      lim = kend - 1;
    } else {
      lim = rvalid ? a.q_pos0 + static_cast<int>(qrow / H) : kend - 1;
    }
    // Q latent half -> TMEM (A operand: fp16 pairs, row = lane).
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_lat) + qrow * kLatent +
                                                        256 * rank);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = rvalid ? __ldg(src + c * 8 + v) : make_uint4(0, 0, 0, 0);
          r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
        }
        tc::tmem_st32(tmem + lanes + kTmQ + c * 32, r);
      }
      tc::tmem_st_wait();
      if (rank == 0) {                // RoPE query part -> smem (bf16 -> fp16)
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_pe) + qrow * kRope);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = rvalid ? __ldg(qp + u) : make_uint4(0, 0, 0, 0);
          st_unit(sQr, i, u, bf16x8_to_f16x8(x));
        }
        tc::fence_proxy_async();
      }
      tc::fence_before_sync();
      mbar_arrive(&B.q_ready);
    }

    const uint32_t peer_x = tc::mapa(smem_u32(sX), peer);
    const uint32_t peer_xbar = tc::mapa(smem_u32(&B.x_full[0]), peer);
    const float sl = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int b = j & 1;
      ok = wait_all(&B.s_full[b], (j >> 1) & 1, a);
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t own[32];
      {
        uint32_t r0[32], r1[32];
        tc::tmem_ld32(tmem + lanes + kTmS + b * 64, r0);
        tc::tmem_ld32(tmem + lanes + kTmS + b * 64 + 32, r1);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        mbar_arrive(&B.s_free[b]);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          own[k] = pack_f16x2(__uint_as_float(r0[2 * k]) * sl, __uint_as_float(r0[2 * k + 1]) * sl);
          own[16 + k] = pack_f16x2(__uint_as_float(r1[2 * k]) * sl, __uint_as_float(r1[2 * k + 1]) * sl);
        }
      }
      // exchange the fp16 partial scores with the peer
#pragma unroll
      for (int g = 0; g < 8; ++g)
        tc::st_async_v4(peer_x + b * kXBytes + (g * kRows + i) * 16,
                        make_uint4(own[4 * g], own[4 * g + 1], own[4 * g + 2], own[4 * g + 3]),
                        peer_xbar + b * 8);
      if (i == 0) mbar_arrive_expect_tx(&B.x_full[b], kXBytes);
      ok = __all_sync(0xffffffffu, tc::mbar_wait_cluster_bounded(&B.x_full[b], (j >> 1) & 1, a.polls, a.err));
      if (!ok) break;
      float s[64];
      float mt = -INFINITY;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint4 pv = *reinterpret_cast<const uint4*>(sX + b * kXBytes + (g * kRows + i) * 16);
        const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = f16x2_to_f32(own[4 * g + e]);
          const float2 y = f16x2_to_f32(pw[e]);
          const int k = 8 * g + 2 * e;
          const int kk = j * kBK + k;
          s[k] = kk <= lim ? x.x + y.x : -INFINITY;
          s[k + 1] = kk + 1 <= lim ? x.y + y.y : -INFINITY;
          mt = fmaxf(mt, fmaxf(s[k], s[k + 1]));
        }
      }
      const float m_new = fmaxf(m_run, mt);
      const bool need = m_new > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = exp2f(m_run - m_new);
        m_run = m_new;
      }
      const bool warp_need = __any_sync(0xffffffffu, need);
      uint32_t pk[32];
      float lsum = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        pk[k] = pack_f16x2(exp2f(s[2 * k] - m_run), exp2f(s[2 * k + 1] - m_run));
        const float2 f = f16x2_to_f32(pk[k]);
        lsum += f.x + f.y;
      }
      l_run = l_run * alpha + lsum;
      if (j >= 1) {
        ok = wait_all(&B.pv_done, (j - 1) & 1, a);
        if (!ok) break;
        tc::fence_after_sync();
        if (warp_need) {              // rescale this warp's 32 output rows
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[32];
            tc::tmem_ld32(tmem + lanes + kTmO + c * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::tmem_st32(tmem + lanes + kTmO + c * 32, o);
          }
          tc::tmem_st_wait();
        }
      }
#pragma unroll
      for (int g = 0; g < 8; ++g) st_unit(sP, i, g, make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]));
      tc::fence_proxy_async();
      tc::fence_before_sync();
      mbar_arrive(&B.p_full);
    }
    if (ok) ok = wait_all(&B.pv_done, (n_tiles - 1) & 1, a);
    if (ok) {
      tc::fence_after_sync();
      const float inv = 1.f / l_run;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lanes + kTmO + c * 32, o);
        tc::tmem_ld_wait();
        if (!rvalid) continue;
        if constexpr (kDecode) {
          uint4* dst = reinterpret_cast<uint4*>(a.ws_o + (slot0 + i) * kLatent + 256 * rank + c * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v) dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o_lat) + qrow * kLatent + 256 * rank + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_f16x2(__uint_as_float(o[8 * v]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_f16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_f16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_f16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (rank == 0 && rvalid) {
        if constexpr (kDecode) {
          a.ws_ml[2 * (slot0 + i)] = m_run;
          a.ws_ml[2 * (slot0 + i) + 1] = l_run;
        } else if (a.lse != nullptr) {
          a.lse[qrow] = (m_run + log2f(l_run)) * kLn2;
        }
      }
    }
    if (!ok) B.abort = 1;
  } else if (warp < 8) {
    // ============================ producer =====================================
    const int pt = threadIdx.x - 128;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int st = j % kStages;
      if (j >= kStages) ok = mbar_wait_bounded(&B.kv_empty[st], ((j / kStages) - 1) & 1, a.polls, a.err);
      if (!ok) break;
      uint8_t* stage = sKV + st * kKvStage;
      const int k0 = j * kBK;
      if constexpr (!kQ8) {
        // units of 8 values: per key 32 latent units (+8 RoPE units on rank 0)
        const int upk = nch * 8;
        const int nu = kBK * upk / 128;                 // 20 or 16 per thread
        uint4 v[20];
#pragma unroll
        for (int t = 0; t < 20; ++t) {
          if (t < nu) {
            const int idx = pt + t * 128;
            const int key = idx / upk, cu = idx % upk;
            const int dim = cu < 32 ? 256 * static_cast<int>(rank) + cu * 8 : kLatent + (cu - 32) * 8;
            v[t] = make_uint4(0, 0, 0, 0);
            if (k0 + key < kend)
              v[t] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.kv) +
                                                          (key_base + k0 + key) * kRow + dim));
          }
        }
#pragma unroll
        for (int t = 0; t < 20; ++t) {
          if (t < nu) {
            const int idx = pt + t * 128;
            const int key = idx / upk, cu = idx % upk;
            st_unit(stage + (cu >> 3) * kKvChunk, key, cu & 7, bf16x8_to_f16x8(v[t]));
          }
        }
      } else {
        // units of 16 codes: per key 16 latent units (+4 RoPE units on rank 0)
        const int upk = nch * 4;
        const int nu = kBK * upk / 128;                 // 10 or 8 per thread
        uint4 v[10];
        float d[10];
#pragma unroll
        for (int t = 0; t < 10; ++t) {
          if (t < nu) {
            const int idx = pt + t * 128;
            const int key = idx / upk, cu = idx % upk;
            const int dim = cu < 16 ? 256 * static_cast<int>(rank) + cu * 16 : kLatent + (cu - 16) * 16;
            v[t] = make_uint4(0, 0, 0, 0);
            d[t] = 0.f;
            if (k0 + key < kend) {
              const int64_t row = key_base + k0 + key;
              v[t] = __ldg(reinterpret_cast<const uint4*>(a.kv_q + row * kRow + dim));
              d[t] = __half2float(__ushort_as_half(__ldg(a.kv_d + static_cast<int64_t>(dim >> 5) * a.ld_d + row)));
            }
          }
        }
#pragma unroll
        for (int t = 0; t < 10; ++t) {
          if (t < nu) {
            const int idx = pt + t * 128;
            const int key = idx / upk, cu = idx % upk;
            const int c = cu >> 2, u = (cu & 3) * 2;    // chunk and first 8-element unit
            uint4 lo, hi;
            lo.x = i8x2_to_f16x2(v[t].x, 0, d[t]);  lo.y = i8x2_to_f16x2(v[t].x, 16, d[t]);
            lo.z = i8x2_to_f16x2(v[t].y, 0, d[t]);  lo.w = i8x2_to_f16x2(v[t].y, 16, d[t]);
            hi.x = i8x2_to_f16x2(v[t].z, 0, d[t]);  hi.y = i8x2_to_f16x2(v[t].z, 16, d[t]);
            hi.z = i8x2_to_f16x2(v[t].w, 0, d[t]);  hi.w = i8x2_to_f16x2(v[t].w, 16, d[t]);
            st_unit(stage + c * kKvChunk, key, u, lo);
            st_unit(stage + c * kKvChunk, key, u + 1, hi);
          }
        }
      }
      tc::fence_proxy_async();
      mbar_arrive(&B.kv_full[st]);
    }
    if (!ok) B.abort = 1;
  } else if (lane == 0) {
    // ============================== MMA issue ==================================
    constexpr uint32_t idesc_qk = tc::idesc_f16(128, kBK, false, false, false);
    constexpr uint32_t idesc_pv = tc::idesc_f16(128, 256, false, false, true);
    bool ok = mbar_wait_bounded(&B.q_ready, 0, a.polls, a.err);
    tc::fence_after_sync();
    auto issue_pv = [&](int jj) -> bool {
      if (!mbar_wait_bounded(&B.p_full, jj & 1, a.polls, a.err)) return false;
      tc::fence_after_sync();
      const uint32_t v0 = smem_u32(sKV + (jj % kStages) * kKvStage);
      const uint32_t p0 = smem_u32(sP);
#pragma unroll
      for (int ks = 0; ks < kBK / 16; ++ks)
        tc::mma_ss(tmem + kTmO, tc::sdesc_sw128(p0 + ks * 32, 16, 1024),
                   tc::sdesc_sw128(v0 + ks * 2048, kKvChunk, 1024), idesc_pv, (jj > 0 || ks > 0) ? 1u : 0u);
      tc::mma_commit(&B.kv_empty[jj % kStages]);
      tc::mma_commit(&B.pv_done);
      return true;
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int st = j % kStages, b = j & 1;
      ok = mbar_wait_bounded(&B.kv_full[st], (j / kStages) & 1, a.polls, a.err);
      if (ok && j >= 2) ok = mbar_wait_bounded(&B.s_free[b], ((j - 2) >> 1) & 1, a.polls, a.err);
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t k0 = smem_u32(sKV + st * kKvStage);
      const uint32_t d = tmem + kTmS + b * 64;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks)        // latent half: A = Q from TMEM
        tc::mma_ts(d, tmem + kTmQ + ks * 8, tc::sdesc_sw128(k0 + (ks >> 2) * kKvChunk + (ks & 3) * 32, 16, 1024),
                   idesc_qk, ks > 0 ? 1u : 0u);
      if (rank == 0) {
        const uint32_t q0 = smem_u32(sQr);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)       // RoPE part: A = Q_pe from smem
          tc::mma_ss(d, tc::sdesc_sw128(q0 + ks * 32, 16, 1024),
                     tc::sdesc_sw128(k0 + 4 * kKvChunk + ks * 32, 16, 1024), idesc_qk, 1u);
      }
      tc::mma_commit(&B.s_full[b]);
      if (j >= 1) ok = issue_pv(j - 1);
    }
    if (ok && n_tiles > 0) ok = issue_pv(n_tiles - 1);
    if (!ok) B.abort = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();                 // no exchange may target a CTA that has left
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <bool kQ8, bool kDecode>
cudaError_t launch_one(const AttnTcArgs& a, int n_items, cudaStream_t stream) {
  auto kern = attn_tc_kernel<kQ8, kDecode>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(2 * n_items), kThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int attn_tc_rows_per_item() { return kRows; }

cudaError_t launch_attn_tc(const AttnTcArgs& a, bool q8, bool decode, int n_items, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (q8) return decode ? launch_one<true, true>(a, n_items, stream) : launch_one<true, false>(a, n_items, stream);
  return decode ? launch_one<false, true>(a, n_items, stream) : launch_one<false, false>(a, n_items, stream);
}

}  // namespace mla
