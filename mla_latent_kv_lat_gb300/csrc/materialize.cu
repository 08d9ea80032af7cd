// The materialised prefill (pp_opt): instead of absorbing the up-projections
// into the query, decompress every visible cache row into per-head keys and
// values once per chunk and run standard causal attention with 192-wide
// queries/keys and 128-wide values ("MLA matrix absorption in ik_llama.cpp",
// sec. 8.4: for prefill chunks of >= 128 tokens over >= 1024 cache rows the
// implementation materialises each head's K/V from the latent cache and
// switches to standard flash attention).  For a long chunk this is ~3x fewer
// FLOPs than the absorbed form (640 vs 2176 per visible pair and head, plus
// 256 x 512 x 2 per cache row and head for the decompression).
//
// Two kernels per head chunk of hc heads:
//   decompress  K16[j][h] = c_kv[j] . wk_b[h]^T and V16[j][h] = c_kv[j] . wv_b[h]
//               (tcgen05, bf16 x bf16 -> fp32, rounded once to fp16).
//   attention   one head x 128 query rows per item, keys in tiles of 128:
//               S = Q K^T (Q in TMEM, K from a 3-stage TMA ring: the nope part
//               from K16, the RoPE part straight from the cache), causal
//               online softmax (8 warps, two threads per row), P written back
//               over S in TMEM as fp16 and used there as the A operand of
//               O += P V (V from a 2-stage ring); 4 warps load each item's Q
//               (q_nope converted to fp16, q_pe as the cache's RoPE keys are)
//               into TMEM and write the previous item's o = O / l.
// The nope keys, values, queries and P are fp16 for the same reason as the
// absorbed path: bf16 keys alone would cost ~1.5e-3 of the 2e-3 mean relative
// error budget.  The RoPE part of the scores multiplies the bf16 q_pe and k_pe
// as they are (with a q8_0 cache: the fp16 staged keys and fp16 q_pe).
#include "kernels.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kFR = 128;                          // query rows per item (MMA M)
constexpr int kFN = 128;                          // keys per tile (MMA N of Q K^T)

// ---------------------------------------------------------------------------
// decompress: CTA (head hl of the chunk, part p, row group g); part 0 makes
// keys (W = wk_b[h] as a K-major B operand: 128 output rows of 512), part 1
// values (W = wv_b[h], N-major).  W stays in shared memory; 128-row tiles of
// the latent cache stream through a 4-stage ring; 4 accumulator slots in TMEM.
// kAF16: the rows are the fp16 staging copy of a q8_0 cache; W (bf16) is then
// converted to fp16 in shared memory by the epilogue warps before the first
// MMA (both operands of an MMA have one type).
// ---------------------------------------------------------------------------
constexpr int kDStages = 5;   // a chunk's MMAs take ~340 cycles: five stages cover the TMA latency
constexpr int kDChunk = 128 * 128;                // 16 KB: 128 rows x 64 bf16
constexpr int kDWBytes = 128 * 1024;              // W: 512 x 128 bf16
constexpr int kDStgBytes = 4 * 2048;
constexpr int kDSmem = 1024 + kDWBytes + kDStages * kDChunk + kDStgBytes + 256;
static_assert(kDSmem <= 232448, "shared memory");
constexpr int kDThreads = 192;

struct DecompArgs {
  uint16_t* k16;     // fp16 [rows][hc][128]
  uint16_t* v16;     // fp16 [rows][hc][128]
  int64_t rows;
  int hc, h0, row_tiles;
  int* err;
  uint32_t wait_us;
};

// Store 64 bytes of each of a warp's 32 rows (lane = row) to dst_row0 +
// row * row_stride through the warp's 2 KB slice: each store instruction
// writes 8 rows x 64 contiguous bytes.  Rows >= nrows are not stored.
MLA_DEVINL void store_rows64_pp(uint8_t* stg, int lane, const uint4 (&w)[4], uint8_t* dst_row0, int64_t row_stride,
                                int nrows) {
#pragma unroll
  for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(stg + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) = w[v];
  __syncwarp();
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int rr = (lane >> 2) + 8 * m, part = lane & 3;
    const uint4 x = *reinterpret_cast<const uint4*>(stg + rr * 64 + ((part ^ ((rr >> 1) & 3)) << 4));
    if (rr < nrows) *reinterpret_cast<uint4*>(dst_row0 + rr * row_stride + part * 16) = x;
  }
  __syncwarp();
}

template <bool kAF16>
__global__ void __launch_bounds__(kDThreads, 1)
    pp_decompress_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmWk,
                            const __grid_constant__ CUtensorMap tmWv, DecompArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sW = sm;
  uint8_t* sA = sm + kDWBytes;
  uint8_t* sStg = sA + kDStages * kDChunk;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + kDStgBytes);
  uint64_t* a_full = bars;
  uint64_t* a_empty = bars + kDStages;
  uint64_t* acc_full = bars + 2 * kDStages;
  uint64_t* acc_empty = acc_full + 4;
  uint64_t* w_full = acc_empty + 4;
  uint64_t* w_conv = w_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(w_conv + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = blockIdx.x, part = blockIdx.y, grp = blockIdx.z, G = gridDim.z;
  const int h = g.h0 + hl;
  const int n_tiles = (g.row_tiles - grp + G - 1) / G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 128);
    }
    mbar_init(w_full, 1);
    mbar_init(w_conv, 128);
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
      mbar_arrive_expect_tx(w_full, kDWBytes);
      if (part == 0) {         // wk_b[h]: [128 out][512 in] -> 8 K-major chunks of [128][64]
        for (int c = 0; c < 8; ++c) tc::tma_load_3d(sW + c * kDChunk, &tmWk, w_full, c * 64, 0, h);
      } else {                 // wv_b[h]: [512 in][128 out] -> 2 N-major chunks of [512][64], two boxes each
        for (int c = 0; c < 2; ++c)
          for (int r = 0; r < 2; ++r) tc::tma_load_3d(sW + c * 65536 + r * 32768, &tmWv, w_full, c * 64, r * 256, h);
      }
      bool ok = true;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int tt = grp + i * G;
        for (int kc = 0; kc < 8; ++kc) {
          const int u = i * 8 + kc, st = u % kDStages;
          if (u >= kDStages && !mbar_wait_bounded(&a_empty[st], ((u / kDStages) - 1) & 1, g.wait_us, g.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&a_full[st], kDChunk);
          tc::tma_load_3d(sA + st * kDChunk, &tmA, &a_full[st], kc * 64, tt * 128, 0);
        }
      }
    }
  } else if (warp == 1) {
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(kAF16 ? w_conv : w_full, 0, g.wait_us, g.err));
    tc::fence_after_sync();
    const uint32_t idesc = part == 0 ? tc::idesc_f16(128, 128, !kAF16, false, false)
                                     : tc::idesc_f16(128, 128, !kAF16, false, true);
    const uint32_t w0 = smem_u32(sW);
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int slot = i & 3;
      if (i >= 4) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[slot], ((i >> 2) - 1) & 1, g.wait_us, g.err));
      tc::fence_after_sync();
      for (int kc = 0; ok && kc < 8; ++kc) {
        const int u = i * 8 + kc, st = u % kDStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&a_full[st], (u / kDStages) & 1, g.wait_us, g.err));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t a0 = smem_u32(sA + st * kDChunk);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const int k = kc * 4 + ks;      // 16-wide step of the 512 latent dims
          const uint64_t bd = part == 0 ? tc::sdesc_sw128(w0 + (k >> 2) * kDChunk + (k & 3) * 32, 16, 1024)
                                        : tc::sdesc_sw128(w0 + k * 2048, 65536, 1024);
          tc::mma_ss_warp(tmem + slot * 128, tc::sdesc_sw128(a0 + ks * 32, 16, 1024), bd, idesc, (kc | ks) != 0);
        }
        tc::mma_commit_warp(&a_empty[st]);
      }
      if (ok) tc::mma_commit_warp(&acc_full[slot]);
    }
  } else {
    const int q = warp & 3;
    uint8_t* stg = sStg + (warp - 2) * 2048;
    uint16_t* out = part == 0 ? g.k16 : g.v16;
    const int64_t row_stride = static_cast<int64_t>(g.hc) * kVHead * 2;   // bytes
    float amax = 0.f;
    bool ok = true;
    if constexpr (kAF16) {
      // W bf16 -> fp16 in place: a 16-byte unit holds 8 consecutive values of
      // one row, so the swizzle does not matter
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(w_full, 0, g.wait_us, g.err));
      uint4* w = reinterpret_cast<uint4*>(sW);
      for (int x = threadIdx.x - 64; x < kDWBytes / 16; x += 128) {
        const uint4 v = w[x];
        uint4 o;
        float2 f;
        f = bf16x2_to_f32(v.x); o.x = pack_f16x2(f.x, f.y);
        f = bf16x2_to_f32(v.y); o.y = pack_f16x2(f.x, f.y);
        f = bf16x2_to_f32(v.z); o.z = pack_f16x2(f.x, f.y);
        f = bf16x2_to_f32(v.w); o.w = pack_f16x2(f.x, f.y);
        w[x] = o;
      }
      tc::fence_proxy_async();
      mbar_arrive(w_conv);
    }
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int tt = grp + i * G, slot = i & 3;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[slot], (i >> 2) & 1, g.wait_us, g.err));
      if (!ok) break;
      tc::fence_after_sync();
      const int64_t row0 = static_cast<int64_t>(tt) * 128 + q * 32;
      uint8_t* dst = reinterpret_cast<uint8_t*>(out + (row0 * g.hc + hl) * kVHead);
      const int nrows = static_cast<int>(min(static_cast<int64_t>(32), g.rows - row0));
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + slot * 128 + c * 32, r);
        tc::tmem_ld_wait();
        uint4 w[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = f32_absmax(amax, __uint_as_float(r[8 * v + e]));
          w[v].x = pack_f16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
          w[v].y = pack_f16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
          w[v].z = pack_f16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
          w[v].w = pack_f16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
        }
        store_rows64_pp(stg, lane, w, dst + c * 64, row_stride, nrows);
      }
      tc::fence_before_sync();
      mbar_arrive(&acc_empty[slot]);
    }
    if (f32_overflows_f16(amax)) record_error(g.err, MLA_ERR_RANGE);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// attention (see the file comment)
// ---------------------------------------------------------------------------
constexpr int kKChunk = kFN * 128;               // 16 KB: 128 keys x 64 fp16
constexpr int kKStage = 3 * kKChunk;             // 48 KB: nope 0-63, nope 64-127, rope
constexpr int kVStage = 2 * kKChunk;             // 32 KB: value dims 0-63, 64-127
constexpr int kKStages = 3, kVStages = 2;
constexpr int kFOffV = kKStages * kKStage;
constexpr int kFOffStg = kFOffV + kVStages * kVStage;
constexpr int kFStgBytes = 4 * 2048;
constexpr int kFOffAux = kFOffStg + kFStgBytes;
// row maxima [tile parity][thread of row][row], row sums [thread][row], row
// sums for the epilogue [item parity][row], failure flags [tile parity][warp]
constexpr int kFAuxBytes = (2 * 2 * kFR + 2 * kFR + 2 * kFR) * 4 + 2 * 8 * 4;
constexpr int kFOffBar = kFOffAux + kFAuxBytes;
constexpr int kFSmem = 1024 + kFOffBar + 256;
static_assert(kFSmem <= 232448, "shared memory");
constexpr int kFSoftWarps = 8, kFEpiWarp = 8, kFLoadWarp = 12, kFMmaWarp = 13;
constexpr int kFThreads = 14 * 32;
// TMEM: Q (192 fp16 = 96 columns), two score buffers (P written over their
// first 64 columns), O (128 fp32 columns).
constexpr uint32_t kTmQ = 0, kTmS = 128, kTmO = 384;
constexpr float kFRescale = 8.0f;

struct FaArgs {
  const uint16_t* q_nope;   // bf16 [T][H][128]
  const uint16_t* q_pe;     // bf16 [T][H][64]
  float* o;            // fp32 [T][H][128]
  float* lse;          // fp32 [T][H] or null
  int T, H, q_pos0, h0, hc, n_qt, n_items;
  float scale_log2;
  int* err;
  uint32_t wait_us;
};

struct FaItem {
  int hl, t0, nvalid, n_tiles;
};

// Items are (head, query tile), head-major so that the CTAs running at one
// time share the heads whose keys and values they read (L2); within a head
// the last query tiles (most keys) first.
MLA_DEVINL FaItem fa_item(const FaArgs& a, int idx) {
  FaItem it;
  it.hl = idx / a.n_qt;
  const int qt = a.n_qt - 1 - idx % a.n_qt;
  it.t0 = qt * kFR;
  it.nvalid = min(kFR, a.T - it.t0);
  const int kend = a.q_pos0 + it.t0 + it.nvalid;           // keys [0, kend) are visible to some row
  it.n_tiles = (kend + kFN - 1) / kFN;
  return it;
}

MLA_DEVINL int fa_round_item(int c, int g, int r) { return r * g + ((r & 1) ? g - 1 - c : c); }

struct FaBars {
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t pv_done;
  uint64_t q_ready, q_free, o_ready, o_free;
  uint64_t l_ready[2];
  uint32_t tmem;
};

template <bool kRopeBf16>
__global__ void __launch_bounds__(kFThreads, 1)
    pp_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmR, FaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = sm;
  uint8_t* sV = sm + kFOffV;
  uint8_t* sStg = sm + kFOffStg;
  float* aux_m = reinterpret_cast<float*>(sm + kFOffAux);   // [2][2][128]
  float* aux_l = aux_m + 4 * kFR;                           // [2][128]
  float* aux_lrow = aux_l + 2 * kFR;                        // [2][128]
  int* aux_fail = reinterpret_cast<int*>(aux_lrow + 2 * kFR);   // [2][8]
  FaBars& B = *reinterpret_cast<FaBars*>(sm + kFOffBar);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first = blockIdx.x, stride = gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
    }
    mbar_init(&B.s_full[0], 1);
    mbar_init(&B.s_full[1], 1);
    mbar_init(&B.p_full, kFSoftWarps * 32);
    mbar_init(&B.pv_done, 1);
    mbar_init(&B.q_ready, 128);
    mbar_init(&B.q_free, 1);
    mbar_init(&B.o_ready, 1);
    mbar_init(&B.o_free, 128);
    mbar_init(&B.l_ready[0], kFSoftWarps * 32);
    mbar_init(&B.l_ready[1], kFSoftWarps * 32);
    tc::fence_mbar_init();
  }
  if (warp == kFMmaWarp) {
    tc::tmem_alloc(&B.tmem, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = B.tmem;

  if (warp < kFSoftWarps) {
    // ============================ softmax ======================================
    const int q4 = warp & 3, hh = warp >> 2;
    const int i = q4 * 32 + lane;                 // query row of the item == TMEM lane
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    const float c2 = a.scale_log2;
    const int bar_id = 1 + q4;
    bool dead = false;
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
      if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, a.wait_us, a.err));
    };
    auto group_meet = [&](float* base, float val, int phase) {
      base[hh * kFR + i] = val;
      if (lane == 0) aux_fail[(phase & 1) * 8 + warp] = dead ? 1 : 0;
      tc::named_bar_sync(bar_id, 64);
      if (aux_fail[(phase & 1) * 8 + q4] != 0 || aux_fail[(phase & 1) * 8 + q4 + 4] != 0) dead = true;
    };
    bool range = false;
    int u0 = 0, k = 0;
#pragma unroll 1
    for (int rnd = 0; rnd * stride < a.n_items; ++rnd) {
      const int idx = fa_round_item(first, stride, rnd);
      if (idx >= a.n_items) continue;
      const FaItem it = fa_item(a, idx);
      const int lim = a.q_pos0 + it.t0 + i;       // last visible key of this row
      float m_run = -INFINITY, l_h = 0.f;
#pragma unroll 1
      for (int t = 0; t < it.n_tiles; ++t) {
        const int u = u0 + t, sb = u & 1;
        wait_ok(&B.s_full[sb], (u >> 1) & 1);
        uint32_t r[64];
        if (!dead) {
          tc::fence_after_sync();
          tc::tmem_ld<64>(tmem + lanes + kTmS + sb * 128 + 64 * hh, r);
          tc::tmem_ld_wait();
        }
        const int k0 = t * kFN + 64 * hh;
        if (k0 + 63 > lim) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (k0 + e > lim) r[e] = __float_as_uint(-INFINITY);
        }
        float mx[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) mx[e] = fmaxf(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
        float* mslot = aux_m + (u & 1) * 2 * kFR;
        group_meet(mslot, mx[0] * c2, u);         // after both threads read S: P may overwrite it
        const float mrow = fmaxf(mslot[i], mslot[kFR + i]);
        float alpha = 1.f;
        if (mrow > m_run + kFRescale) {
          alpha = tc::exp2_approx(m_run - mrow);
          m_run = mrow;
          l_h *= alpha;
        }
        // P.V of the previous tile has finished (O is stable for a rescale;
        // the barrier's phases are followed one by one).
        if (u >= 1) wait_ok(&B.pv_done, (u - 1) & 1);
        if (!dead && t >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            const uint32_t col = tmem + lanes + kTmO + 64 * hh + 32 * c;
            tc::tmem_ld32(col, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::tmem_st32(col, o);
          }
        }
        uint32_t pk[32];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          pk[e] = tc::exp2_approx_f16x2(pack_f16x2(fmaf(__uint_as_float(r[2 * e]), c2, -m_run),
                                                   fmaf(__uint_as_float(r[2 * e + 1]), c2, -m_run)));
          ls[e & 3] = tc::add_f16hi_f32(pk[e], tc::add_f16lo_f32(pk[e], ls[e & 3]));
        }
        l_h += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        if (dead) continue;
        tc::tmem_st32(tmem + lanes + kTmS + sb * 128 + 32 * hh, pk);    // P over S, fp16 pairs
        tc::tmem_st_wait();
        tc::fence_before_sync();
        mbar_arrive(&B.p_full);
      }
      // end of item: row sums to the epilogue warps
      if (i < it.nvalid && !dead && !(m_run < INFINITY)) range = true;
      group_meet(aux_l, l_h, u0 + it.n_tiles);
      const float l_row = aux_l[i] + aux_l[kFR + i];
      if (hh == 0) {
        aux_lrow[(k & 1) * kFR + i] = l_row;
        if (a.lse != nullptr && i < it.nvalid)
          a.lse[static_cast<int64_t>(it.t0 + i) * a.H + a.h0 + it.hl] = (m_run + log2f(l_row)) * 0.6931471805599453f;
      }
      mbar_arrive(&B.l_ready[k & 1]);
      u0 += it.n_tiles;
      ++k;
    }
    if (range) record_error(a.err, MLA_ERR_RANGE);
  } else if (warp < kFLoadWarp) {
    // ===================== Q loading and epilogue =============================
    const int q4 = warp & 3;
    const int i = q4 * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    uint8_t* stg = sStg + (warp - kFEpiWarp) * 2048;
    bool ok = true;
    auto epilogue = [&](const FaItem& pv, int kk) {
      ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&B.o_ready, kk & 1, a.wait_us, a.err));
      ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&B.l_ready[kk & 1], (kk >> 1) & 1, a.wait_us, a.err));
      if (!ok) return;
      tc::fence_after_sync();
      const float inv = 1.f / aux_lrow[(kk & 1) * kFR + i];
      uint8_t* dst = reinterpret_cast<uint8_t*>(
          a.o + (static_cast<int64_t>(pv.t0 + q4 * 32) * a.H + a.h0 + pv.hl) * kVHead);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lanes + kTmO + 32 * c, o);
        tc::tmem_ld_wait();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint4 w[4];
#pragma unroll
          for (int v = 0; v < 4; ++v)
            w[v] = make_uint4(__float_as_uint(__uint_as_float(o[16 * h2 + 4 * v]) * inv),
                              __float_as_uint(__uint_as_float(o[16 * h2 + 4 * v + 1]) * inv),
                              __float_as_uint(__uint_as_float(o[16 * h2 + 4 * v + 2]) * inv),
                              __float_as_uint(__uint_as_float(o[16 * h2 + 4 * v + 3]) * inv));
          store_rows64_pp(stg, lane, w, dst + (32 * c + 16 * h2) * 4, static_cast<int64_t>(a.H) * kVHead * 4,
                          pv.nvalid - q4 * 32);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&B.o_free);
    };
    FaItem prev;
    int k = 0;
    uint32_t qrun = 0;                            // query values converted to fp16: range check
#pragma unroll 1
    for (int rnd = 0; ok && rnd * stride < a.n_items; ++rnd) {
      const int idx = fa_round_item(first, stride, rnd);
      if (idx >= a.n_items) continue;
      const FaItem it = fa_item(a, idx);
      if (k > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&B.q_free, (k - 1) & 1, a.wait_us, a.err));
      if (!ok) break;
      tc::fence_after_sync();
      // Q row i: q_nope as fp16 (TMEM columns 0-63), q_pe as the RoPE keys are
      // stored (columns 64-95).  Once per item of ~300 key tiles, so the loads
      // need not be coalesced.
      const bool rvalid = i < it.nvalid;
      const int64_t th = static_cast<int64_t>(it.t0 + i) * a.H + a.h0 + it.hl;
      const uint4* qn = reinterpret_cast<const uint4*>(a.q_nope + th * kNope);
      const uint4* qp = reinterpret_cast<const uint4*>(a.q_pe + th * kRope);
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {               // 8 units = 32 TMEM columns per step
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x = rvalid ? __ldg(c < 2 ? qn + 8 * c + v : qp + v) : make_uint4(0, 0, 0, 0);
          if (c < 2 || !kRopeBf16) {
            qrun = bf16x2_absmax(bf16x2_absmax(qrun, x.x), x.y);
            qrun = bf16x2_absmax(bf16x2_absmax(qrun, x.z), x.w);
            uint4 y;
            float2 f;
            f = bf16x2_to_f32(x.x); y.x = pack_f16x2(f.x, f.y);
            f = bf16x2_to_f32(x.y); y.y = pack_f16x2(f.x, f.y);
            f = bf16x2_to_f32(x.z); y.z = pack_f16x2(f.x, f.y);
            f = bf16x2_to_f32(x.w); y.w = pack_f16x2(f.x, f.y);
            x = y;
          }
          r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
        }
        tc::tmem_st32(tmem + lanes + kTmQ + 32 * c, r);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      mbar_arrive(&B.q_ready);
      if (k > 0) epilogue(prev, k - 1);
      prev = it;
      ++k;
    }
    if (ok && k > 0) epilogue(prev, k - 1);
    if (bf16x2_absmax_overflows(qrun)) record_error(a.err, MLA_ERR_RANGE);
  } else if (warp == kFLoadWarp) {
    // ============================== loader =====================================
    if (lane == 0) {
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      tc::prefetch_tmap(&tmR);
      int u = 0;
      bool ok = true;
      for (int rnd = 0; ok && rnd * stride < a.n_items; ++rnd) {
        const int idx = fa_round_item(first, stride, rnd);
        if (idx >= a.n_items) continue;
        const FaItem it = fa_item(a, idx);
        for (int t = 0; t < it.n_tiles; ++t, ++u) {
          const int ks = u % kKStages, vs = u % kVStages, key = t * kFN;
          if (u >= kKStages && !mbar_wait_bounded(&B.k_empty[ks], ((u / kKStages) - 1) & 1, a.wait_us, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&B.k_full[ks], kKStage);
          uint8_t* kst = sK + ks * kKStage;
          tc::tma_load_3d(kst, &tmK, &B.k_full[ks], 0, it.hl, key);
          tc::tma_load_3d(kst + kKChunk, &tmK, &B.k_full[ks], 64, it.hl, key);
          tc::tma_load_3d(kst + 2 * kKChunk, &tmR, &B.k_full[ks], 0, 0, key);
          if (u >= kVStages && !mbar_wait_bounded(&B.v_empty[vs], ((u / kVStages) - 1) & 1, a.wait_us, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&B.v_full[vs], kVStage);
          uint8_t* vst = sV + vs * kVStage;
          tc::tma_load_3d(vst, &tmV, &B.v_full[vs], 0, it.hl, key);
          tc::tma_load_3d(vst + kKChunk, &tmV, &B.v_full[vs], 64, it.hl, key);
        }
      }
    }
  } else {
    // ============================== MMA issue ==================================
    // One warp issues every MMA, in the order QK(0), QK(1), PV(0), QK(2), PV(1),
    // ...: the tensor core runs them in issue order, so QK(u + 2), which
    // overwrites the score buffer holding P(u), always follows PV(u).
    constexpr uint32_t idesc_qk = tc::idesc_f16(kFR, kFN, false, false, false);
    constexpr uint32_t idesc_rope = tc::idesc_f16(kFR, kFN, kRopeBf16, false, false);
    constexpr uint32_t idesc_pv = tc::idesc_f16(kFR, kVHead, false, false, true);
    bool ok = true;
    auto issue_qk = [&](int u) {
      const int ks = u % kKStages, sb = u & 1;
      ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&B.k_full[ks], (u / kKStages) & 1, a.wait_us, a.err));
      if (!ok) return;
      tc::fence_after_sync();
      const uint32_t k0 = smem_u32(sK + ks * kKStage);
#pragma unroll
      for (int s = 0; s < 12; ++s)
        tc::mma_ts_warp(tmem + kTmS + sb * 128, tmem + kTmQ + s * 8,
                        tc::sdesc_sw128(k0 + (s >> 2) * kKChunk + (s & 3) * 32, 16, 1024), s < 8 ? idesc_qk : idesc_rope,
                        s > 0 ? 1u : 0u);
      tc::mma_commit_warp(&B.k_empty[ks]);
      tc::mma_commit_warp(&B.s_full[sb]);
    };
    int u = 0, k = 0;
#pragma unroll 1
    for (int rnd = 0; ok && rnd * stride < a.n_items; ++rnd) {
      const int idx = fa_round_item(first, stride, rnd);
      if (idx >= a.n_items) continue;
      const FaItem it = fa_item(a, idx);
      const int n = it.n_tiles;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&B.q_ready, k & 1, a.wait_us, a.err));
      if (!ok) break;
      tc::fence_after_sync();
      issue_qk(u);
      if (ok && n == 1) tc::mma_commit_warp(&B.q_free);
#pragma unroll 1
      for (int t = 0; ok && t < n; ++t) {
        if (t + 1 < n) {
          issue_qk(u + t + 1);
          if (ok && t + 2 == n) tc::mma_commit_warp(&B.q_free);   // Q may be replaced
        }
        const int uu = u + t, vs = uu % kVStages;
        ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&B.p_full, uu & 1, a.wait_us, a.err));
        if (ok && t == 0 && k > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&B.o_free, (k - 1) & 1, a.wait_us, a.err));
        ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&B.v_full[vs], (uu / kVStages) & 1, a.wait_us, a.err));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t v0 = smem_u32(sV + vs * kVStage);
        const uint32_t p0 = tmem + kTmS + (uu & 1) * 128;
#pragma unroll
        for (int s = 0; s < kFN / 16; ++s)
          tc::mma_ts_warp(tmem + kTmO, p0 + s * 8, tc::sdesc_sw128(v0 + s * 2048, kKChunk, 1024), idesc_pv,
                          (t > 0 || s > 0) ? 1u : 0u);
        tc::mma_commit_warp(&B.v_empty[vs]);
        tc::mma_commit_warp(&B.pv_done);
      }
      if (ok) tc::mma_commit_warp(&B.o_ready);
      u += n;
      ++k;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kFMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}


}  // namespace

// Workspace: K16 and V16 of one head chunk and, for a q8_0 cache, the fp16
// staging copy of its rows.
size_t pp_workspace_bytes(int H, int32_t T, int32_t q_pos0, int hc, bool q8) {
  (void)H;
  auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(q_pos0) + T;
  return 2 * up(rows * hc * kVHead * 2) + (q8 ? up(rows * kRow * 2) : 0);
}

cudaError_t launch_pp_prefill(const PpArgs& p, cudaStream_t stream) {
  auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  const int H = p.H, T = p.T;
  const int n_qt = (T + kFR - 1) / kFR;
  const int64_t rows = static_cast<int64_t>(p.q_pos0) + T;     // rows past the last query are never read
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  uint16_t* k16 = reinterpret_cast<uint16_t*>(ws);
  ws += up(static_cast<size_t>(rows) * p.hc * kVHead * 2);
  uint16_t* v16 = reinterpret_cast<uint16_t*>(ws);
  ws += up(static_cast<size_t>(rows) * p.hc * kVHead * 2);

  const bool q8 = p.kv == nullptr;
  cudaError_t e;
  const void* rows_src = p.kv;                 // the rows the decompression reads
  if (q8) {                                    // q8_0 cache: fp16 staging copy of the rows, RoPE keys included
    void* staged = ws;
    ws += up(static_cast<size_t>(rows) * kRow * 2);
    e = launch_stage_cache_f16(nullptr, p.kv_q, p.kv_d, p.ld_d, rows, staged, p.err, stream);
    if (e != cudaSuccess) return e;
    rows_src = staged;
  }

  CUtensorMap tmA, tmWk, tmWv, tmK, tmV, tmR;
  e = make_tmap_3d(&tmA, rows_src, !q8, kRow, static_cast<uint64_t>(rows), 1, kRow * 2,
                   static_cast<uint64_t>(rows) * kRow * 2, 64, 128, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tmWk, p.wk_b, true, kLatent, kNope, H, kLatent * 2, kLatent * kNope * 2, 64, 128, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tmWv, p.wv_b, true, kVHead, kLatent, H, kVHead * 2, kLatent * kVHead * 2, 64, 256, 1);
  if (e != cudaSuccess) return e;
  // the RoPE keys: columns 512-575 of the rows (bf16 cache, or the fp16 staged
  // rows of a q8_0 cache), base at column 512, row stride 1152 bytes
  e = make_tmap_3d(&tmR, static_cast<const uint16_t*>(rows_src) + kLatent, !q8, kRope, 1,
                   static_cast<uint64_t>(rows), kRow * 2, kRow * 2, 64, 1, kFN);
  if (e != cudaSuccess) return e;
  auto decomp = q8 ? pp_decompress_tc_kernel<true> : pp_decompress_tc_kernel<false>;
  e = cudaFuncSetAttribute(decomp, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
  if (e != cudaSuccess) return e;
  auto attn = q8 ? pp_attn_tc_kernel<false> : pp_attn_tc_kernel<true>;
  e = cudaFuncSetAttribute(attn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int row_tiles = static_cast<int>((rows + 127) / 128);
  for (int h0 = 0; h0 < H; h0 += p.hc) {
    const int hc = min(p.hc, H - h0);
    e = make_tmap_3d(&tmK, k16, false, kVHead, static_cast<uint64_t>(hc), static_cast<uint64_t>(rows), kVHead * 2,
                     static_cast<uint64_t>(hc) * kVHead * 2, 64, 1, kFN);
    if (e != cudaSuccess) return e;
    e = make_tmap_3d(&tmV, v16, false, kVHead, static_cast<uint64_t>(hc), static_cast<uint64_t>(rows), kVHead * 2,
                     static_cast<uint64_t>(hc) * kVHead * 2, 64, 1, kFN);
    if (e != cudaSuccess) return e;
    DecompArgs d;
    d.k16 = k16;
    d.v16 = v16;
    d.rows = rows;
    d.hc = hc;
    d.h0 = h0;
    d.row_tiles = row_tiles;
    d.err = p.err;
    d.wait_us = p.wait_us;
    // about twelve waves of CTAs (one per SM): row groups per (head, part)
    int G = static_cast<int>((12.0 * sms) / (2.0 * hc) + 0.5);
    G = max(1, min(G, row_tiles));
    decomp<<<dim3(hc, 2, G), kDThreads, kDSmem, stream>>>(tmA, tmWk, tmWv, d);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    FaArgs f;
    f.q_nope = static_cast<const uint16_t*>(p.q_nope);
    f.q_pe = static_cast<const uint16_t*>(p.q_pe);
    f.o = p.o;
    f.lse = p.lse;
    f.T = T;
    f.H = H;
    f.q_pos0 = p.q_pos0;
    f.h0 = h0;
    f.hc = hc;
    f.n_qt = n_qt;
    f.n_items = hc * n_qt;
    f.scale_log2 = p.scale_log2;
    f.err = p.err;
    f.wait_us = p.wait_us;
    const int grid = min(f.n_items, sms);
    attn<<<grid, kFThreads, kFSmem, stream>>>(tmK, tmV, tmR, f);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mla
