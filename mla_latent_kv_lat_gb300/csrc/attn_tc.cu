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
//     of the score contraction, and RoPE dimensions [32r, 32r+32).
//   * Each CTA computes its partial scores on tcgen05 into TMEM: the latent
//     part as fp16 x fp16 with Q from TMEM, the RoPE part as bf16 x bf16 (the
//     bf16 cache and q_pe enter it unrounded; with a q8_0 cache both are fp16)
//     into the same fp32 accumulator.  The partial is rounded to fp16 and sent
//     to the peer with st.async into distributed shared memory; both CTAs add
//     the same two fp16 partials in fp32, so their scores, maxima and
//     probabilities agree.
//   * Score MMAs run three tiles ahead of the P.V MMAs: the softmax sends tile
//     j+1's partial before it processes tile j, so the exchange latency and
//     the score MMAs overlap the softmax.
//   * P (fp16) goes to one of two shared-memory buffers (so P of tile j+1 may
//     be written while P.V of tile j runs); O_r += P V_r runs on tcgen05 with
//     V_r read in place from the latent cache tile (MN-major view).
//   * Cache tiles.  Prefill: every cluster reads every visible cache row, so
//     the rows are staged once as fp16 (latent and RoPE parts) before the
//     kernel, and one thread brings each tile in by TMA, already in the
//     128-byte-swizzled layout the tensor core reads.  Decode reads each row
//     once.  bf16 cache: the tiles arrive by TMA (each CTA first asks L2 for
//     the tile's whole rows) and six warps convert the latent part to fp16 in
//     place (exact); the RoPE part is used as bf16.  q8_0 cache: seven producer
//     warps load a tile's codes and scales while they wait for its stage,
//     dequantise (fp16 scale x int8 code) and store the fp16 tiles swizzled.
//   * Roles per CTA: warps 0-7 softmax / exchange (two threads per row, lanes
//     l and l + 16 of one warp, 32 keys of each 64-key tile each, so the row
//     maximum is one shuffle); then the epilogue warps, the loader (prefill:
//     one TMA warp; decode: TMA and converter warps, or seven q8_0 producer
//     warps); the last warp(s) issue the MMAs.  Every mbarrier wait is bounded.
#include <string.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kRows = 128;                   // query rows per cluster (MMA M)
constexpr int kBK = 64;                      // keys per tile
constexpr int kChunk = kBK * 128;            // 8 KB: 64 keys x 64 16-bit values
constexpr int kLatStage = 4 * kChunk;        // 32 KB: this CTA's 256 latent dims
constexpr int kLatStages = 4;
constexpr int kRopeStages = 2;   // a RoPE tile is done with long before its latent stage
// The 64 RoPE dims are split between the CTAs too: CTA r owns dims [32r, 32r+32)
// of the query and key RoPE parts (64-byte rows, 64-byte swizzle), so each CTA
// holds half a RoPE query tile and half a RoPE key ring; the 16 KB this frees
// pays for the second P buffer.
constexpr int kRopeHalf = 32;
constexpr int kRopeChunk = kBK * kRopeHalf * 2;   // 4 KB: 64 keys x 32 dims
constexpr int kQRopeBytes = kRows * kRopeHalf * 2;   // 8 KB: 128 rows x 32 dims
constexpr int kPBytes = kRows * 128;         // 16 KB: 128 rows x 64 keys fp16 (two buffers)
constexpr int kXBytes = kRows * kBK * 2;     // 16 KB: one exchange buffer (fp16 partial scores)
constexpr int kOffLat = kQRopeBytes;
constexpr int kOffRope = kOffLat + kLatStages * kLatStage;
constexpr int kOffP = kOffRope + kRopeStages * kRopeChunk;
constexpr int kOffX = kOffP + 2 * kPBytes;
constexpr int kOffAux = kOffX + 2 * kXBytes;
// Two softmax threads per query row, each taking 32 keys of every tile: lanes
// l and l + 16 of one warp, which reads its 16 TMEM lanes in two column
// halves (tcgen05.ld 16x32bx2).  (One thread per row, or four over two warps,
// measured slower; two in two warps, meeting at a named barrier for the row
// maximum, 4-5% slower on prefill.)
constexpr int kTpr = 2;
// the row sums handed to the epilogue warps [item % 4][row]
constexpr int kAuxBytes = 4 * kRows * 4;
// Epilogue warps' output staging: 2 KB per warp (32 rows x 64 B), so that the
// global stores leave as 64-byte row pieces, not 16-byte pieces of 32 rows.
constexpr int kStgBytes = 4 * 2048;
constexpr int kOffStg = kOffAux + kAuxBytes;
constexpr int kOffBar = kOffStg + kStgBytes;
constexpr int kBarBytes = 512;
constexpr int kSmem = 1024 + kOffBar + kBarBytes;
constexpr int kProducerWarps = 7;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kConvWarps = 2;
// bf16 decode: the two converter warps and the four epilogue warps convert
// each tile (the epilogue warps have little else to do in decode).
constexpr int kConvThreads = (kConvWarps + 4) * 32;
// Warp roles, in this order:
//   softmax (8) | epilogue (4; not for the q8_0 decode) | loader | MMA issue
// The epilogue warps (one per TMEM lane quadrant) load each item's Q into
// tensor memory as soon as the previous item's last score MMA has completed
// and write each item's output once its last P.V has, so the softmax warps go
// straight from one item's last tile to the next item's first.
// Loader: prefill, one TMA warp (the cache is staged as fp16 beforehand);
// bf16 decode, one TMA warp plus two warps converting each tile to fp16 in
// place; q8_0 decode, seven producer warps that load, dequantise and store.
// MMA issue: prefill, one warp for the score MMAs and one for P.V, so that a
// score tile waiting for its cache tile never holds back a P.V; decode, one.
__host__ __device__ constexpr int softmax_warps(bool, bool) { return 4 * kTpr; }
__host__ __device__ constexpr int epi_warps(bool q8, bool decode) { return decode && q8 ? 0 : 4; }
__host__ __device__ constexpr int loader_warps(bool q8, bool decode) {
  return !decode ? 1 : (q8 ? kProducerWarps : 1 + kConvWarps);
}
__host__ __device__ constexpr int loader_warp(bool q8, bool decode) {
  return softmax_warps(q8, decode) + epi_warps(q8, decode);
}
__host__ __device__ constexpr int mma_warp(bool q8, bool decode) {
  return loader_warp(q8, decode) + loader_warps(q8, decode);
}
__host__ __device__ constexpr int mma_warps(bool, bool decode) { return decode ? 1 : 2; }
__host__ __device__ constexpr int threads(bool q8, bool decode) {
  return (mma_warp(q8, decode) + mma_warps(q8, decode)) * 32;
}
// Registers per thread: warps go to the four SM sub-partitions in turn, and
// each sub-partition's 16384 registers are shared by its warps (allocated in
// steps of 8 a thread): 15 or 16 warps -> 128.
__host__ __device__ constexpr int max_regs(bool q8, bool decode) {
  return (16384 / (((threads(q8, decode) / 32 + 3) / 4) * 32)) / 8 * 8 > 255
             ? 248 : (16384 / (((threads(q8, decode) / 32 + 3) / 4) * 32)) / 8 * 8;
}
// TMEM columns: Q latent half (A operand, 256 fp16 = 128 cols), two fp32 score
// buffers of 64 columns, the fp32 output half (256 cols).
constexpr uint32_t kTmQ = 0, kTmS = 128, kTmO = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units: P stays <= 256 in fp16

// Where a decode cluster's tile range starts: computed once per CTA, by one
// warp during setup (a lane per sequence, so the sequence table costs two
// round trips however many roles walk it), and read by every role.
struct DecodeStart {
  int64_t lo, hi;   // the cluster's range [lo, hi) in the run of all sequences' costs
  int64_t S;        // where sequence b's costs start in that run
  int b;            // the first sequence that ends after lo (n_seq: none)
};

// Barriers that count arrivals from several warps are deep enough that a warp
// running ahead cannot arrive for a later use before every warp has arrived for
// the earlier one.  The softmax warps are coupled only through barriers and
// may drift a tile or two apart, so: one P barrier per P buffer (a warp stores
// P of tile u+2 only after P.V(u) has read that buffer, which needed every
// warp's P of tile u), and four row-sum slots (a warp ends item k+4 only after
// P.V of item k+2's first tile, which waited for the epilogue of item k+1).
struct Bars {
  uint64_t lat_full[kLatStages];
  uint64_t lat_tma[kLatStages];   // bf16 decode: the TMA tile has landed (before conversion)
  uint64_t lat_empty[kLatStages];
  uint64_t rope_full[kRopeStages];
  uint64_t rope_empty[kRopeStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t x_full[2];
  uint64_t x_empty[2];
  uint64_t p_full[2];    // by P buffer: all softmax threads have stored their P of the tile using it
  uint64_t pv_done[2];   // by P buffer: P.V of the tile that used it has completed
  uint64_t q_ready;   // arrival per item: Q of the next item is in TMEM
  uint64_t o_free;    // arrival per item: the epilogue has read O
  uint64_t q_free;    // commit per item (prefill): its last score MMA has completed
  uint64_t o_ready;   // commit per item (prefill): its last P.V has completed
  uint64_t l_ready[4];   // arrival per item (prefill, bf16 decode), by item % 4: row sums in aux
  uint32_t tmem;
  DecodeStart ds;        // decode: this cluster's start (written in setup)
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block");
static_assert(kSmem <= 232448, "shared memory");

MLA_DEVINL bool wait_all(uint64_t* bar, uint32_t parity, const AttnTcArgs& a) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, a.wait_us, a.err));
}

// Store one 16-byte unit (8 halves) into a 128-byte-swizzled K-major tile.
MLA_DEVINL void st_unit(uint8_t* base, int row, int u, uint4 v) {
  *reinterpret_cast<uint4*>(base + row * 128 + ((u ^ (row & 7)) << 4)) = v;
}

// The same for a 64-byte-swizzled tile (rows of 32 halves): unit u in [0, 4).
MLA_DEVINL void st_unit64(uint8_t* base, int row, int u, uint4 v) {
  *reinterpret_cast<uint4*>(base + row * 64 + ((u ^ ((row >> 1) & 3)) << 4)) = v;
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


// ---------------------------------------------------------------------------
// q8_0 decode producer: one 64-key tile of this CTA's cache part, the 256
// latent dims (16 units of 16 codes per key) plus this CTA's 32 RoPE dims (2
// units), dequantised to fp16 (fp16 scale x int8 code).  The 1152 units of a
// tile are dealt out so that each warp load instruction reads 4 keys x 8
// latent units: 128 contiguous code bytes of each key and 4 scales from each
// of 4 block rows, 8 cache lines in all.  (Dealt out key by key, 18 units at a
// time, an instruction touched ~19 lines, and the loads' L1 wavefronts made
// the q8_0 decode 11% slower.)
// ---------------------------------------------------------------------------
struct Q8Producer {
  static constexpr int UPK = 16 + 2;
  static constexpr int NUNITS = kBK * UPK;
  static constexpr int NU = (NUNITS + kProducerThreads - 1) / kProducerThreads;
  uint4 v[NU];
  uint32_t d[NU];   // raw fp16 scale bits: converted at store time, so no
                    // instruction waits on the load before then

  // Unit idx of a tile -> (key, code unit cu): idx < 1024 are the latent units,
  // 32 consecutive ones = units [8g, 8g + 8) of 4 consecutive keys; then the
  // RoPE units, two per key.
  MLA_DEVINL static void unit_of(int idx, int& key, int& cu) {
    static_assert(kBK == 64 && UPK == 18, "unit_of deals 64-key tiles of 18 units");
    if (idx < kBK * 16) {
      key = (idx >> 3) & (kBK - 1);
      cu = ((idx >> 9) << 3) + (idx & 7);
    } else {
      key = (idx - kBK * 16) >> 1;
      cu = 16 + (idx & 1);
    }
  }

  // Per-thread constants of the thread's units, the same for every tile
  // (computed once: the address arithmetic per unit and tile cost 4% of the
  // q8_0 decode): so = byte offset of the unit's low 16 bytes in its stage
  // (latent or RoPE; the high 16 bytes sit at so ^ 16), lc = key (bits 0-5),
  // scale block (bits 6-10) and code offset from the tile's first row (bits
  // 16-31, < 64 x 576).  pt's range lets the compiler resolve which rounds
  // hold latent units, which RoPE units and which none (3.5%).
  struct Plan {
    uint32_t so[NU], lc[NU];
  };
  MLA_DEVINL static void plan(Plan& p, int rank, int pt) {
    __builtin_assume(pt >= 0 && pt < kProducerThreads);
#pragma unroll
    for (int t = 0; t < NU; ++t) {
      const int idx = pt + t * kProducerThreads;
      int key, cu;
      unit_of(idx, key, cu);
      const int u = (cu & 3) * 2;
      const int dim = cu < 16 ? 256 * rank + cu * 16 : kLatent + kRopeHalf * rank + (cu - 16) * 16;
      p.so[t] = cu < 16 ? (cu >> 2) * kChunk + key * 128 + ((u ^ (key & 7)) << 4)   // st_unit's layout
                        : key * 64 + ((u ^ ((key >> 1) & 3)) << 4);                 // st_unit64's
      p.lc[t] = static_cast<uint32_t>(key) | (static_cast<uint32_t>(dim >> 5) << 6) |
                (static_cast<uint32_t>(key * kRow + dim) << 16);
    }
  }

  MLA_DEVINL void load(const AttnTcArgs& a, const Plan& p, int pt, int64_t key_base, int k0, int kend) {
    __builtin_assume(pt >= 0 && pt < kProducerThreads);
    const int64_t r0 = key_base + k0;
    const int8_t* codes = a.kv_q + r0 * kRow;
    const uint16_t* scales = a.kv_d + r0;
#pragma unroll
    for (int t = 0; t < NU; ++t) {
      const int idx = pt + t * kProducerThreads;
      v[t] = make_uint4(0, 0, 0, 0);
      d[t] = 0u;
      const int key = static_cast<int>(p.lc[t] & 63u);
      if (idx < NUNITS && k0 + key < kend) {
        v[t] = __ldg(reinterpret_cast<const uint4*>(codes + (p.lc[t] >> 16)));
        d[t] = __ldg(scales + static_cast<int64_t>((p.lc[t] >> 6) & 31u) * a.ld_d + key);
      }
    }
  }

  MLA_DEVINL void store(const Plan& p, uint8_t* lat, uint8_t* rope, int pt) const {
    __builtin_assume(pt >= 0 && pt < kProducerThreads);
#pragma unroll
    for (int t = 0; t < NU; ++t) {
      const int idx = pt + t * kProducerThreads;
      if (idx >= NUNITS) break;
      uint4 lo, hi;
      const uint32_t d2 = d[t] | (d[t] << 16);
      i8x4_to_f16x4(v[t].x, d2, lo.x, lo.y);
      i8x4_to_f16x4(v[t].y, d2, lo.z, lo.w);
      i8x4_to_f16x4(v[t].z, d2, hi.x, hi.y);
      i8x4_to_f16x4(v[t].w, d2, hi.z, hi.w);
      uint8_t* base = idx < kBK * 16 ? lat : rope;
      *reinterpret_cast<uint4*>(base + p.so[t]) = lo;
      *reinterpret_cast<uint4*>(base + (p.so[t] ^ 16u)) = hi;
    }
  }
};

// ---------------------------------------------------------------------------
// Work items.  With G clusters, cluster c runs one item per round r: item
// index rG + c in even rounds and rG + (G-1-c) in odd ones.  Prefill items
// come longest first, so the snake order pairs long with short and keeps the
// clusters' totals close.  Every role of both CTAs walks the same sequence,
// and every ring and barrier phase counts tiles across items, so one item's
// first tiles load and start while the previous item drains.
// ---------------------------------------------------------------------------
MLA_DEVINL int round_item(int c, int g, int r) { return r * g + ((r & 1) ? g - 1 - c : c); }

struct Item {
  int64_t key_base;   // cache row of item key 0
  int kend;           // keys [0, kend) of this item (0: nothing to do)
  int nvalid;         // valid query rows
  int64_t qrow0;      // flattened (token, head) index (prefill) or sequence x H (decode) of row 0
  int64_t slot0;      // decode: partial slot of row 0
  int n_tiles;
};

// Prefill: row tile `item` (the snake order over G clusters picks them).
MLA_DEVINL Item prefill_item(const AttnTcArgs& a, int idx) {
  Item it;
  const int item = a.n_items - 1 - idx;       // long prefill rows (late tokens) first
  const int64_t rho0 = static_cast<int64_t>(item) * kRows;
  it.nvalid = static_cast<int>(min(static_cast<int64_t>(kRows), a.n_qrows - rho0));
  it.kend = a.q_pos0 + static_cast<int>((rho0 + it.nvalid - 1) / a.n_head) + 1;
  it.key_base = 0;
  it.qrow0 = rho0;
  it.slot0 = 0;
  it.n_tiles = (it.kend + kBK - 1) / kBK;
  return it;
}

// This cluster's items in order.  Prefill: one row tile per round (snake
// order).  Decode: the pieces of the cluster's tile range (see
// decode_cluster_lo), one per sequence it meets.  (Two types, so that the
// prefill warps carry no decode state in registers.)
template <bool kDecode>
struct ItemIter;

// Whole warp.  Invalid sequences cost nothing (they are skipped).
MLA_DEVINL DecodeStart decode_start(const AttnTcArgs& a, int c, int g, int lane) {
  auto tiles = [&](int q) -> int64_t {
    return q < a.n_seq ? decode_seq_cost(decode_valid_len(a.seq_start, a.seq_len, q, a.max_len, a.n_rows),
                                         a.piece_cost)
                       : 0;
  };
  int64_t T = 0;
  for (int q0 = 0; q0 < a.n_seq; q0 += 32) T += tiles(q0 + lane);
  T = warp_sum_i64(T);
  const int64_t lo = decode_cluster_lo(T, g, c), hi = decode_cluster_lo(T, g, c + 1);
  int b = a.n_seq;
  int64_t S = T, run = 0;
  for (int q0 = 0; q0 < a.n_seq; q0 += 32) {
    const int64_t t = tiles(q0 + lane);
    int64_t incl = t;                         // inclusive scan over the lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, q0 + lane < a.n_seq && run + incl > lo);
    if (hit != 0u) {
      const int f = __ffs(hit) - 1;
      b = q0 + f;
      S = run + __shfl_sync(0xffffffffu, incl - t, f);
      break;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  DecodeStart out;
  out.lo = lo;
  out.hi = hi;
  out.S = S;
  out.b = b;
  return out;
}

template <>
struct ItemIter<false> {
  const AttnTcArgs* a;
  int c, g, r;
  MLA_DEVINL void init(const AttnTcArgs& args, int cluster, int clusters, const DecodeStart*) {
    a = &args; c = cluster; g = clusters; r = 0;
  }
  MLA_DEVINL bool next(Item& it) {
    while (r * g < a->n_items) {
      const int idx = round_item(c, g, r++);
      if (idx < a->n_items) {
        it = prefill_item(*a, idx);
        return true;
      }
    }
    return false;
  }
};

template <>
struct ItemIter<true> {
  const AttnTcArgs* a;
  int c;
  int b;                       // next sequence
  int64_t lo, hi, S;           // cluster range, start of sequence b (in cost units)
  MLA_DEVINL void init(const AttnTcArgs& args, int cluster, int, const DecodeStart* ds) {
    a = &args; c = cluster;
    lo = ds->lo; hi = ds->hi; S = ds->S; b = ds->b;
  }
  MLA_DEVINL bool next(Item& it) {
    while (b < a->n_seq && S < hi) {
      const int32_t len = decode_valid_len(a->seq_start, a->seq_len, b, a->max_len, a->n_rows);   // 0: skipped
      const int64_t cost = decode_seq_cost(len, a->piece_cost);
      const int64_t r0 = S + (len > 0 ? a->piece_cost : 0);   // where the sequence's tiles start
      const int64_t p_lo = max(lo, r0), p_hi = min(hi, S + cost);
      const int bb = b;
      S += cost;
      ++b;
      if (p_lo >= p_hi) continue;
      const int64_t k0 = (p_lo - r0) * kBK;          // first key of the piece in its sequence
      it.key_base = a->seq_start[bb] + k0;
      it.kend = static_cast<int>(min(static_cast<int64_t>(len) - k0, (p_hi - p_lo) * kBK));
      it.nvalid = a->n_head;
      it.qrow0 = static_cast<int64_t>(bb) * a->n_head;
      it.slot0 = static_cast<int64_t>(bb + c) * a->n_head;
      it.n_tiles = static_cast<int>(p_hi - p_lo);
      return true;
    }
    return false;
  }
};

// Walks this cluster's tiles in order across its items.
template <bool kDecode>
struct TileCursor {
  ItemIter<kDecode> iter;
  Item it;
  int t;              // tile within the item
  bool more;
  MLA_DEVINL void skip_empty() {
    while (more && t >= it.n_tiles) {
      more = iter.next(it);
      t = 0;
    }
  }
  MLA_DEVINL void init(const AttnTcArgs& args, int cluster, int clusters, const DecodeStart* ds) {
    iter.init(args, cluster, clusters, ds);
    t = 0;
    more = iter.next(it);
    skip_empty();
  }
  MLA_DEVINL bool valid() const { return more; }
  MLA_DEVINL void next() { ++t; skip_empty(); }
};

// bf16 -> fp16 in place of this thread's share (thread ct of kConvThreads) of
// a landed latent tile.  A 16-byte unit holds 8 consecutive values of one key,
// so the swizzle does not matter; exact over fp16's normal range.  (A value
// too large for fp16 becomes inf here; every key of a tile goes through P.V,
// so it makes the piece's output infinite or NaN, which the epilogue checks:
// a check per value here would lengthen the tile's conversion step.)
MLA_DEVINL void convert_share(uint8_t* stage, int ct) {
  constexpr int kUnits = kLatStage / 16;
  constexpr int kPer = (kUnits + kConvThreads - 1) / kConvThreads;
  uint4* st = reinterpret_cast<uint4*>(stage);
  uint4 v[kPer];
#pragma unroll
  for (int m = 0; m < kPer; ++m)
    if (ct + m * kConvThreads < kUnits) v[m] = st[ct + m * kConvThreads];
#pragma unroll
  for (int m = 0; m < kPer; ++m)
    if (ct + m * kConvThreads < kUnits) st[ct + m * kConvThreads] = bf16x8_to_f16x8(v[m]);
}

// Store 64 bytes of each of a warp's 32 rows (lane = row, `w` = the row's four
// 16-byte units) to dst_row0 + row * row_stride (bytes): through the warp's
// 2 KB staging slice, so that each store instruction writes 8 rows x 64
// contiguous bytes.  Units are XOR-swizzled by row pair (no bank conflicts).
// Rows >= nrows are not stored.  Whole warp.
MLA_DEVINL void store_rows64(uint8_t* stg, int lane, const uint4 (&w)[4], uint8_t* dst_row0, int64_t row_stride,
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

// bf16 decode: before waiting for tile u's stage, each CTA asks for the whole
// rows of tile u (both CTAs' parts) as one contiguous L2 prefetch, so the
// rows are on their way while the stage drains.  Measured against the TMA
// loads alone (B=32 decode): 7% faster; prefetching 1, 2, 4 or 8 tiles ahead
// instead, with or without an evict-last hint, gave back most or all of it.
MLA_DEVINL void prefetch_rows_l2(const AttnTcArgs& a, int64_t row0, int64_t nrows) {
  const int64_t rows = min(nrows, a.n_rows - row0);
  if (rows > 0)
    tc::prefetch_l2(static_cast<const uint16_t*>(a.kv) + row0 * kRow, static_cast<uint32_t>(rows * kRow * 2));
}

// q8_0 decode: L2 prefetch of the rows kPrefetchTiles tiles ahead of the
// producers' loads.
constexpr int kPrefetchTiles = 8;

// q8_0 tiles ahead, by one warp (`lane` its lane): the codes as one bulk L2
// prefetch, and the scales of the tile's rows in each of the 18 scale blocks
// (lanes 0..17: the first and the last cache line of the block's run).
MLA_DEVINL void prefetch_q8_tile(const AttnTcArgs& a, const TileCursor<true>& c, int lane) {
  const int64_t row0 = c.it.key_base + static_cast<int64_t>(c.t) * kBK;
  const int64_t rows = min(static_cast<int64_t>(kBK), a.n_rows - row0);
  if (rows <= 0) return;
  if (lane == 0) tc::prefetch_l2(a.kv_q + row0 * kRow, static_cast<uint32_t>(rows * kRow));
  if (lane < kQ8Blocks) {
    const uint16_t* d = a.kv_d + static_cast<int64_t>(lane) * a.ld_d + row0;
    tc::prefetch_line_l2(d);
    tc::prefetch_line_l2(d + rows - 1);
  }
}

// The q8_0 decode's producer warps (thread pt of kProducerThreads): every
// tile of this cluster's range into the latent and RoPE rings.  Tile u counts
// this cluster's tiles across items.
MLA_DEVINL void run_q8_producer(const AttnTcArgs& a, Bars& B, uint8_t* sLat, uint8_t* sRope, int rank, int pt,
                                int first, int stride) {
  using P = Q8Producer;
  TileCursor<true> cur;
  cur.init(a, first, stride, &B.ds);
  if (!cur.valid()) return;
  // One warp keeps the rows of the tiles kPrefetchTiles ahead on their way into
  // L2: the last one, which has a unit fewer per tile than the first.
  TileCursor<true> ahead = cur;
  const bool pf = pt >= kProducerThreads - 32 && rank == 0;
  const int pl = pt - (kProducerThreads - 32);
  for (int d = 0; d < kPrefetchTiles && ahead.valid(); ++d) {
    if (pf) prefetch_q8_tile(a, ahead, pl);
    ahead.next();
  }
  P::Plan plan;
  P::plan(plan, rank, pt);
  P x;
  uint32_t dmax = 0;                          // largest |scale| bit pattern (fp16 range check)
  x.load(a, plan, pt, cur.it.key_base, cur.t * kBK, cur.it.kend);
  cur.next();
  // One register set: tile u+1's loads go out as soon as tile u is stored and
  // are in flight while the producer waits for tile u+1's stage.  (Two sets,
  // tile u+1 loaded before tile u's stage wait and moved into place after its
  // store, cost 30 register moves per tile and 15% of the q8_0 decode; a
  // second copy of the loop instead of the moves misses the instruction cache.)
#pragma unroll 1
  for (int u = 0;; ++u) {
    if (ahead.valid()) {
      if (pf) prefetch_q8_tile(a, ahead, pl);
      ahead.next();
    }
    const int ls = u % kLatStages, rs = u % kRopeStages;
    if (u >= kLatStages && !mbar_wait_bounded(&B.lat_empty[ls], ((u / kLatStages) - 1) & 1, a.wait_us, a.err))
      break;
    if (u >= kRopeStages && !mbar_wait_bounded(&B.rope_empty[rs], ((u / kRopeStages) - 1) & 1, a.wait_us, a.err))
      break;
    x.store(plan, sLat + ls * kLatStage, sRope + rs * kRopeChunk, pt);
#pragma unroll
    for (int t = 0; t < P::NU; ++t) dmax = max(dmax, x.d[t] & 0x7FFFu);
    tc::fence_proxy_async();
    mbar_arrive(&B.lat_full[ls]);
    if (!cur.valid()) break;
    x.load(a, plan, pt, cur.it.key_base, cur.t * kBK, cur.it.kend);
    cur.next();
  }
  if (f16_scale_overflows(dmax)) record_error(a.err, MLA_ERR_RANGE);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// kDecode = false: prefill from the fp16 staging copy (kQ8 unused).
template <bool kQ8, bool kDecode>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(max_regs(kQ8, kDecode))
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_cache, const __grid_constant__ CUtensorMap tm_rope,
                   AttnTcArgs a) {
  // fp16 RoPE operands (prefill staging copy, q8_0 decode) or bf16 (bf16 decode).
  constexpr bool kRopeF16 = kQ8 || !kDecode;
  constexpr int kMmaWarp = mma_warp(kQ8, kDecode);
  constexpr bool kEpi = epi_warps(kQ8, kDecode) > 0;
  constexpr int kLoaderWarp = loader_warp(kQ8, kDecode);
  constexpr int kSoftmaxWarps = softmax_warps(kQ8, kDecode);
  constexpr int kKpt = kBK / kTpr;          // keys of each tile per softmax thread: 32 or 16
  constexpr int kUpt = kKpt / 8;            // the same as 16-byte units of fp16: 4 or 2
  constexpr int kOpt = 256 / kTpr;          // output columns (of this CTA's half) per thread: 128 or 64
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so that
  // accesses through it stay shared-memory (not generic) accesses.
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQr = sm;
  uint8_t* sLat = sm + kOffLat;
  uint8_t* sRope = sm + kOffRope;
  uint8_t* sP = sm + kOffP;
  uint8_t* sX = sm + kOffX;
  uint8_t* sStg = sm + kOffStg;
  float* aux_lrow = reinterpret_cast<float*>(sm + kOffAux);     // [4][128] row sums for the epilogue warps
  Bars& B = *reinterpret_cast<Bars*>(sm + kOffBar);

  const uint32_t rank = tc::cluster_ctarank(), peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.n_head;
  const int first = static_cast<int>(blockIdx.x >> 1);      // this cluster's first item index
  const int stride = static_cast<int>(gridDim.x >> 1);      // clusters

  // ---- setup -----------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int i = 0; i < kLatStages; ++i) {
      mbar_init(&B.lat_full[i], !kDecode ? 1 : (kQ8 ? kProducerThreads : kConvThreads));   // converters + epilogue warps
      mbar_init(&B.lat_tma[i], 1);
      mbar_init(&B.lat_empty[i], 1);
    }
    for (int i = 0; i < kRopeStages; ++i) {
      mbar_init(&B.rope_full[i], 1);
      mbar_init(&B.rope_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_free[i], kSoftmaxWarps * 32);
      mbar_init(&B.x_full[i], 1);
      mbar_init(&B.x_empty[i], kSoftmaxWarps);
    }
    mbar_init(&B.p_full[0], kSoftmaxWarps * 32);
    mbar_init(&B.p_full[1], kSoftmaxWarps * 32);
    mbar_init(&B.pv_done[0], 1);
    mbar_init(&B.pv_done[1], 1);
    mbar_init(&B.q_ready, kEpi ? 128 : kSoftmaxWarps * 32);
    mbar_init(&B.o_free, kEpi ? 128 : kSoftmaxWarps * 32);
    mbar_init(&B.q_free, 1);
    mbar_init(&B.o_ready, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&B.l_ready[i], kSoftmaxWarps * 32);
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&B.tmem, 512);
    tc::tmem_relinquish();
  }
  if constexpr (kDecode) {
    if (warp == 1) {
      const DecodeStart ds = decode_start(a, first, stride, lane);
      if (lane == 0) {
        B.ds = ds;
        // The first item's queries on their way into L2 (its Q load is the
        // longest step before the first tile).
        if (ds.b < a.n_seq) {
          const int64_t r0 = static_cast<int64_t>(ds.b) * a.n_head;
          if (rank == 0)
            tc::prefetch_l2(static_cast<const uint16_t*>(a.q_lat) + r0 * kLatent, static_cast<uint32_t>(a.n_head) * kLatent * 2);
          else
            tc::prefetch_l2(static_cast<const uint16_t*>(a.q_pe) + r0 * kRope, static_cast<uint32_t>(a.n_head) * kRope * 2);
        }
      }
    }
  }
  tc::fence_before_sync();
  tc::cluster_sync();                 // peer barriers initialised before any remote arrival
  tc::fence_after_sync();
  const uint32_t tmem = B.tmem;
  // Decode: the combine kernel, launched as a programmatic dependent, may be
  // scheduled now; it waits for this grid's completion before reading.
  if constexpr (kDecode) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp < kSoftmaxWarps) {
    // ======================= softmax / exchange / epilogue =====================
    // Warp w serves the 16 TMEM lanes (query rows) 32 (w % 4) + 16 (w / 4) ..
    // +15; lanes l and l + 16 share row l % 16: thread hh = l / 16 takes keys
    // [kKpt*hh, kKpt*hh + kKpt) of every tile and output columns
    // [kOpt*hh, kOpt*hh + kOpt) of this CTA's half.
    static_assert(kTpr == 2, "two threads per row: lanes l and l + 16 of one warp");
    const int q4 = warp & 3;                    // TMEM lane quadrant
    const int hh = lane >> 4;                   // which half of the row's keys and output columns
    const int i = q4 * 32 + (warp >> 2) * 16 + (lane & 15);   // query row == TMEM lane
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32 + (warp >> 2) * 16) << 16;   // the warp's 16 lanes
    const float c2 = a.scale_log2;              // raw score -> log2 units
    const uint32_t peer_x = tc::mapa(smem_u32(sX), peer);
    const uint32_t peer_xfull = tc::mapa(smem_u32(&B.x_full[0]), peer);
    const uint32_t peer_xempty = tc::mapa(smem_u32(&B.x_empty[0]), peer);
    // A wait that gave up makes the warp "dead" (every wait is warp-wide, so
    // the whole warp): it skips every later wait, tensor-memory access and
    // arrival.
    bool dead = false;
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
      if (!dead) dead = !wait_all(bar, parity, a);
    };

    // Read this thread's kKpt partial scores of tile u (counted across
    // items), free the score buffer and keep them as fp16 pairs.  `ready`: an
    // earlier non-blocking check already saw the phase complete.
    auto fetch = [&](int u, uint32_t (&own)[kKpt / 2], bool ready) {
      const int sb = u & 1;
      if (!ready) wait_ok(&B.s_full[sb], (u >> 1) & 1);
      if (dead) return;
      tc::fence_after_sync();
      uint32_t r[kKpt];
      tc::tmem_ld16x2<kKpt>(tmem + lanes + kTmS + sb * 64, r);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      mbar_arrive(&B.s_free[sb]);
#pragma unroll
      for (int k = 0; k < kKpt / 2; ++k) own[k] = pack_f16x2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
    };

    // Send tile u's fp16 partials to the peer, once it has finished with the
    // exchange buffer's previous contents (tile u-2).
    auto send = [&](int u, const uint32_t (&own)[kKpt / 2]) {
      const int sb = u & 1;
      if (u >= 2 && !dead)
        dead = !__all_sync(0xffffffffu, tc::mbar_wait_cluster_bounded(&B.x_empty[sb], ((u >> 1) - 1) & 1, a.wait_us,
                                                                      a.err));
      if (dead) return;
#pragma unroll
      for (int g = 0; g < kUpt; ++g)
        tc::st_async_v4(peer_x + sb * kXBytes + ((kUpt * hh + g) * kRows + i) * 16,
                        make_uint4(own[4 * g], own[4 * g + 1], own[4 * g + 2], own[4 * g + 3]), peer_xfull + sb * 8);
      if (threadIdx.x == 0) mbar_arrive_expect_tx(&B.x_full[sb], kXBytes);
    };

    uint32_t own[kKpt / 2], nxt[kKpt / 2];
    uint32_t qrun = 0;                          // q_pe converted here (q8_0 decode): fp16 range check
    bool score_range = false;                   // a row maximum became infinite or NaN
    int u0 = 0;                                 // this item's first tile, counted across items
    int k = 0;                                  // items done
    ItemIter<kDecode> items;
    items.init(a, first, stride, &B.ds);
    Item it;
#pragma unroll 1
    while (items.next(it)) {
      const bool rvalid = i < it.nvalid;
      const int64_t qrow = it.qrow0 + i;
      int lim;                                  // last visible key index (item-relative)
      if constexpr (kDecode) {
        lim = it.kend - 1;
      } else {
        lim = rvalid ? a.q_pos0 + static_cast<int>(qrow / H) : it.kend - 1;
      }
      // Decode: Q latent half -> TMEM (fp16 A operand), this thread: dims
      // [kOpt*hh, kOpt*hh + kOpt) of the half.  The previous item's score MMAs
      // have all completed (this thread read every one of their results), so
      // the Q region and the RoPE query tile are free.  (Prefill: the epilogue
      // warps do this.)
      if constexpr (!kEpi) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_lat) + qrow * kLatent +
                                                          256 * rank + kOpt * hh);
        // All loads first (one round trip), then the stores.
        uint32_t r[kOpt / 64][32];
        uint4 qpe[4 / kTpr];
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_pe) + qrow * kRope);
#pragma unroll
        for (int c = 0; c < kOpt / 64; ++c)
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = rvalid ? __ldg(src + c * 8 + v) : make_uint4(0, 0, 0, 0);
            r[c][4 * v] = x.x; r[c][4 * v + 1] = x.y; r[c][4 * v + 2] = x.z; r[c][4 * v + 3] = x.w;
          }
#pragma unroll
        for (int v = 0; v < 4 / kTpr; ++v)      // this CTA's 32 RoPE dims: units 4 rank .. 4 rank + 3
          qpe[v] = rvalid ? __ldg(qp + 4 * rank + (4 / kTpr) * hh + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < kOpt / 64; ++c) tc::tmem_st16x2<kOpt / 2>(tmem + lanes + kTmQ + 32 * c, r[c]);
        tc::tmem_st_wait();
        {                                       // RoPE query part -> smem (bf16 as is, or fp16)
#pragma unroll
          for (int v = 0; v < 4 / kTpr; ++v) {
            if (kRopeF16) {
              qrun = bf16x2_absmax(bf16x2_absmax(qrun, qpe[v].x), qpe[v].y);
              qrun = bf16x2_absmax(bf16x2_absmax(qrun, qpe[v].z), qpe[v].w);
            }
            st_unit64(sQr, i, (4 / kTpr) * hh + v, kRopeF16 ? bf16x8_to_f16x8(qpe[v]) : qpe[v]);
          }
          tc::fence_proxy_async();
        }
        tc::fence_before_sync();
        mbar_arrive(&B.q_ready);
      }

      float m_run = -INFINITY, l_h = 0.f;
      const int n = it.n_tiles;

      // Softmax of item tile t (tile u = u0 + t overall) from the two fp16 partials.
      auto process = [&](int t, const uint32_t (&own_t)[kKpt / 2], bool ready) {
        const int u = u0 + t, xb = u & 1;
        if (!dead && !ready)
          dead = !__all_sync(0xffffffffu, tc::mbar_wait_cluster_bounded(&B.x_full[xb], (u >> 1) & 1, a.wait_us, a.err));
        float s[kKpt];
#pragma unroll
        for (int g = 0; g < kUpt; ++g) {
          const uint4 pv = *reinterpret_cast<const uint4*>(sX + xb * kXBytes + ((kUpt * hh + g) * kRows + i) * 16);
          const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = f16x2_to_f32(own_t[4 * g + e]);
            s[8 * g + 2 * e] = tc::add_f16lo_f32(pw[e], x.x);
            s[8 * g + 2 * e + 1] = tc::add_f16hi_f32(pw[e], x.y);
          }
        }
        const int k0 = t * kBK + kKpt * hh;
        if (k0 + kKpt - 1 > lim) {
#pragma unroll
          for (int e = 0; e < kKpt; ++e)
            if (k0 + e > lim) s[e] = -INFINITY;
        }
        // Row maximum of this share as a tree (short dependency chain).
        float mx[kKpt / 2];
#pragma unroll
        for (int e = 0; e < kKpt / 2; ++e) mx[e] = fmaxf(s[2 * e], s[2 * e + 1]);
#pragma unroll
        for (int w = kKpt / 4; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
        const float mown = mx[0] * c2;
        const float mrow = fmaxf(mown, __shfl_xor_sync(0xffffffffu, mown, 16));
        // Lazy rescale: only when the row max grew by more than the threshold (always on the first tile).
        float alpha = 1.f;
        if (mrow > m_run + kRescaleThreshold) {
          alpha = tc::exp2_approx(m_run - mrow);
          m_run = mrow;
          l_h *= alpha;
        }
        // p = 2^(s*c - m) on packed halves; the row sum stays in fp32.
        uint32_t pk[kKpt / 2];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};      // four independent partial sums
#pragma unroll
        for (int e = 0; e < kKpt / 2; ++e) {
          pk[e] = tc::exp2_approx_f16x2(pack_f16x2(fmaf(s[2 * e], c2, -m_run), fmaf(s[2 * e + 1], c2, -m_run)));
          ls[e & 3] = tc::add_f16hi_f32(pk[e], tc::add_f16lo_f32(pk[e], ls[e & 3]));
        }
        l_h += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P buffer u&1 is free once P.V of tile u-2 has finished; O is stable for
        // a rescale once P.V of tile u-1 has (waited for only when a rescale is
        // due).  (A new item's O restarts with its first P.V: nothing to
        // rescale.)  Each pv_done barrier's phases are followed one by one.
        if (u >= 2) wait_ok(&B.pv_done[u & 1], ((u >> 1) - 1) & 1);
        if (!dead && t >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
          wait_ok(&B.pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1);
          if (!dead) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < kOpt / 32; ++c) {
              uint32_t o[32];
              const uint32_t col = tmem + lanes + kTmO + 32 * c;
              tc::tmem_ld16x2<kOpt>(col, o);
              tc::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tc::tmem_st16x2<kOpt>(col, o);
            }
            tc::tmem_st_wait();
          }
        }
        if (dead) return;
#pragma unroll
        for (int g = 0; g < kUpt; ++g)
          st_unit(sP + (u & 1) * kPBytes, i, kUpt * hh + g, make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]));
        tc::fence_proxy_async();
        tc::fence_before_sync();
        mbar_arrive(&B.p_full[u & 1]);
        // This warp has long finished reading exchange buffer xb (every value read
        // from it fed the scores above): tell the peer it may refill it.  A relaxed
        // arrival suffices and avoids the ~1.4k-cycle cluster-scope release.
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote_relaxed(peer_xempty + xb * 8);
      };

      // One loop body (a register copy per tile keeps the hot code small).
      if constexpr (kDecode) {
        // Decode: the first fetch in the loop too (step t = -1), so that
        // fetch, send and process each have one call site: the decode kernel
        // is instruction-fetch bound.
#pragma unroll 1
        for (int t = -1; t < n; ++t) {
          const int u = u0 + t;
          bool s_ready = false, x_ready = false;
          if (t >= 0) {
            const bool s_test = mbar_test(&B.s_full[(u + 1) & 1], ((u + 1) >> 1) & 1);
            const bool x_test = tc::mbar_test_cluster(&B.x_full[u & 1], (u >> 1) & 1);
            s_ready = __all_sync(0xffffffffu, s_test) && t + 1 < n;
            x_ready = __all_sync(0xffffffffu, x_test);
          }
          if (t + 1 < n) {
            fetch(u + 1, nxt, s_ready);
            send(u + 1, nxt);
          }
          if (t >= 0) process(t, own, x_ready);
#pragma unroll
          for (int e = 0; e < kKpt / 2; ++e) own[e] = nxt[e];
        }
      } else {
        fetch(u0, own, false);
        send(u0, own);
#pragma unroll 1
        for (int t = 0; t < n; ++t) {
          const int u = u0 + t;
          // Check both phases this tile needs first, so that their latencies
          // overlap; a phase not yet complete is waited for where it is needed.
          const bool s_test = mbar_test(&B.s_full[(u + 1) & 1], ((u + 1) >> 1) & 1);
          const bool x_test = tc::mbar_test_cluster(&B.x_full[u & 1], (u >> 1) & 1);
          const bool s_ready = __all_sync(0xffffffffu, s_test) && t + 1 < n;
          const bool x_ready = __all_sync(0xffffffffu, x_test);
          if (t + 1 < n) {
            fetch(u + 1, nxt, s_ready);
            send(u + 1, nxt);
          }
          process(t, own, x_ready);
#pragma unroll
          for (int e = 0; e < kKpt / 2; ++e) own[e] = nxt[e];
        }
      }
      // ---- end of item -----------------------------------------------------------
      // A partial score past fp16's range makes the row maximum infinite (or NaN).
      if (rvalid && !dead && !(m_run < INFINITY)) score_range = true;
      if constexpr (kEpi) {
        // Prefill: hand the row sums to the epilogue warps and go on.
        const float l_row = l_h + __shfl_xor_sync(0xffffffffu, l_h, 16);   // a + b == b + a: the same in both threads
        if (hh == 0) aux_lrow[(k & 3) * kRows + i] = l_row;
        if (rank == 0 && hh == 0 && rvalid) {
          if constexpr (kDecode) {
            a.ws_ml[2 * (it.slot0 + i)] = m_run;
            a.ws_ml[2 * (it.slot0 + i) + 1] = l_row;
          } else if (a.lse != nullptr) {
            a.lse[qrow] = (m_run + log2f(l_row)) * kLn2;
          }
        }
        mbar_arrive(&B.l_ready[k & 3]);
      } else {
        // Decode: O / l -> the fp32 partials, with the running max and sum.
        wait_ok(&B.pv_done[(u0 + n - 1) & 1], ((u0 + n - 1) >> 1) & 1);
        if (!dead) {
          tc::fence_after_sync();
          const float l_row = l_h + __shfl_xor_sync(0xffffffffu, l_h, 16);
          const float inv = 1.f / l_row;
#pragma unroll 1
          for (int c = 0; c < kOpt / 32; ++c) {
            uint32_t o[32];
            tc::tmem_ld16x2<kOpt>(tmem + lanes + kTmO + 32 * c, o);
            tc::tmem_ld_wait();
            if (!rvalid) continue;
            const int col = 256 * static_cast<int>(rank) + kOpt * hh + 32 * c;
            uint4* dst = reinterpret_cast<uint4*>(a.ws_o + (it.slot0 + i) * kLatent + col);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_uint4(__float_as_uint(__uint_as_float(o[4 * v]) * inv),
                                  __float_as_uint(__uint_as_float(o[4 * v + 1]) * inv),
                                  __float_as_uint(__uint_as_float(o[4 * v + 2]) * inv),
                                  __float_as_uint(__uint_as_float(o[4 * v + 3]) * inv));
          }
          if (rank == 0 && hh == 0 && rvalid) {
            a.ws_ml[2 * (it.slot0 + i)] = m_run;
            a.ws_ml[2 * (it.slot0 + i) + 1] = l_row;
          }
          // O has been read: the next item's first P.V may overwrite it.
          tc::fence_before_sync();
          mbar_arrive(&B.o_free);
        }
      }
      u0 += n;
      ++k;
    }
    if (score_range || bf16x2_absmax_overflows(qrun)) record_error(a.err, MLA_ERR_RANGE);
  } else if (kEpi && (warp < kLoaderWarp || (kDecode && !kQ8 && warp > kLoaderWarp && warp < kMmaWarp))) {
    if constexpr (!kDecode) {
    // ======================= Q loading and epilogue (prefill) ==================
    // Warp 8+q serves TMEM lane quadrant q: thread = query row i, the whole
    // 256-column half of the row.  Per item k: once item k-1's last score MMA
    // has completed (q_free), Q of item k -> TMEM (and Q_pe -> smem on rank 0),
    // then q_ready; then, once item k-1's last P.V has completed (o_ready) and
    // its row sums are in (l_ready), O / l -> o_lat and o_free.
    const int q4 = warp & 3;
    const int i = q4 * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    bool ok = true;
    auto epilogue = [&](const Item& pv, int kk) {
      ok = ok && wait_all(&B.o_ready, kk & 1, a);
      ok = ok && wait_all(&B.l_ready[kk & 3], (kk >> 2) & 1, a);
      if (!ok) return;
      tc::fence_after_sync();
      const float inv = 1.f / aux_lrow[(kk & 3) * kRows + i];
      // This warp's 32 rows, 32 columns (64 B of fp16) per step, through its staging slice.
      uint8_t* dst = reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(a.o_lat) + (pv.qrow0 + q4 * 32) * kLatent +
                                                256 * rank);
      uint8_t* stg = sStg + (warp - kSoftmaxWarps) * 2048;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lanes + kTmO + 32 * c, o);
        tc::tmem_ld_wait();
        uint4 w[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          w[v].x = pack_f16x2(__uint_as_float(o[8 * v]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
          w[v].y = pack_f16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
          w[v].z = pack_f16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
          w[v].w = pack_f16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
        }
        store_rows64(stg, lane, w, dst + c * 64, kLatent * 2, pv.nvalid - q4 * 32);
      }
      tc::fence_before_sync();
      mbar_arrive(&B.o_free);
    };
    Item prev;
    int k = 0;
    uint32_t qrun = 0;                          // q_pe values converted to fp16: range check
#pragma unroll 1
    for (int rnd = 0; ok && rnd * stride < a.n_items; ++rnd) {
      const int idx = round_item(first, stride, rnd);
      if (idx >= a.n_items) continue;
      const Item it = prefill_item(a, idx);
      if (it.n_tiles == 0) continue;
      if (k > 0) ok = wait_all(&B.q_free, (k - 1) & 1, a);
      if (!ok) break;
      tc::fence_after_sync();
      const bool rvalid = i < it.nvalid;
      const int64_t qrow = it.qrow0 + i;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_lat) + qrow * kLatent +
                                                        256 * rank);
#pragma unroll 1
      for (int h2 = 0; h2 < 2; ++h2) {          // two rounds of 16 loads (128 dims each)
        uint32_t r[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = rvalid ? __ldg(src + (2 * h2 + c) * 8 + v) : make_uint4(0, 0, 0, 0);
            r[c][4 * v] = x.x; r[c][4 * v + 1] = x.y; r[c][4 * v + 2] = x.z; r[c][4 * v + 3] = x.w;
          }
#pragma unroll
        for (int c = 0; c < 2; ++c) tc::tmem_st32(tmem + lanes + kTmQ + 32 * (2 * h2 + c), r[c]);
      }
      tc::tmem_st_wait();
      {                                         // this CTA's 32 RoPE query dims -> smem, fp16
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_pe) + qrow * kRope) +
                          4 * rank;
        uint4 qpe[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) qpe[v] = rvalid ? __ldg(qp + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          qrun = bf16x2_absmax(bf16x2_absmax(qrun, qpe[v].x), qpe[v].y);
          qrun = bf16x2_absmax(bf16x2_absmax(qrun, qpe[v].z), qpe[v].w);
          st_unit64(sQr, i, v, bf16x8_to_f16x8(qpe[v]));
        }
        tc::fence_proxy_async();
      }
      tc::fence_before_sync();
      mbar_arrive(&B.q_ready);
      // Bring the next item's queries into L2 meanwhile.
      if (lane == 0 && q4 == 0 && (rnd + 1) * stride < a.n_items) {
        const int nidx = round_item(first, stride, rnd + 1);
        if (nidx < a.n_items) {
          const Item nx = prefill_item(a, nidx);
          if (rank == 0)
            tc::prefetch_l2(static_cast<const uint16_t*>(a.q_lat) + nx.qrow0 * kLatent,
                            static_cast<uint32_t>(nx.nvalid) * kLatent * 2);
          else
            tc::prefetch_l2(static_cast<const uint16_t*>(a.q_pe) + nx.qrow0 * kRope,
                            static_cast<uint32_t>(nx.nvalid) * kRope * 2);
        }
      }
      if (k > 0) epilogue(prev, k - 1);
      prev = it;
      ++k;
    }
    if (ok && k > 0) epilogue(prev, k - 1);
    if (bf16x2_absmax_overflows(qrun)) record_error(a.err, MLA_ERR_RANGE);
    } else {
    // ============ Q loading, tile conversion and epilogue (bf16 decode) ========
    // As for prefill, per item (piece): Q once the previous item's last score
    // MMA has completed, the fp32 partial once its last P.V has.  In between,
    // these warps convert their share of every tile to fp16 (see
    // convert_share): in decode they have little else to do.  (A separate
    // copy of the prefill code: sharing it cost the prefill kernel ~10%.)
    // The two converter warps after the loader warp run the same loop without
    // the Q and output steps (one copy of the hot code: the decode kernel is
    // instruction-fetch bound).
    const bool epi = warp < kLoaderWarp;
    const int q4 = warp & 3;
    const int i = q4 * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    float amax = 0.f;                           // |O| of the partials (fp16 range check)
    bool ok = true;
    auto epilogue = [&](const Item& pv, int kk) {
      ok = ok && wait_all(&B.o_ready, kk & 1, a);
      ok = ok && wait_all(&B.l_ready[kk & 3], (kk >> 2) & 1, a);
      if (!ok) return;
      tc::fence_after_sync();
      const float inv = 1.f / aux_lrow[(kk & 3) * kRows + i];
      // fp32 partial of this piece, normalised by its own sum: this warp's 32
      // rows, 16 columns (64 B) per step, through its staging slice.
      uint8_t* dst = reinterpret_cast<uint8_t*>(a.ws_o + (pv.slot0 + q4 * 32) * kLatent + 256 * rank);
      uint8_t* stg = sStg + (warp - kSoftmaxWarps) * 2048;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lanes + kTmO + 32 * c, o);
        tc::tmem_ld_wait();
        if (i < pv.nvalid) {                    // a cache value past fp16 made O infinite or NaN
#pragma unroll
          for (int e = 0; e < 32; ++e) amax = f32_absmax(amax, __uint_as_float(o[e]));
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint4 w[4];
#pragma unroll
          for (int v = 0; v < 4; ++v)
            w[v] = make_uint4(__float_as_uint(__uint_as_float(o[16 * h2 + 4 * v]) * inv),
                              __float_as_uint(__uint_as_float(o[16 * h2 + 4 * v + 1]) * inv),
                              __float_as_uint(__uint_as_float(o[16 * h2 + 4 * v + 2]) * inv),
                              __float_as_uint(__uint_as_float(o[16 * h2 + 4 * v + 3]) * inv));
          store_rows64(stg, lane, w, dst + (32 * c + 16 * h2) * 4, kLatent * 4, pv.nvalid - q4 * 32);
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&B.o_free);
    };
    // Q of item k -> TMEM / smem, once item k-1's last score MMA has completed;
    // `peek` is the item iterator positioned after `it` (for the L2 prefetch).
    auto q_load = [&](const Item& it, int k, const ItemIter<kDecode>& peek_from) {
      if (k > 0) ok = ok && wait_all(&B.q_free, (k - 1) & 1, a);
      if (!ok) return;
      tc::fence_after_sync();
      const bool rvalid = i < it.nvalid;
      const int64_t qrow = it.qrow0 + i;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_lat) + qrow * kLatent +
                                                        256 * rank);
#pragma unroll 1
      for (int h2 = 0; h2 < 2; ++h2) {          // two rounds of 16 loads (128 dims each)
        uint32_t r[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = rvalid ? __ldg(src + (2 * h2 + c) * 8 + v) : make_uint4(0, 0, 0, 0);
            r[c][4 * v] = x.x; r[c][4 * v + 1] = x.y; r[c][4 * v + 2] = x.z; r[c][4 * v + 3] = x.w;
          }
#pragma unroll
        for (int c = 0; c < 2; ++c) tc::tmem_st32(tmem + lanes + kTmQ + 32 * (2 * h2 + c), r[c]);
      }
      tc::tmem_st_wait();
      {                                         // this CTA's 32 RoPE query dims -> smem (fp16, or bf16 for the bf16 decode)
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_pe) + qrow * kRope) +
                          4 * rank;
        uint4 qpe[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) qpe[v] = rvalid ? __ldg(qp + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int v = 0; v < 4; ++v) st_unit64(sQr, i, v, kRopeF16 ? bf16x8_to_f16x8(qpe[v]) : qpe[v]);
        tc::fence_proxy_async();
      }
      tc::fence_before_sync();
      mbar_arrive(&B.q_ready);
      // Bring the next item's queries into L2 meanwhile.
      if (lane == 0 && q4 == 0) {
        ItemIter<kDecode> peek = peek_from;
        Item nx;
        if (peek.next(nx)) {
          if (rank == 0)
            tc::prefetch_l2(static_cast<const uint16_t*>(a.q_lat) + nx.qrow0 * kLatent,
                            static_cast<uint32_t>(nx.nvalid) * kLatent * 2);
          else
            tc::prefetch_l2(static_cast<const uint16_t*>(a.q_pe) + nx.qrow0 * kRope,
                            static_cast<uint32_t>(nx.nvalid) * kRope * 2);
        }
      }
    };
    Item prev;
    int k = 0;
    {
      // Conversion share 64 + 32 q4 + lane (epilogue warps) or 32 (w - 1) +
      // lane (converter warp w after the loader warp); at an item's first
      // tile, its Q first, then the tile, then the previous item's epilogue
      // (its P.V has to finish anyway before the new item's first P.V may
      // start).
      const int ct = epi ? 64 + q4 * 32 + lane : (warp - kLoaderWarp - 1) * 32 + lane;
      TileCursor<kDecode> cur;
      cur.init(a, first, stride, &B.ds);
      // One pass past the last tile writes the last item's output (one call
      // site of the epilogue: the decode kernel is instruction-fetch bound).
#pragma unroll 1
      for (int u = 0; ok; ++u, cur.next()) {
        const bool has = cur.valid();
        const bool first_tile = epi && has && cur.t == 0;
        if (first_tile) q_load(cur.it, k, cur.iter);
        if (has) {
          const int ls = u % kLatStages;
          ok = ok && wait_all(&B.lat_tma[ls], (u / kLatStages) & 1, a);
          if (!ok) break;
          convert_share(sLat + ls * kLatStage, ct);
          tc::fence_proxy_async();
          mbar_arrive(&B.lat_full[ls]);
        }
        if (!epi && !has) break;
        if (first_tile || !has) {
          if (k > 0) epilogue(prev, k - 1);
          if (!has) break;
          prev = cur.it;
          ++k;
        }
      }
      if (!(amax < INFINITY)) record_error(a.err, MLA_ERR_RANGE);   // O = l x o_lat may pass 65504: finiteness only
    }
    }
  } else if (warp < kMmaWarp) {
    // ============================ loader =======================================
    const int pt = threadIdx.x - kLoaderWarp * 32;
    if constexpr (!kDecode || !kQ8) {
      if (pt == 0) {
        // One thread: each tile's four 64-dim latent chunks of this CTA's half
        // and its 32 RoPE dims by TMA, as soon as the stage is free.  Prefill
        // reads the fp16 staging copy (the tile is ready on arrival); the bf16
        // decode reads the cache itself and the tile is converted before the
        // MMAs may read it.
        uint64_t* landed = kDecode ? B.lat_tma : B.lat_full;
        TileCursor<kDecode> cur;
        cur.init(a, first, stride, &B.ds);
        for (int u = 0; cur.valid(); ++u, cur.next()) {
          const int ls = u % kLatStages, rs = u % kRopeStages;
          const int key = static_cast<int>(cur.it.key_base) + cur.t * kBK;
          if (kDecode) prefetch_rows_l2(a, key, min(kBK, cur.it.kend - cur.t * kBK));
          if (u >= kLatStages && !mbar_wait_bounded(&B.lat_empty[ls], ((u / kLatStages) - 1) & 1, a.wait_us, a.err))
            break;
          mbar_arrive_expect_tx(&landed[ls], kLatStage);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tc::tma_load_3d(sLat + ls * kLatStage + c * kChunk, &tm_cache, &landed[ls], 256 * rank + 64 * c, key, 0);
          if (u >= kRopeStages &&
              !mbar_wait_bounded(&B.rope_empty[rs], ((u / kRopeStages) - 1) & 1, a.wait_us, a.err))
            break;
          mbar_arrive_expect_tx(&B.rope_full[rs], kRopeChunk);   // this CTA's 32 RoPE dims
          tc::tma_load_3d(sRope + rs * kRopeChunk, &tm_rope, &B.rope_full[rs], kLatent + kRopeHalf * rank, key, 0);
        }
      }
      // (bf16 decode: the two converter warps after this one run the
      // epilogue warps' conversion loop.)
    } else {
      run_q8_producer(a, B, sLat, sRope, static_cast<int>(rank), pt, first, stride);
    }
  } else {
    // ============================== MMA issue ==================================
    // The whole warp runs this loop (see mma_ss_warp); one lane issues.  With
    // two MMA warps, the first issues the score MMAs, the second P.V; the P.V
    // commit frees the cache stage, which the score MMA of the same tile had
    // finished reading before the softmax could produce P.  Tiles u count
    // this cluster's tiles across items.
    constexpr uint32_t idesc_lat = tc::idesc_f16(128, kBK, false, false, false);
    constexpr uint32_t idesc_rope = tc::idesc_f16(128, kBK, !kRopeF16, false, false);
    constexpr uint32_t idesc_pv = tc::idesc_f16(128, 256, false, false, true);
    bool ok = true;
    auto issue_qk = [&](int u) -> bool {
      const int ls = u % kLatStages, rs = u % kRopeStages, sb = u & 1;
      if (!wait_all(&B.lat_full[ls], (u / kLatStages) & 1, a)) return false;
      // RoPE tiles by TMA (prefill, bf16 decode); the q8_0 producer writes them
      // with the latent part, under lat_full.
      if ((!kDecode || !kQ8) && !wait_all(&B.rope_full[rs], (u / kRopeStages) & 1, a)) return false;
      if (u >= 2 && !wait_all(&B.s_free[sb], ((u >> 1) - 1) & 1, a)) return false;
      tc::fence_after_sync();
      const uint32_t k0 = smem_u32(sLat + ls * kLatStage);
      const uint32_t d = tmem + kTmS + sb * 64;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks)        // latent half: A = Q from TMEM
        tc::mma_ts_warp(d, tmem + kTmQ + ks * 8, tc::sdesc_sw128(k0 + (ks >> 2) * kChunk + (ks & 3) * 32, 16, 1024),
                        idesc_lat, ks > 0 ? 1u : 0u);
      {                                      // RoPE part, this CTA's 32 dims: A = Q_pe from smem
        const uint32_t q0 = smem_u32(sQr), r0 = smem_u32(sRope + rs * kRopeChunk);
#pragma unroll
        for (int ks = 0; ks < kRopeHalf / 16; ++ks)
          tc::mma_ss_warp(d, tc::sdesc_sw64(q0 + ks * 32), tc::sdesc_sw64(r0 + ks * 32), idesc_rope, 1u);
        tc::mma_commit_warp(&B.rope_empty[rs]);
      }
      tc::mma_commit_warp(&B.s_full[sb]);
      return true;
    };
    // `t0`: first tile of its item (O restarts; the previous item's epilogue
    // must have read O, the k-th arrival on o_free).
    auto issue_pv = [&](int u, bool t0, int k) -> bool {
      if (!wait_all(&B.p_full[u & 1], (u >> 1) & 1, a)) return false;
      if (t0 && k > 0 && !wait_all(&B.o_free, (k - 1) & 1, a)) return false;
      tc::fence_after_sync();
      const uint32_t v0 = smem_u32(sLat + (u % kLatStages) * kLatStage);
      const uint32_t p0 = smem_u32(sP + (u & 1) * kPBytes);
#pragma unroll
      for (int ks = 0; ks < kBK / 16; ++ks)
        tc::mma_ss_warp(tmem + kTmO, tc::sdesc_sw128(p0 + ks * 32, 16, 1024),
                        tc::sdesc_sw128(v0 + ks * 2048, kChunk, 1024), idesc_pv, (!t0 || ks > 0) ? 1u : 0u);
      tc::mma_commit_warp(&B.lat_empty[u % kLatStages]);
      tc::mma_commit_warp(&B.pv_done[u & 1]);
      return true;
    };
    if constexpr (mma_warps(kQ8, kDecode) == 2) {
      // Each stream in order, each as soon as its operands are ready (the
      // score MMAs are bounded by the two score buffers, so they run at most
      // three tiles ahead of P.V).
      int u = 0, k = 0;
      ItemIter<kDecode> items;
      items.init(a, first, stride, &B.ds);
      Item it;
      while (ok && items.next(it)) {
        if (warp == kMmaWarp) {
          // Q of item k in TMEM (the k-th arrival on q_ready).
          ok = wait_all(&B.q_ready, k & 1, a);
          tc::fence_after_sync();
          for (int t = 0; ok && t < it.n_tiles; ++t) ok = issue_qk(u + t);
          if (ok && kEpi) tc::mma_commit_warp(&B.q_free);     // Q and Q_pe may be replaced
        } else {
          for (int t = 0; ok && t < it.n_tiles; ++t) ok = issue_pv(u + t, t == 0, k);
          if (ok && kEpi) tc::mma_commit_warp(&B.o_ready);    // O of item k is final
        }
        u += it.n_tiles;
        ++k;
      }
    } else {
      // One warp: scores run up to three tiles ahead of P.V within an item; at
      // an item boundary the next item's first scores wait until its Q is in
      // TMEM, which is loaded only after the current item's last score MMA
      // (epilogue warps) or after its last P (softmax warps), so they are
      // issued after the current item's last P.V.
      int u = 0, k = 0;
      ItemIter<kDecode> items;
      items.init(a, first, stride, &B.ds);
      Item it;
      while (ok && items.next(it)) {
        const int n = it.n_tiles;
        ok = wait_all(&B.q_ready, k & 1, a);
        tc::fence_after_sync();
        // Step t: P.V of tile t (t >= 0), then the scores of tile t + 3.  One
        // call site of each (the decode kernel is instruction-fetch bound).
#pragma unroll 1
        for (int t = -3; ok && t < n; ++t) {
          if (t >= 0) ok = issue_pv(u + t, t == 0, k);
          if (ok && t + 3 < n) {
            ok = issue_qk(u + t + 3);
            if (ok && kEpi && t + 3 == n - 1) tc::mma_commit_warp(&B.q_free);
          }
        }
        if (ok && kEpi) tc::mma_commit_warp(&B.o_ready);
        u += n;
        ++k;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();                 // no exchange may target a CTA that has left
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <bool kQ8, bool kDecode>
cudaError_t launch_one(const CUtensorMap& tm, const CUtensorMap& tm_rope, const AttnTcArgs& a, int n_clusters,
                       cudaStream_t stream) {
  auto kern = attn_tc_kernel<kQ8, kDecode>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(2 * n_clusters), threads(kQ8, kDecode), kSmem, stream>>>(tm, tm_rope, a);
  return cudaGetLastError();
}

}  // namespace

int attn_tc_rows_per_item() { return kRows; }

int decode_clusters() { return max(1, device_sm_count() / 2); }

cudaError_t launch_attn_tc(const AttnTcArgs& args, bool q8, bool decode, int n_items, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  AttnTcArgs a = args;
  a.n_items = n_items;
  // Prefill: persistent clusters, one per SM pair (one CTA per SM fits), each
  // looping over its items.  Decode: one cluster per item (the item lengths
  // are known only on the device, so the hardware's dynamic scheduling of
  // clusters balances them).
  const int n_clusters = decode ? n_items : min(n_items, max(1, device_sm_count() / 2));
  // Tensor map of the cache rows the kernel may address (64 dims x 64 keys
  // boxes, 128-byte swizzle; rows past n_rows read as zero): the fp16 staging
  // copy for a prefill, the bf16 cache (RoPE tiles) for a bf16 decode.
  // The RoPE part (32 dims x 64 keys per CTA) through a second map with 64-byte
  // swizzle.
  CUtensorMap tm, tm_rope;
  if (!decode || !q8) {
    const uint64_t rows = static_cast<uint64_t>(a.n_rows);
    cudaError_t e = make_tmap_3d(&tm, a.kv, decode, kRow, rows, 1, kRow * 2, rows * kRow * 2, 64, kBK, 1);
    if (e != cudaSuccess) return e;
    e = make_tmap_3d(&tm_rope, a.kv, decode, kRow, rows, 1, kRow * 2, rows * kRow * 2, kRopeHalf, kBK, 1, 64);
    if (e != cudaSuccess) return e;
  } else {
    memset(&tm, 0, sizeof(tm));
    memset(&tm_rope, 0, sizeof(tm_rope));
  }
  if (!decode) return launch_one<false, false>(tm, tm_rope, a, n_clusters, stream);
  return q8 ? launch_one<true, true>(tm, tm_rope, a, n_clusters, stream)
            : launch_one<false, true>(tm, tm_rope, a, n_clusters, stream);
}

}  // namespace mla
