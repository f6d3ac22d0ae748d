// ra_bwd.cu -- blockwise backward of ring attention for sm_103a.
//
// Recomputation backward (the first page's "The Backward Pass and Gradient
// Exchange"; the fourth page's "The Backward Pass: Symmetric Ring
// Operation"): with the saved LSE and D = rowsum(dO * O),
//     P  = exp(S - LSE),      S = scale Q K^T
//     dV_j += P^T dO,         dP = dO V^T,       dS = P * (dP - D)
//     dK_j += scale dS^T Q,   dQ_i += scale dS K
// One CTA handles one 128-key tile of one KV head against one query shard i
// and one query head of its GQA group: K, V stay in shared memory and the
// unit's dK, dV accumulate in tensor memory over every query tile of shard i
// the causal rule does not mask completely (packed documents: against one
// query shard and all g heads).  The key/value block of the
// pages carries its gradient accumulators around the ring and meets shard
// (j + s) mod N at step s; here the N shards (and g heads) of a tile are
// separate units whose dK, dV partials are summed into the fp32 dk, dv with
// bulk reductions, as the dQ partial tiles are into dq.  The sum does not
// depend on the order.  Splitting by shard keeps the dq tiles that the
// resident CTAs add into (one shard and head: n_qtiles x 64 KB) inside L2.
//
// Precision: bf16 operands with fp32 accumulation lose up to 2^-9 of each
// product term, which on query rows with few visible keys (large weights)
// reaches the 1e-2 parity budget.  dS is always formed from the fp32 P; on
// steps whose query tile has a row seeing fewer than kSplitKeys keys, P and
// dS also go to the tensor cores as a bf16 pair hi + lo (lo = the rounding
// residual): dV += P_hi^T dO + P_lo^T dO, dK += dS_hi^T Q + dS_lo^T Q,
// dQ = dS_hi K + dS_lo K.  Peaked attention: a softmax warp that meets an
// entry of P above kPeakP on a plain step marks the unit, and once every
// role has finished the unit's steps (an mbarrier the softmax warps arrive
// on, waited with the usual bound) a marked unit walks its plain steps a
// second time, adding only the residual terms P_lo^T dO, dS_lo^T Q and
// dS_lo K: the sum is what the hi + lo path would have given.  Units that
// meet no such entry (all of them on diffuse inputs) pay only the max.
//
// Warp roles (16 warps):
//   warps 0-7  "softmax", two warpgroups each owning 64 of the 128 query
//              columns for all 128 keys (thread = key row): P^T =
//              exp2(S^T - LSE2) to TMEM as bf16 (and its residual on split
//              steps); dS^T = P^T (dP^T - D) to shared memory (its residual to
//              the staging buffer, on split steps)
//   warps 8-11 dQ drain: TMEM -> registers -> staging buffer -> TMA bulk
//              reduce-add into dq, 32 rows per warp; then the dK / dV
//              epilogue the same way
//   warp 12    TMA producer: K, V once; Q tiles (with their rows' LSE2 and
//              D) into a 2-deep ring, dO tiles into one buffer
//   warp 13    TMEM allocator and MMA issuer (lane 0)
//   warps 14-15 idle
// TMEM columns: S^T [0,128), then P^T over it: query columns 64h..64h+63
// as bf16 pairs hi at 64h + [0,32), lo at 64h + [32,64); dP^T then dQ
// [128,256); dV [256,..); dK [384,..).
// MMAs per step: S^T = K Q^T, dP^T = V dO^T (SS, both K-major);
// dV += P^T dO (A from TMEM, dO MN-major); dK += dS^T Q (dS^T K-major, Q
// MN-major); dQ = dS K (dS^T read MN-major, K MN-major).
#include <climits>
#include <cmath>
#include <type_traits>

#include "ra_internal.cuh"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr unsigned int kFull = 0xffffffffu;
// A plain step whose P (normalised, <= 1) holds an entry above this gets its
// residual terms added in a second round: one rounded bf16 P or dS then
// carries at most 2^-8 / 16 of a row's weight (peaked attention).
constexpr float kPeakP = 1.0f / 16.0f;

template <int D>
struct BwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kTile * 128;
  static constexpr int kTileBytes = kHalves * kHalfBytes;  // 128 rows x D bf16
  static constexpr int kDsBytes = 2 * kHalfBytes;          // 128 keys x 128 queries bf16
  static constexpr int kQSt = 2;
  static constexpr int kRowStatBytes = kTile * 4;          // one float per query row
  // Shared memory: K, V (resident); Q ring with each stage's LSE2 and D rows;
  // one dO tile; dS^T (hi); staging (dS_lo^T on split steps, then dQ).
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kDoOff = kQOff + kQSt * kTileBytes;
  static constexpr int kDsOff = kDoOff + kTileBytes;
  static constexpr int kStgOff = kDsOff + kDsBytes;
  static constexpr int kStatOff = kStgOff + kDsBytes;
  static constexpr int kBarOff = kStatOff + kQSt * 2 * kRowStatBytes;
  static constexpr int bKV = 0;
  static constexpr int bQFull = 1;
  static constexpr int bQEmpty = bQFull + kQSt;
  static constexpr int bDoFull = bQEmpty + kQSt;
  static constexpr int bDoEmpty = bDoFull + 1;
  static constexpr int bSFull = bDoEmpty + 1;
  static constexpr int bDpFull = bSFull + 1;
  static constexpr int bPReady = bDpFull + 1;
  static constexpr int bDsReady = bPReady + 1;
  static constexpr int bDsEmpty = bDsReady + 1;
  static constexpr int bDqFull = bDsEmpty + 1;
  static constexpr int bDqEmpty = bDqFull + 1;
  static constexpr int bStgEmpty = bDqEmpty + 1;
  static constexpr int bDone = bStgEmpty + 1;
  static constexpr int bDrain = bDone + 1;
  static constexpr int bRound = bDrain + 1;  // the softmax warps finished round one
  static constexpr int kNumBars = bRound + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // misc: TMEM base, abort flag, and at +8 the "redo" word (a softmax warp
  // met a P above kPeakP on a plain step: the unit takes a second round)
  static constexpr int kSmemBytes = kMiscOff + 16;
  // Alignment slack for the 1024-byte aligned tiles: as much as the 227 KB
  // limit leaves (the kernel checks at run time that its base needs no more).
  static constexpr int kMaxSmem = 232448;
  static constexpr int kSlack = kSmemBytes + 1024 <= kMaxSmem ? 1024 : kMaxSmem - kSmemBytes;
  static_assert(kSlack >= 0, "shared memory layout too large");
  static constexpr int kSmemAlloc = kSmemBytes + kSlack;
  static constexpr int kThreads = 512;
  // 128 registers per thread at launch = 128 x (152 + 152 softmax halves
  // + 96 dQ drain + 112 producer / MMA) re-split per warpgroup.
  static constexpr int kLaunchRegs = 128;
  static constexpr int kSoftmaxRegs = 152;
  static constexpr int kDrainRegs = 96;
  static constexpr int kOtherRegs = 112;
  static_assert(128 * (2 * kSoftmaxRegs + kDrainRegs + kOtherRegs) == kThreads * kLaunchRegs,
                "register re-split must use exactly the launch pool");
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kDrainWarp0 = 8;
  static constexpr int kProducerWarp = 12;
  static constexpr int kMmaWarp = 13;
  static constexpr int kHalfCols = 64;  // query columns per softmax warpgroup
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384;
  static constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t kIdescDv = idesc_bf16_f32(128, D, false, true);     // dV
  // Each drain warp adds its 32 rows of the dQ tile into dq with TMA bulk
  // reductions from its 8 KB of the staging buffer, 32 columns x 32 rows per
  // box (128-byte swizzled), two boxes per round, D / 64 rounds; the unit's
  // dK and dV leave the same way.
  static constexpr int kDqRounds = D / 64;
  static constexpr int kDqBoxBytes = 32 * 32 * 4;
  static constexpr int kDqWarpStgBytes = 2 * kDqBoxBytes;
};

enum : unsigned int {
  kSiteBProdKV = 0x51, kSiteBProdQ = 0x52,
  kSiteBMmaKV = 0x61, kSiteBMmaQ = 0x62, kSiteBMmaP = 0x63, kSiteBMmaDs = 0x64, kSiteBMmaDq = 0x65,
  kSiteBMmaDo = 0x66,
  kSiteBSmS = 0x71, kSiteBSmDp = 0x72, kSiteBSmDs = 0x73, kSiteBSmStg = 0x74, kSiteBRound = 0x75,
  kSiteBDq = 0x81, kSiteBDone = 0x82, kSiteBProdDo = 0x53,
};

struct KvUnit {
  int bb, kh, j, c;   // batch, kv head, kv shard, kv tile
  int i, hq;          // the (first) query shard it meets; unpacked: and the query head
  int g_cnt;          // unpacked: query shards i .. i + g_cnt - 1 in turn
  int kmin, kmax;     // token positions of the tile's first and last existing key
  int a_lo, a_hi;     // query tiles [a_lo, a_hi) of shard i see a key of the tile
  int a_flo;          // query tiles a >= a_flo see every key of the tile (no mask) ...
  int a_fhi;          // ... and, packed, a < a_fhi (the tile's documents end later)
  int ds0, de0, ds1, de1;  // packed: documents of the first and last key
};

// Units (unpacked): one 128-key tile against a group of qgroup consecutive
// query shards (one shard when shards are long; enough of them to make
// ~32K query rows when they are short) and one query head of its KV group;
// dK and dV of the tile are summed over its units with reductions.  Units
// run grouped by (batch, kv head, shard group, query head) with the key
// tiles innermost, so the CTAs resident together read the same Q / dO
// tiles and add their dQ partials into the same 64 KB dq tiles: one group's
// dq rows (~32K rows x 512 B = 16 MB) stay in L2 while every key tile adds
// to them.
// Units (packed documents): one 128-key tile against one query shard, with
// the g query heads of its KV head inside the unit (a tile sees only its own
// documents' query tiles, so a unit per head would be a few steps long).
// Units run grouped by (batch, kv head, query shard) with the key tiles
// innermost, so the resident CTAs add into one shard's dq rows of g heads.
// First index r in [0, n] with pos[r] >= v (pos increasing).
__device__ __forceinline__ int lower_bound_pos(const int32_t *pos, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(pos + mid) < v)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// Unpacked: the query tiles [lo, n_qtiles) of shard i see a key of the unit's
// key tile (positions kmin .. kmax), and those at or after flo see all of it.
template <bool kBlock>
__device__ __forceinline__ void shard_bounds(const BwdParams &p, int kmin, int kmax, int i,
                                             int &lo, int &flo) {
  if (!p.causal) {
    lo = 0;
    flo = 0;
    return;
  }
  // visible query tiles: those whose last row sees the tile's first key
  const int r_vis = kBlock ? lower_bound_pos(p.q_pos, p.L, kmin)
                           : max(0, first_row_at_or_after(p.layout, p.L, p.N, i, kmin));
  lo = r_vis >= p.L ? p.n_qtiles : r_vis / kTile;
  // unmasked query tiles: every row sees the tile's last key
  const int r_full = kBlock ? lower_bound_pos(p.q_pos, p.L, kmax)
                            : max(0, first_row_at_or_after(p.layout, p.L, p.N, i, kmax));
  flo = min(p.n_qtiles, (r_full + kTile - 1) / kTile);
}

template <bool kDocs, bool kBlock, bool kGroup>
__device__ __forceinline__ KvUnit decode_kv_unit(const BwdParams &p, long long u) {
  KvUnit x;
  x.c = static_cast<int>(u % p.n_ktiles);
  long long g = u / p.n_ktiles;
  x.j = static_cast<int>(g % p.N);
  g /= p.N;
  if constexpr (!kDocs) {
    const int hh = static_cast<int>(g % p.g);
    g /= p.g;
    x.i = static_cast<int>(g % p.n_groups) * p.qgroup;
    x.g_cnt = min(p.qgroup, p.N - x.i);
    g /= p.n_groups;
    x.kh = static_cast<int>(g % p.n_kv);
    x.bb = static_cast<int>(g / p.n_kv);
    x.hq = x.kh * p.g + hh;
  } else {
    x.i = static_cast<int>(g % p.N);
    x.g_cnt = 1;
    g /= p.N;
    x.kh = static_cast<int>(g % p.n_kv);
    x.bb = static_cast<int>(g / p.n_kv);
    x.hq = -1;
  }
  const int r0 = x.c * kTile;
  if constexpr (kBlock) {
    // positions of the key block's rows: given only under the causal rule
    x.kmin = p.causal ? __ldg(p.k_pos + r0) : 0;
    x.kmax = p.causal ? __ldg(p.k_pos + min(r0 + kTile, p.Lk) - 1) : 0;
  } else {
    const int r1 = min(r0 + kTile, p.L) - 1;
    x.kmin = token_at(p.layout, p.L, p.N, x.j, r0);
    x.kmax = token_at(p.layout, p.L, p.N, x.j, r1);
  }
  x.a_fhi = p.n_qtiles;
  if constexpr (!kDocs) {
    x.a_hi = p.n_qtiles;
    if constexpr (kGroup) {
      // the unit has work if some shard of its group sees the key tile
      x.a_lo = p.n_qtiles;
      x.a_flo = 0;
      for (int gi = 0; gi < x.g_cnt; ++gi) {
        int lo, flo;
        shard_bounds<kBlock>(p, x.kmin, x.kmax, x.i + gi, lo, flo);
        x.a_lo = min(x.a_lo, lo);
      }
    } else {
      shard_bounds<kBlock>(p, x.kmin, x.kmax, x.i, x.a_lo, x.a_flo);
    }
  } else {
    // A query at t sees key kp iff kp lies in t's document [ds, de) and,
    // causal, kp <= t: iff t >= (causal ? kp : ds(kp)) and t < de(kp).
    // Query rows of shard i are increasing positions, so the rows that see
    // some key of the tile and those that see all of them are row ranges.
    doc_of(p.cu, p.n_docs, x.bb, p.S, x.kmin, x.ds0, x.de0);
    doc_of(p.cu, p.n_docs, x.bb, p.S, x.kmax, x.ds1, x.de1);
    const int r_vis = max(0, first_row_at_or_after(p.layout, p.L, p.N, x.i,
                                                   p.causal ? x.kmin : x.ds0));
    const int r_end = min(p.L, first_row_at_or_after(p.layout, p.L, p.N, x.i, x.de1));
    x.a_lo = r_vis / kTile;
    x.a_hi = r_vis >= r_end ? x.a_lo : (r_end + kTile - 1) / kTile;
    const int r_flo = max(0, first_row_at_or_after(p.layout, p.L, p.N, x.i,
                                                   p.causal ? x.kmax : x.ds1));
    const int r_fhi = min(p.L, first_row_at_or_after(p.layout, p.L, p.N, x.i, x.de0));
    x.a_flo = (r_flo + kTile - 1) / kTile;
    x.a_fhi = r_fhi >= p.L ? p.n_qtiles : r_fhi / kTile;
  }
  return x;
}

struct QIter {
  int a = INT_MAX;
  // unpacked: the current shard of the unit's group and its visible and
  // unmasked query-tile bounds
  int gi = -1, lo = 0, flo = 0;
  bool done = false;
  // packed documents: the query shard, query head, the documents of the
  // current tile's first and last rows, and whether the tile has a row that
  // sees fewer than kSplitKeys keys (found once per tile, kept for its heads)
  int i = 0, hh = 0;
  int d0 = -1, d1 = -1;
  bool tile_split = false;
};

// Document index of position t, starting from a document index at or after
// it (the query tiles are visited in decreasing position order).
__device__ __forceinline__ int doc_walk(const int32_t *c, int n_docs, int d, int t) {
  if (d < 0 || d >= n_docs) {  // first use: binary search
    int lo = 0, hi = n_docs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (c[mid] <= t)
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  }
  while (d > 0 && c[d] > t) --d;
  return d;
}

// Next query tile of the unit, from the last down to the first visible one
// (every key tile of a group starts on the same query tile).  `partial` marks
// steps that need the element mask; `split` steps whose query tile has a row
// seeing fewer than kSplitKeys keys.  In the second round of a marked unit
// (kLo) only the steps the first round took plain come back, each marked
// split: their residual terms are what the round adds.
template <bool kDocs, bool kBlock, bool kGroup, bool kLo = false>
__device__ __forceinline__ bool q_next(const BwdParams &p, const KvUnit &x, QIter &it, int &i,
                                       int &a, int &hq, bool &partial, bool &split) {
  if constexpr (!kDocs && !kGroup) {
    // one query shard: its visible tiles from the last down
    for (;;) {
      it.a = it.a == INT_MAX ? p.n_qtiles - 1 : it.a - 1;
      if (it.a < x.a_lo) return false;
      i = x.i;
      a = it.a;
      hq = x.hq;
      partial = it.a < x.a_flo;
      if constexpr (kBlock)
        split = p.causal ? (__ldg(p.q_pos + it.a * kTile) + 1 < kSplitKeys) : (p.Lk < kSplitKeys);
      else
        split = p.causal ? (token_at(p.layout, p.L, p.N, x.i, it.a * kTile) + 1 < kSplitKeys)
                         : (p.S < kSplitKeys);
      if constexpr (!kLo) return true;
      if (!split) {
        split = true;
        return true;
      }
    }
  }
  if constexpr (!kDocs && kGroup) {
    // the shards of the unit's group in turn, each from its last visible tile
    for (;;) {
      if (it.done) return false;
      if (it.a == INT_MAX || it.a - 1 < it.lo) {
        // the next shard of the group with a visible tile, from its last tile
        int gi = it.a == INT_MAX ? 0 : it.gi + 1;
        int lo = 0, flo = 0;
        for (; gi < x.g_cnt; ++gi) {
          shard_bounds<kBlock>(p, x.kmin, x.kmax, x.i + gi, lo, flo);
          if (lo < p.n_qtiles) break;
        }
        if (gi >= x.g_cnt) {
          it.done = true;
          return false;
        }
        it.gi = gi;
        it.lo = lo;
        it.flo = flo;
        it.a = p.n_qtiles - 1;
      } else {
        --it.a;
      }
      i = x.i + it.gi;
      a = it.a;
      hq = x.hq;
      partial = it.a < it.flo;
      // a causal row at position t sees t + 1 keys of its sequence; a block
      // step without the causal rule takes its key block's length as the bound
      if constexpr (kBlock)
        split = p.causal ? (__ldg(p.q_pos + it.a * kTile) + 1 < kSplitKeys) : (p.Lk < kSplitKeys);
      else
        split = p.causal ? (token_at(p.layout, p.L, p.N, i, it.a * kTile) + 1 < kSplitKeys)
                         : (p.S < kSplitKeys);
      if constexpr (!kLo) return true;
      if (!split) {
        split = true;
        return true;
      }
    }
  }
  // The unit's query shard: its visible query tiles from the last down, and
  // for each the g query heads of the key tile's KV head.
  for (;;) {
    if (it.a == INT_MAX) {
      it.a = x.a_hi - 1;
      it.hh = 0;
      it.d0 = it.d1 = -1;
    } else if (++it.hh >= p.g) {
      it.hh = 0;
      --it.a;
    }
    if (it.a < x.a_lo) return false;
    it.i = x.i;
    i = it.i;
    a = it.a;
    hq = x.kh * p.g + it.hh;
    partial = it.a < x.a_flo || it.a >= x.a_fhi;
    if (it.hh == 0) {  // a new query tile
      const int t0 = token_at(p.layout, p.L, p.N, it.i, it.a * kTile);
      const int t1 = token_at(p.layout, p.L, p.N, it.i, min(it.a * kTile + kTile, p.L) - 1);
      const int32_t *cb = p.cu + static_cast<size_t>(x.bb) * (p.n_docs + 1);
      it.d0 = doc_walk(cb, p.n_docs, it.d0, t0);
      it.d1 = doc_walk(cb, p.n_docs, it.d1, t1);
      const int ds0 = cb[it.d0], de0 = cb[it.d0 + 1], ds1 = cb[it.d1], de1 = cb[it.d1 + 1];
      int minvis;
      if (p.causal)
        minvis = ds1 > t0 ? 1 : t0 - ds0 + 1;  // a document starting inside: 1
      else
        minvis = de0 < ds1 ? 1 : min(de0 - ds0, de1 - ds1);
      it.tile_split = minvis < kSplitKeys;
    }
    split = it.tile_split;
    if constexpr (!kLo) return true;
    if (!split) {
      split = true;
      return true;
    }
  }
}

// D = A B^T style: both operands K-major 128 x D tiles (M = N = 128).
template <int D>
__device__ __forceinline__ void mma_kk(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                       uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
    mma_ss(d_tmem, smem_desc_sw128(a_saddr + off, 16, 1024),
           smem_desc_sw128(b_saddr + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
  }
}

// dK (+)= dS^T Q: A = dS^T (keys x queries, K-major), B = Q MN-major.
template <int D>
__device__ __forceinline__ void issue_dk(uint32_t d_tmem, uint32_t ds_saddr, uint32_t q_saddr,
                                         bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    mma_ss(d_tmem, smem_desc_sw128(ds_saddr + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024),
           smem_desc_sw128(q_saddr + kk * 16 * 128, kTile * 128, 1024),
           idesc_bf16_f32(128, D, false, true), (accumulate || kk > 0) ? 1u : 0u);
}

// dQ = dS K: A = dS (queries x keys) read from dS^T MN-major, B = K MN-major;
// issue_dq_acc adds to what is there.
template <int D>
__device__ __forceinline__ void issue_dq_step(uint32_t d_tmem, uint32_t ds_saddr, uint32_t k_saddr,
                                              bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    mma_ss(d_tmem, smem_desc_sw128(ds_saddr + kk * 16 * 128, kTile * 128, 1024),
           smem_desc_sw128(k_saddr + kk * 16 * 128, kTile * 128, 1024),
           idesc_bf16_f32(128, D, true, true), (accumulate || kk > 0) ? 1u : 0u);
}
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint32_t ds_saddr, uint32_t k_saddr) {
  issue_dq_step<D>(d_tmem, ds_saddr, k_saddr, false);
}
template <int D>
__device__ __forceinline__ void issue_dq_acc(uint32_t d_tmem, uint32_t ds_saddr, uint32_t k_saddr) {
  issue_dq_step<D>(d_tmem, ds_saddr, k_saddr, true);
}

// 64 columns of a P^T row (fp32), query columns [c_base, c_base + 64), to
// TMEM as bf16 pairs over the S^T columns they came from: at c_base + [0,32),
// and with kSplit the rounding residual at c_base + [32,64).  Each softmax
// warpgroup so overwrites only the S^T columns it has itself read.
template <bool kSplit>
__device__ __forceinline__ void store_p_half(const float (&pf)[64], uint32_t tS, int c_base) {
#pragma unroll
  for (int q2 = 0; q2 < 2; ++q2) {
    uint32_t hi[16];
    uint32_t lo[kSplit ? 16 : 1];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int c = q2 * 32 + 2 * e;
      hi[e] = pack_bf16x2(pf[c], pf[c + 1]);
      if constexpr (kSplit)
        lo[e] = pack_bf16x2(pf[c] - __uint_as_float(hi[e] << 16),
                            pf[c + 1] - __uint_as_float(hi[e] & 0xffff0000u));
    }
    tmem_st16(tS + c_base + q2 * 16, hi);
    if constexpr (kSplit) tmem_st16(tS + c_base + 32 + q2 * 16, lo);
  }
}

template <int D, bool kDocs, bool kBlock, bool kGroup>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    bwd_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap domap,
               const __grid_constant__ CUtensorMap dqmap,
               const __grid_constant__ CUtensorMap dkmap,
               const __grid_constant__ CUtensorMap dvmap) {
  using C = BwdCfg<D>;
  const KvUnit x = decode_kv_unit<kDocs, kBlock, kGroup>(p, blockIdx.x);
  if (x.a_lo >= x.a_hi) return;  // no query of this shard sees the tile: nothing to add
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(C::kSlack)) {  // uniform: never touch smem beyond the allocation
    if (threadIdx.x == 0) raise_error(kErrLayout, 0x5F);
    return;
  }
  uint8_t *smem = smem_raw + pad;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);

  if (threadIdx.x == 0) {
    mbar_init(&bars[C::bKV], 1);
    for (int s = 0; s < C::kQSt; ++s) {
      mbar_init(&bars[C::bQFull + s], 1);
      mbar_init(&bars[C::bQEmpty + s], 1);
    }
    mbar_init(&bars[C::bDoFull], 1);
    mbar_init(&bars[C::bDoEmpty], 1);
    mbar_init(&bars[C::bSFull], 1);
    mbar_init(&bars[C::bDpFull], 1);
    mbar_init(&bars[C::bPReady], 8);
    mbar_init(&bars[C::bDsReady], 8);
    mbar_init(&bars[C::bDsEmpty], 1);
    mbar_init(&bars[C::bDqFull], 1);
    mbar_init(&bars[C::bDqEmpty], 4);
    mbar_init(&bars[C::bStgEmpty], 4);
    mbar_init(&bars[C::bDone], 1);
    mbar_init(&bars[C::bDrain], 1);
    mbar_init(&bars[C::bRound], 8);
    *abort_flag = 0;
    *reinterpret_cast<volatile int *>(smem + C::kMiscOff + 8) = 0;
    fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Every role, after its first round over the unit, learns whether a
  // softmax warp met a P above kPeakP on a plain step; the unit then takes a
  // second round over those steps for their residual terms (warp-collective).
  auto second_round = [&]() -> bool {
    int r = 0;
    if (lane == 0 && mbar_wait(&bars[C::bRound], 0, abort_flag, kSiteBRound))
      r = *reinterpret_cast<volatile int *>(smem + C::kMiscOff + 8);
    r = __shfl_sync(kFull, r, 0);
    return r != 0 && *abort_flag == 0;
  };

  if (warp >= C::kProducerWarp) {
    regs_set<C::kOtherRegs, C::kLaunchRegs>();
    if (warp == C::kProducerWarp) {
      // ---------------------------------------------------------- producer
      int q_par[C::kQSt] = {-1, -1};
      int do_par = -1;
      if (lane == 0) {
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
        prefetch_tmap(&domap);
        int c2, c3;
        map_coords(p.layout, p.L, p.N, x.j, x.c * kTile, c2, c3);
        mbar_arrive_expect_tx(&bars[C::bKV], 2 * C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_load_5d(smem + C::kKOff + hf * C::kHalfBytes, &kmap, &bars[C::bKV], hf * 64, x.kh,
                      c2, c3, x.bb);
          tma_load_5d(smem + C::kVOff + hf * C::kHalfBytes, &vmap, &bars[C::bKV], hf * 64, x.kh,
                      c2, c3, x.bb);
        }
      }
      QIter it;
      int i, a, hq, n = 0;
      bool partial, split;
      // one step's loads: the Q tile with its rows' LSE2 and D, and dO
      auto load_step = [&]() -> bool {
        if (lane == 0) {
          int c2, c3;
          map_coords(p.layout, p.L, p.N, i, a * kTile, c2, c3);
          const int st = n % C::kQSt;
          const uint32_t ph = (n / C::kQSt) & 1;
          bool go = mbar_wait(&bars[C::bQEmpty + st], ph ^ 1, abort_flag, kSiteBProdQ);
          if (go) {
            mbar_arrive_expect_tx(&bars[C::bQFull + st], C::kTileBytes + 2 * C::kRowStatBytes);
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_5d(smem + C::kQOff + st * C::kTileBytes + hf * C::kHalfBytes, &qmap,
                          &bars[C::bQFull + st], hf * 64, hq, c2, c3, x.bb);
            const size_t qrow0 =
                ((static_cast<size_t>(x.bb) * p.h + hq) * p.N + i) * p.Lpad + a * kTile;
            uint8_t *stat = smem + C::kStatOff + st * 2 * C::kRowStatBytes;
            bulk_copy_g2s(stat, p.lse2 + qrow0, C::kRowStatBytes, &bars[C::bQFull + st]);
            bulk_copy_g2s(stat + C::kRowStatBytes, p.dvec + qrow0, C::kRowStatBytes,
                          &bars[C::bQFull + st]);
            q_par[st] = static_cast<int>(ph);
            go = mbar_wait(&bars[C::bDoEmpty], (n & 1) ^ 1, abort_flag, kSiteBProdDo);
          }
          if (go) {
            mbar_arrive_expect_tx(&bars[C::bDoFull], C::kTileBytes);
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_5d(smem + C::kDoOff + hf * C::kHalfBytes, &domap, &bars[C::bDoFull],
                          hf * 64, hq, c2, c3, x.bb);
            do_par = n & 1;
          }
        }
        __syncwarp();
        if (*abort_flag) return false;
        ++n;
        return true;
      };
      while (q_next<kDocs, kBlock, kGroup>(p, x, it, i, a, hq, partial, split))
        if (!load_step()) break;
      if (!*abort_flag && second_round()) {
        QIter it2;
        while (q_next<kDocs, kBlock, kGroup, true>(p, x, it2, i, a, hq, partial, split))
          if (!load_step()) break;
      }
      if (lane == 0 && *abort_flag) {
        // Let every copy this warp started land before the CTA unwinds.
        mbar_wait_budget(&bars[C::bKV], 0, kWaitBudgetCycles);
        for (int s = 0; s < C::kQSt; ++s)
          if (q_par[s] >= 0) mbar_wait_budget(&bars[C::bQFull + s], q_par[s], kWaitBudgetCycles);
        if (do_par >= 0) mbar_wait_budget(&bars[C::bDoFull], do_par, kWaitBudgetCycles);
      }
    } else if (warp == C::kMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&bars[C::bKV], 0, abort_flag, kSiteBMmaKV);
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (ok) {
        tc_fence_after();
        const uint32_t k_s = sbase + C::kKOff;
        const uint32_t v_s = sbase + C::kVOff;
        const uint32_t do_s = sbase + C::kDoOff;
        const uint32_t ds_s = sbase + C::kDsOff;
        const uint32_t dslo_s = sbase + C::kStgOff;
        QIter it;
        int i, a, hq, n = 0;
        bool partial, split;
        // S^T of step n_s into the S^T columns once its Q tile has landed
        auto issue_s = [&](int n_s) -> bool {
          const int st = n_s % C::kQSt;
          if (!mbar_wait(&bars[C::bQFull + st], (n_s / C::kQSt) & 1, abort_flag, kSiteBMmaQ))
            return false;
          tc_fence_after();
          mma_kk<D>(tmem + C::kColS, k_s, sbase + C::kQOff + st * C::kTileBytes, C::kIdescKK);
          mma_commit(&bars[C::bSFull]);
          return true;
        };
        bool has = q_next<kDocs, kBlock, kGroup>(p, x, it, i, a, hq, partial, split);
        if (has && lane == 0) issue_s(0);
        __syncwarp();
        while (has && !*abort_flag) {
          const bool cur_split = split;
          const bool has_next = q_next<kDocs, kBlock, kGroup>(p, x, it, i, a, hq, partial, split);
          if (lane == 0) {
            const int st = n % C::kQSt;
            const uint32_t q_s = sbase + C::kQOff + st * C::kTileBytes;
            bool go = true;
            if (n > 0) go = mbar_wait(&bars[C::bDqEmpty], (n - 1) & 1, abort_flag, kSiteBMmaDq);
            if (go) go = mbar_wait(&bars[C::bDoFull], n & 1, abort_flag, kSiteBMmaDo);
            if (go) {
              tc_fence_after();
              // dP^T = V dO^T
              mma_kk<D>(tmem + C::kColDp, v_s, do_s, C::kIdescKK);
              mma_commit(&bars[C::bDpFull]);
              go = mbar_wait(&bars[C::bPReady], n & 1, abort_flag, kSiteBMmaP);
            }
            if (go) {
              tc_fence_after();
              // dV += P_hi^T dO (+ P_lo^T dO): A from TMEM (bf16 pairs), B = dO MN-major
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + C::kColDv, tmem + C::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                       smem_desc_sw128(do_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv,
                       (n > 0 || kk > 0) ? 1u : 0u);
              if (cur_split)
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                  mma_ts(tmem + C::kColDv, tmem + C::kColS + (kk >> 2) * 64 + 32 + (kk & 3) * 8,
                         smem_desc_sw128(do_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv,
                         1u);
              mma_commit(&bars[C::bDoEmpty]);
              if (has_next) {
                const int st1 = (n + 1) % C::kQSt;
                go = mbar_wait(&bars[C::bQFull + st1], ((n + 1) / C::kQSt) & 1, abort_flag,
                               kSiteBMmaQ);
                if (go) {
                  tc_fence_after();
                  mma_kk<D>(tmem + C::kColS, k_s, sbase + C::kQOff + st1 * C::kTileBytes,
                            C::kIdescKK);
                  mma_commit(&bars[C::bSFull]);
                }
              }
            }
            if (go) go = mbar_wait(&bars[C::bDsReady], n & 1, abort_flag, kSiteBMmaDs);
            if (go) {
              tc_fence_after();
              if (!cur_split) {
                // dQ first, so the drain (and with it the next dP^T) starts
                // while dK accumulates
                issue_dq<D>(tmem + C::kColDp, ds_s, k_s);
                mma_commit(&bars[C::bDqFull]);
                issue_dk<D>(tmem + C::kColDk, ds_s, q_s, n > 0);
              } else {
                // the drain stages dQ where dS_lo^T is: every reader of
                // dS_lo^T completes before dQ is handed over
                issue_dk<D>(tmem + C::kColDk, ds_s, q_s, n > 0);
                issue_dk<D>(tmem + C::kColDk, dslo_s, q_s, true);
                issue_dq<D>(tmem + C::kColDp, ds_s, k_s);
                issue_dq_acc<D>(tmem + C::kColDp, dslo_s, k_s);
                mma_commit(&bars[C::bDqFull]);
              }
              mma_commit(&bars[C::bDsEmpty]);
              mma_commit(&bars[C::bQEmpty + st]);
            }
          }
          __syncwarp();
          ++n;
          has = has_next;
        }
        // Second round of a marked unit: the plain steps again, adding only
        // their residual terms (every accumulator keeps adding).
        if (!*abort_flag && second_round()) {
          QIter it2;
          has = q_next<kDocs, kBlock, kGroup, true>(p, x, it2, i, a, hq, partial, split);
          if (has && lane == 0) issue_s(n);
          __syncwarp();
          while (has && !*abort_flag) {
            const bool has_next = q_next<kDocs, kBlock, kGroup, true>(p, x, it2, i, a, hq, partial, split);
            if (lane == 0) {
              const int st = n % C::kQSt;
              const uint32_t q_s = sbase + C::kQOff + st * C::kTileBytes;
              bool go = mbar_wait(&bars[C::bDqEmpty], (n - 1) & 1, abort_flag, kSiteBMmaDq);
              if (go) go = mbar_wait(&bars[C::bDoFull], n & 1, abort_flag, kSiteBMmaDo);
              if (go) {
                tc_fence_after();
                mma_kk<D>(tmem + C::kColDp, v_s, do_s, C::kIdescKK);
                mma_commit(&bars[C::bDpFull]);
                go = mbar_wait(&bars[C::bPReady], n & 1, abort_flag, kSiteBMmaP);
              }
              if (go) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                  mma_ts(tmem + C::kColDv, tmem + C::kColS + (kk >> 2) * 64 + 32 + (kk & 3) * 8,
                         smem_desc_sw128(do_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv,
                         1u);
                mma_commit(&bars[C::bDoEmpty]);
                if (has_next) go = issue_s(n + 1);
              }
              if (go) go = mbar_wait(&bars[C::bDsReady], n & 1, abort_flag, kSiteBMmaDs);
              if (go) {
                tc_fence_after();
                issue_dk<D>(tmem + C::kColDk, dslo_s, q_s, true);
                issue_dq<D>(tmem + C::kColDp, dslo_s, k_s);
                mma_commit(&bars[C::bDqFull]);
                mma_commit(&bars[C::bDsEmpty]);
                mma_commit(&bars[C::bQEmpty + st]);
              }
            }
            __syncwarp();
            ++n;
            has = has_next;
          }
        }
        if (lane == 0) mma_commit(&bars[C::bDone]);
      }
      if (lane == 0) {
        // Every MMA this thread issued has finished before TMEM is released.
        mma_commit(&bars[C::bDrain]);
        mbar_wait_budget(&bars[C::bDrain], 0, kWaitBudgetCycles);
      }
      __syncwarp();
    }
  } else if (warp < C::kSoftmaxWarps) {
    regs_set<C::kSoftmaxRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------ softmax (thread = key)
    const int half = warp >> 2;          // which 64 query columns
    const int cb = half * C::kHalfCols;  // first query column of this warpgroup
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS;
    const uint32_t tDp = tmem + lane_off + C::kColDp + cb;
    const int kr = x.c * kTile + row;
    const int n_keys = kBlock ? p.Lk : p.L;
    const bool key_exists = kr < n_keys;
    // this key's position (a block step without the causal rule has none:
    // nothing below reads it then)
    int kp;
    if constexpr (kBlock)
      kp = p.causal ? __ldg(p.k_pos + (key_exists ? kr : n_keys - 1)) : 0;
    else
      kp = token_at(p.layout, p.L, p.N, x.j, key_exists ? kr : p.L - 1);
    // this key is seen by the query positions [kq_lo, kq_hi)
    int kq_lo = kp, kq_hi = p.S;
    if constexpr (kDocs) {
      int kds;
      doc_of(p.cu, p.n_docs, x.bb, p.S, kp, kds, kq_hi);
      if (!p.causal) kq_lo = kds;
    }
    const float sl2 = p.scale_log2;
    // this warpgroup's 64 query columns are one 128-byte-swizzled half of dS^T
    uint8_t *ds_row = smem + C::kDsOff + half * (kTile * 128) + row * 128;
    uint8_t *dslo_row = smem + C::kStgOff + half * (kTile * 128) + row * 128;
    QIter it;
    int i, a, hq, n = 0;
    bool partial, split;
    // one step; the second round of a marked unit (kLoRound) detects nothing
    auto sm_step = [&](auto lo_tag) -> bool {
      constexpr bool kLoRound = decltype(lo_tag)::value;
      // this step's LSE2 and D rows, staged by the producer with the Q tile
      const float4 *lse4 = reinterpret_cast<const float4 *>(
                               smem + C::kStatOff + (n % C::kQSt) * 2 * C::kRowStatBytes) +
                           cb / 4;
      const float4 *d4 = lse4 + kTile / 4;
      // query columns cb + c with c < c0 or c >= c1 are masked for this key
      int c0 = 0, c1 = C::kHalfCols;
      if (partial) {
        c0 = (kBlock ? lower_bound_pos(p.q_pos, p.L, kq_lo)
                     : first_row_at_or_after(p.layout, p.L, p.N, i, kq_lo)) -
             a * kTile - cb;
        if constexpr (kDocs)
          c1 = first_row_at_or_after(p.layout, p.L, p.N, i, kq_hi) - a * kTile - cb;
      }
      if (!key_exists) {
        c0 = C::kHalfCols;
        partial = true;
      }
      if (!__all_sync(kFull, mbar_wait(&bars[C::bSFull], n & 1, abort_flag, kSiteBSmS))) return false;
      tc_fence_after();
      float pf[C::kHalfCols];  // this warpgroup's half of the P^T row, fp32
      {
        uint32_t sr[2][32];
        tmem_ld32_start(tS + cb, sr[0]);
        tmem_ld32_start(tS + cb + 32, sr[1]);
        float4 l4[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) l4[e] = lse4[e];
        tmem_ld_wait_regs(sr[0]);
        tmem_ld_wait_regs(sr[1]);
        const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
        for (int e4 = 0; e4 < 16; ++e4) {
          const int c = e4 * 4;
          float x0, x1, x2, x3;
          f2unpack(ffma2(f2pack(__uint_as_float(sr[c >> 5][(c + 0) & 31]),
                                __uint_as_float(sr[c >> 5][(c + 1) & 31])),
                         sl2x2, f2pack(l4[e4].x, l4[e4].y)), x0, x1);
          f2unpack(ffma2(f2pack(__uint_as_float(sr[c >> 5][(c + 2) & 31]),
                                __uint_as_float(sr[c >> 5][(c + 3) & 31])),
                         sl2x2, f2pack(l4[e4].z, l4[e4].w)), x2, x3);
          pf[c + 0] = ex2(x0);
          pf[c + 1] = ex2(x1);
          pf[c + 2] = ex2(x2);
          pf[c + 3] = ex2(x3);
        }
      }
      if (partial) {  // causal diagonal: columns before c0 do not see this key
#pragma unroll
        for (int c = 0; c < C::kHalfCols; ++c)
          if (c < c0 || (kDocs && c >= c1)) pf[c] = 0.f;
      }
      // A P above kPeakP on a plain step: the unit takes a second round
      // for the residual terms of its plain steps.
      if (!kLoRound && !split) {
        float pm = 0.f;
#pragma unroll
        for (int c = 0; c < C::kHalfCols; c += 2) pm = fmax3(pm, pf[c], pf[c + 1]);
        if (__any_sync(kFull, pm > kPeakP) && lane == 0)
          *reinterpret_cast<volatile int *>(smem + C::kMiscOff + 8) = 1;
      }
      if (split)
        store_p_half<true>(pf, tS, cb);
      else
        store_p_half<false>(pf, tS, cb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::bPReady]);

      bool go = mbar_wait(&bars[C::bDpFull], n & 1, abort_flag, kSiteBSmDp);
      if (go) go = mbar_wait(&bars[C::bDsEmpty], (n & 1) ^ 1, abort_flag, kSiteBSmDs);
      // the residual goes to the staging buffer once the drain is done with it
      if (go && split && n > 0)
        go = mbar_wait(&bars[C::bStgEmpty], (n - 1) & 1, abort_flag, kSiteBSmStg);
      if (!__all_sync(kFull, go)) return false;
      tc_fence_after();
      // all 64 dP^T columns of this half in one round of loads; dS = P (dP - D)
      // on f32x2 pairs
      uint32_t r4[4][16];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld16_start(tDp + ch * 16, r4[ch]);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld_wait_regs16(r4[ch]);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float sv[16];
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const float4 dd = d4[ch * 4 + e4];
          const int c = ch * 16 + e4 * 4;
          const uint64_t t0 = fadd2(f2pack(__uint_as_float(r4[ch][e4 * 4 + 0]), __uint_as_float(r4[ch][e4 * 4 + 1])),
                                    f2pack(dd.x, dd.y));
          const uint64_t t1 = fadd2(f2pack(__uint_as_float(r4[ch][e4 * 4 + 2]), __uint_as_float(r4[ch][e4 * 4 + 3])),
                                    f2pack(dd.z, dd.w));
          f2unpack(fmul2(f2pack(pf[c + 0], pf[c + 1]), t0), sv[e4 * 4 + 0], sv[e4 * 4 + 1]);
          f2unpack(fmul2(f2pack(pf[c + 2], pf[c + 3]), t1), sv[e4 * 4 + 2], sv[e4 * 4 + 3]);
        }
        uint32_t whi[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) whi[e] = pack_bf16x2(sv[2 * e], sv[2 * e + 1]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int chunk = (ch * 2 + u) ^ (row & 7);
          *reinterpret_cast<uint4 *>(ds_row + chunk * 16) =
              make_uint4(whi[u * 4 + 0], whi[u * 4 + 1], whi[u * 4 + 2], whi[u * 4 + 3]);
        }
        if (split) {
          uint32_t wlo[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            wlo[e] = pack_bf16x2(sv[2 * e] - __uint_as_float(whi[e] << 16),
                                 sv[2 * e + 1] - __uint_as_float(whi[e] & 0xffff0000u));
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int chunk = (ch * 2 + u) ^ (row & 7);
            *reinterpret_cast<uint4 *>(dslo_row + chunk * 16) =
                make_uint4(wlo[u * 4 + 0], wlo[u * 4 + 1], wlo[u * 4 + 2], wlo[u * 4 + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::bDsReady]);
      ++n;
      return true;
    };
    while (q_next<kDocs, kBlock, kGroup>(p, x, it, i, a, hq, partial, split))
      if (!sm_step(std::false_type{})) break;
    // round one is over for this warp (and its detections are written)
    if (lane == 0) mbar_arrive(&bars[C::bRound]);
    if (!*abort_flag && second_round()) {
      QIter it2;
      while (q_next<kDocs, kBlock, kGroup, true>(p, x, it2, i, a, hq, partial, split))
        if (!sm_step(std::true_type{})) break;
    }
  } else if (warp < C::kDrainWarp0 + 4) {
    regs_set<C::kDrainRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------ dQ drain, then dK/dV
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDq = tmem + lane_off + C::kColDp;
    uint8_t *stg = smem + C::kStgOff + (warp & 3) * C::kDqWarpStgBytes;  // this warp's 32 rows
    QIter it;
    int i, a, hq, n = 0;
    bool partial, split;
    bool aborted = false;
    // one step's dQ partial: TMEM -> registers -> staging -> bulk reduce-add
    auto drain_step = [&]() -> bool {
      if (!__all_sync(kFull, mbar_wait(&bars[C::bDqFull], n & 1, abort_flag, kSiteBDq))) {
        aborted = true;
        return false;
      }
      tc_fence_after();
      {
        // D / 64 rounds of two 32 x 32 boxes through this warp's staging slice;
        // the staging buffer is free: this step's dS_lo^T readers finished
        // before dQ was committed, and the previous round's read completed.
        int c2, c3;
        map_coords(p.layout, p.L, p.N, i, a * kTile + (warp & 3) * 32, c2, c3);
#pragma unroll
        for (int round = 0; round < C::kDqRounds; ++round) {
          uint32_t r[2][32];
          tmem_ld32_start(tDq + round * 64, r[0]);
          tmem_ld32_start(tDq + round * 64 + 32, r[1]);
          tmem_ld_wait_regs(r[0]);
          tmem_ld_wait_regs(r[1]);
          if (round == C::kDqRounds - 1) {  // every dQ column is in registers: TMEM free for dP
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[C::bDqEmpty]);
          }
          if (round > 0) {
            if (lane == 0) bulk_wait_group0<true>();  // the previous round's staging read
            __syncwarp();
          }
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            uint8_t *rowp = stg + bx * C::kDqBoxBytes + lane * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<float4 *>(rowp + ((u ^ (lane & 7)) * 16)) =
                  make_float4(__uint_as_float(r[bx][4 * u + 0]) * p.scale,
                              __uint_as_float(r[bx][4 * u + 1]) * p.scale,
                              __uint_as_float(r[bx][4 * u + 2]) * p.scale,
                              __uint_as_float(r[bx][4 * u + 3]) * p.scale);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int bx = 0; bx < 2; ++bx)
              tma_reduce_add_5d(&dqmap, stg + bx * C::kDqBoxBytes, (round * 2 + bx) * 32, hq, c2,
                                c3, x.bb);
            bulk_commit_group();
          }
        }
        if (lane == 0) {
          bulk_wait_group0<true>();  // the last round's staging read: slice reusable
          mbar_arrive(&bars[C::bStgEmpty]);
        }
        __syncwarp();
      }
      ++n;
      return true;
    };
    while (q_next<kDocs, kBlock, kGroup>(p, x, it, i, a, hq, partial, split))
      if (!drain_step()) break;
    if (!aborted && second_round()) {
      QIter it2;
      while (q_next<kDocs, kBlock, kGroup, true>(p, x, it2, i, a, hq, partial, split))
        if (!drain_step()) break;
    }
    if (lane == 0) bulk_wait_group0<false>();  // this warp's reductions complete
    // dK, dV of this unit, added into dk and dv (other units of the tile add
    // theirs) through this warp's staging slice with bulk reductions.
    bool have = n > 0 && !aborted;
    if (have) have = mbar_wait(&bars[C::bDone], 0, abort_flag, kSiteBDone);
    have = __all_sync(kFull, have && *abort_flag == 0);
    if (have) {
      tc_fence_after();
      const int r0 = x.c * kTile + (warp & 3) * 32;  // this warp's first key row
      {
        uint8_t *stg = smem + C::kStgOff + (warp & 3) * C::kDqWarpStgBytes;
        int c2, c3;
        map_coords(p.layout, p.L, p.N, x.j, r0, c2, c3);
#pragma unroll
        for (int round = 0; round < 2 * C::kDqRounds; ++round) {  // dK, then dV, 64 columns a round
          const bool is_dk = round < C::kDqRounds;
          const int part = round % C::kDqRounds;
          const uint32_t col = (is_dk ? C::kColDk : C::kColDv) + part * 64;
          const float mul = is_dk ? p.scale : 1.f;
          uint32_t r[2][32];
          tmem_ld32_start(tmem + lane_off + col, r[0]);
          tmem_ld32_start(tmem + lane_off + col + 32, r[1]);
          tmem_ld_wait_regs(r[0]);
          tmem_ld_wait_regs(r[1]);
          if (lane == 0) bulk_wait_group0<true>();  // the slice's previous reads
          __syncwarp();
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            uint8_t *rowp = stg + bx * C::kDqBoxBytes + lane * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<float4 *>(rowp + ((u ^ (lane & 7)) * 16)) =
                  make_float4(__uint_as_float(r[bx][4 * u + 0]) * mul,
                              __uint_as_float(r[bx][4 * u + 1]) * mul,
                              __uint_as_float(r[bx][4 * u + 2]) * mul,
                              __uint_as_float(r[bx][4 * u + 3]) * mul);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && r0 < (kBlock ? p.Lk : p.L)) {
#pragma unroll
            for (int bx = 0; bx < 2; ++bx)
              tma_reduce_add_5d(is_dk ? &dkmap : &dvmap, stg + bx * C::kDqBoxBytes,
                                part * 64 + bx * 32, x.kh, c2, c3, x.bb);
            bulk_commit_group();
          }
        }
        if (lane == 0) bulk_wait_group0<false>();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// -D = -rowsum(dO * O) and -LSE2 = -LSE * log2(e) per (batch, head, query
// row), stored negated so the main kernel adds them with f32x2 arithmetic,
// written in shard-local order [b, h, N, Lpad]; padding rows get D = 0 and
// -LSE2 = -inf (their P is exactly 0).  One warp per row, four rows in flight.
template <int D>
__global__ void bwd_pre_kernel(BwdParams p, const float *out, const float *lse,
                               const uint16_t *dout) {
  // blockIdx.y walks the (batch, head, shard) row groups of the workspace,
  // blockIdx.x the rows of a group, four rows in flight per warp.
  constexpr int kRows = 4;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long r0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long groups = static_cast<long long>(p.b) * p.h * p.N;
  for (long long g = blockIdx.y; g < groups; g += gridDim.y) {
    const int i = static_cast<int>(g % p.N);
    const long long bh = g / p.N;
    const int hq = static_cast<int>(bh % p.h);
    const long long bb = bh / p.h;
    for (long long base = r0; base < p.Lpad; base += kRows * warps) {
      // lane e holds columns 4e..4e+3 of each row (d = 64 uses half the warp)
      float4 o[kRows];
      uint2 gg[kRows];
      float lv[kRows];
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const long long r = base + k * warps;
        if (r < p.L) {
          const int tok = token_at(p.layout, p.L, p.N, i, static_cast<int>(r));
          const size_t row = ((bb * p.S + tok) * p.h + hq) * D;
          if (lane < D / 4) {
            o[k] = reinterpret_cast<const float4 *>(out + row)[lane];
            gg[k] = reinterpret_cast<const uint2 *>(dout + row)[lane];
          }
          lv[k] = lse[(bb * p.h + hq) * p.S + tok];
        }
      }
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const long long r = base + k * warps;
        if (r >= p.Lpad) continue;
        float dsum = 0.f, l2 = INFINITY;  // padding rows: D = 0, P = 0
        if (r < p.L) {
          if (lane < D / 4)
            dsum = o[k].x * __uint_as_float(gg[k].x << 16) +
                   o[k].y * __uint_as_float(gg[k].x & 0xffff0000u) +
                   o[k].z * __uint_as_float(gg[k].y << 16) +
                   o[k].w * __uint_as_float(gg[k].y & 0xffff0000u);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(kFull, dsum, off);
          l2 = (lv[k] == -INFINITY) ? INFINITY : lv[k] * kLog2e;
        }
        if (lane == 0) {
          p.dvec[g * p.Lpad + r] = -dsum;
          p.lse2[g * p.Lpad + r] = -l2;
        }
      }
    }
  }
}

template <int D>
cudaError_t launch_bwd_t(const BwdParams &p, const float *out, const float *lse,
                         const uint16_t *dout, const CUtensorMap &qmap, const CUtensorMap &kmap,
                         const CUtensorMap &vmap, const CUtensorMap &domap,
                         const CUtensorMap &dqmap, const CUtensorMap &dkmap,
                         const CUtensorMap &dvmap, long long n_units, int n_sm,
                         cudaStream_t stream) {
  using C = BwdCfg<D>;
  // about eight CTAs of 256 threads per SM: y over the (batch, head, shard)
  // row groups, x over the rows of a group (32 rows per CTA and trip)
  const long long groups = static_cast<long long>(p.b) * p.h * p.N;
  const long long gy = groups < 65535 ? (groups < 1 ? 1 : groups) : 65535;
  long long gx = (p.Lpad + 31) / 32;
  const long long cap = (static_cast<long long>(n_sm) * 8 + gy - 1) / gy;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  bwd_pre_kernel<D><<<dim3(static_cast<unsigned int>(gx), static_cast<unsigned int>(gy)), 256, 0,
                      stream>>>(p, out, lse, dout);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // units over a group of query shards walk them with their own iterator,
  // compiled separately: folded into the one-shard kernel it cost 7 % there
  auto kern = p.block           ? bwd_kernel<D, false, true, false>
              : p.cu != nullptr ? bwd_kernel<D, true, false, false>
              : p.qgroup > 1    ? bwd_kernel<D, false, false, true>
                                : bwd_kernel<D, false, false, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  {
    // The register increases in the kernel wait until the pool covers them.
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    // The re-split assumes each warpgroup starts from exactly kLaunchRegs.
    if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  }
  kern<<<dim3(static_cast<unsigned int>(n_units)), dim3(C::kThreads), C::kSmemAlloc, stream>>>(
      p, qmap, kmap, vmap, domap, dqmap, dkmap, dvmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdParams &p, int d, const float *out, const float *lse,
                       const uint16_t *dout, const CUtensorMap &qmap, const CUtensorMap &kmap,
                       const CUtensorMap &vmap, const CUtensorMap &domap,
                       const CUtensorMap &dqmap, const CUtensorMap &dkmap,
                       const CUtensorMap &dvmap, long long n_units, int n_sm,
                       cudaStream_t stream) {
  if (n_units <= 0) return cudaSuccess;
  if (d == 128)
    return launch_bwd_t<128>(p, out, lse, dout, qmap, kmap, vmap, domap, dqmap, dkmap, dvmap,
                             n_units, n_sm, stream);
  if (d == 64)
    return launch_bwd_t<64>(p, out, lse, dout, qmap, kmap, vmap, domap, dqmap, dkmap, dvmap,
                            n_units, n_sm, stream);
  return cudaErrorInvalidValue;
}

RA_DEFINE_ERROR_WORD_READER(read_error_word_bwd)

}  // namespace ra
