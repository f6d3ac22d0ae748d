// ra_fwd.cu -- forward blockwise ring-attention kernel for sm_103a.
//
// One CTA owns NQ query tiles of 128 rows (NQ = 2: two query heads of the
// same GQA group at the same rows, so every K/V tile it loads serves both)
// and walks the key/value tiles in ring order: shard (i - s) mod N for
// s = 0..N-1 (the fourth page's "The Ring Communication Protocol"), skipping
// tiles the causal rule masks completely.  Per tile and query tile it runs
// the online-softmax update of the first page's "Blockwise Attention and
// Online Softmax Formulations":
//     S = Q K^T;  m' = max(m, rowmax S);  P = exp(S - m');
//     l' = e^(m - m') l + rowsum P;  O' = e^(m - m') O + P V
// with S, P and O held in tensor memory (TMEM) and the two GEMMs issued as
// tcgen05.mma by one thread.  The epilogue either finalizes (O / l and
// LSE = m + ln l, ring mode) or folds the block result into a caller-held
// (m, l, O) state with the second page's rescale-merge (block-step mode).
//
// Warp roles (NQ = 2):
//   warps 0-3  softmax + O rescale + epilogue for query tile 0 (thread = row)
//   warps 4-7  the same for query tile 1
//   warp 8     TMA producer: Q once, then K and V tiles into 2-deep rings
//   warp 9     TMEM allocator and MMA issuer (lane 0)
// TMEM columns: S_t/P_t at [128 t, 128 t + 128), O_t at [128 NQ + 128 t, ...).
// P_t (bf16) overwrites the first 64 columns of S_t and feeds the PV MMA
// straight from TMEM.
//
// Exponentials are base 2 with log2(e) folded into the scale.  The running
// max used as the exponent shift is only raised when a row's max grows by
// more than 8 (log2 units), or when the key that raised it would dominate
// the row's sum so far, so most tiles skip the O rescale; P stays <= 2^8 and
// the result is unchanged because O and l share the same shift.
// Once every row of a warp has a shift, P is formed against it before the
// tile's row max is known (the max is taken while the P stores drain); the
// rare tile whose max passes a row's shift by more than 8 is formed again.
// The exact running max is tracked alongside for the block-step state.
//
// Precision: tiles whose rows see fewer than kSplitKeys keys (and every
// block step) store P as a bf16 pair, P_hi in columns [0,64) and the
// rounding residual P_lo in [64,128) of S_t, and issue a second PV MMA.
#include <climits>
#include <cmath>
#include <type_traits>

#include "ra_internal.cuh"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr float kRescaleThreshold = 8.0f;
// A row also takes its tile max as the exact shift when a key of the tile
// would hold more than 1 / (kDominance + 1) of the row's weight so far: that
// key's P is then exactly 1, and no single rounded bf16 P carries a large
// share of the row (peaked attention on the plain path).
constexpr float kDominance = 8.0f;
// Causal block step in two launches: a query tile whose key range also has
// tiles under the mask moves its fully seen leading tiles to the unmasked
// launch only when there are at least this many.
constexpr int kMinPrefixTiles = 32;
// block mode, causal: words of the CTA's keep bits (then as many mask bits)
constexpr int kBitWords = kBlockKeyTiles / 32;
constexpr unsigned int kFull = 0xffffffffu;

template <int D, int NQ>
struct FwdCfg {
  static constexpr int kHalves = D / 64;          // 64-column (128-byte) swizzle atoms per row
  static constexpr int kHalfBytes = kTile * 128;  // 128 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kKSt = 2;
  static constexpr int kVSt = 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NQ * kTileBytes;
  static constexpr int kVOff = kKOff + kKSt * kTileBytes;
  static constexpr int kBarOff = kVOff + kVSt * kTileBytes;
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;
  static constexpr int bKEmpty = bKFull + kKSt;
  static constexpr int bVFull = bKEmpty + kKSt;
  static constexpr int bVEmpty = bVFull + kVSt;
  static constexpr int bSFull = bVEmpty + kVSt;
  static constexpr int bPReady = bSFull + NQ;
  static constexpr int bODone = bPReady + NQ;
  static constexpr int bDrain = bODone + NQ;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // block mode, causal: keep / mask bits of the CTA's key tiles (16 KB),
  // classified once by the whole CTA
  static constexpr int kBitsOff = kMiscOff + 16;
  static constexpr int kSmemBytes = kBitsOff + 2 * kBitWords * 4;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory layout too large");
  static constexpr int kSoftmaxWarps = 4 * NQ;
  static constexpr int kProducerWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  // NQ = 2: three full warpgroups (the last holds the producer, the MMA
  // issuer and two idle warps) so registers can be re-split per warpgroup:
  // 168 per thread at launch = 2 x 128 x 208 (softmax) + 128 x 88 (rest).
  static constexpr bool kResplit = NQ == 2;
  static constexpr int kThreads = kResplit ? 384 : (kSoftmaxWarps + 2) * 32;
  static constexpr int kLaunchRegs = 168;
  static constexpr int kSoftmaxRegs = 208;
  static constexpr int kOtherRegs = 88;
  static_assert(!kResplit || 128 * (2 * kSoftmaxRegs + kOtherRegs) == kThreads * kLaunchRegs,
                "register re-split must use exactly the launch pool");
  static constexpr uint32_t kTmemCols = NQ == 2 ? 512u : 256u;
  static constexpr uint32_t kOCol0 = NQ * 128u;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
};

// Error sites recorded with a timeout (role * 16 + wait index).
enum : unsigned int {
  kSiteProdK = 0x11, kSiteProdV = 0x12,
  kSiteMmaQ = 0x21, kSiteMmaK = 0x22, kSiteMmaV = 0x23, kSiteMmaP = 0x24,
  kSiteSmS = 0x31, kSiteSmO = 0x32,
};

struct Unit {
  int bb, kh, pr, i, a;
  int qmin, qmax;  // token positions of the tile's first and last existing row
  int kc0, kc1;    // block mode: key tiles [kc0, kc1) of this CTA's key split
  // ring mode: key positions some row of the tile sees form [wlo, whi]; keys
  // in [flo, fhi] are seen by every row; minvis = fewest keys any row sees
  int wlo, whi, flo, fhi, minvis;
  // block mode, causal: the CTA's keep bits (kBitWords words) and then its
  // mask bits in shared memory
  const uint32_t *kbits;
  // block mode, first launch of a two-launch causal step: the tile after the
  // fully seen ones, masked by position in that launch (-1: none)
  int kbound;
};

// Work-unit order: groups of (batch, kv head, query shard); inside a group the
// query tiles run from the last (most key tiles under a causal mask) to the
// first, so concurrently resident CTAs walk the same shards of the same KV
// head (L2 reuse) and long units start first.
__device__ __forceinline__ Unit decode_unit(const FwdParams &p, long long u) {
  Unit x;
  const long long per_group = static_cast<long long>(p.n_qtiles) * p.pairs;
  const long long grp = u / per_group;
  const int w = static_cast<int>(u % per_group);
  x.a = p.n_qtiles - 1 - w / p.pairs;
  x.pr = w % p.pairs;
  x.i = static_cast<int>(grp % p.N);
  const long long g2 = grp / p.N;
  x.kh = static_cast<int>(g2 % p.n_kv);
  x.bb = static_cast<int>(g2 / p.n_kv);
  x.qmin = 0;
  x.qmax = 0;
  x.kbits = nullptr;
  x.kbound = -1;
  // block mode with a key split: blockIdx.y selects split_tiles key tiles
  x.kc0 = p.split_tiles > 0 ? static_cast<int>(blockIdx.y) * p.split_tiles : 0;
  x.kc1 = p.split_tiles > 0 ? min(p.n_ktiles, x.kc0 + p.split_tiles) : p.n_ktiles;
  return x;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Token positions covered by the unit's query tile.  Warp-collective in
// block mode (positions come from q_pos).
template <bool kBlock, bool kDocs, bool kBNc>
__device__ __forceinline__ void unit_qrange(const FwdParams &p, Unit &x) {
  const int r0 = x.a * kTile;
  const int r1 = min(r0 + kTile, p.L) - 1;
  if constexpr (!kBlock) {
    x.qmin = token_at(p.layout, p.L, p.N, x.i, r0);
    x.qmax = token_at(p.layout, p.L, p.N, x.i, r1);
    if constexpr (!kDocs) {
      x.minvis = p.causal ? x.qmin + 1 : p.S;
      return;
    }
    // Rows are increasing positions and document starts do not decrease
    // with the position, so the tile's windows follow from its first and
    // last rows.
    int ds0, de0, ds1, de1;
    doc_of(p.cu, p.n_docs, x.bb, p.S, x.qmin, ds0, de0);
    doc_of(p.cu, p.n_docs, x.bb, p.S, x.qmax, ds1, de1);
    x.wlo = ds0;
    x.whi = p.causal ? x.qmax : de1 - 1;
    x.flo = ds1;
    x.fhi = p.causal ? x.qmin : de0 - 1;
    if (p.causal)
      x.minvis = ds1 > x.qmin ? 1 : x.qmin - ds0 + 1;  // a document starting inside: 1
    else
      x.minvis = de0 < ds1 ? 1 : min(de0 - ds0, de1 - ds1);  // a whole document inside: short
    return;
  }
  int lo = INT_MAX, hi = INT_MIN;
  if (!kBNc && p.causal) {
    for (int r = r0 + (threadIdx.x & 31); r <= r1; r += 32) {
      const int v = p.q_pos[r];
      lo = min(lo, v);
      hi = max(hi, v);
    }
    lo = warp_min(lo);
    hi = warp_max(hi);
  }
  x.qmin = lo;
  x.qmax = hi;
}

struct KvIter {
  int s = -1, j = 0, c = 0, c_end = 0, c_fbeg = 0, c_full = 0;
  bool started = false;  // block mode: c set to the split's first tile
};

// Next key/value tile of the unit in ring order.  Returns false at the end.
// `partial` marks tiles that need an element mask (causal diagonal or the
// ragged last tile).  Warp-collective in block mode.
template <bool kBlock, bool kDocs, bool kBNc>
__device__ __forceinline__ bool kv_next(const FwdParams &p, const Unit &x, KvIter &it, int &j,
                                        int &c, bool &partial) {
  const int n_complete = p.Lk / kTile;
  if constexpr (!kBlock) {
    while (it.c >= it.c_end) {
      if (++it.s >= p.N) return false;
      it.j = kv_shard_at(x.i, it.s, p.N);
      if constexpr (kDocs) {
        // Shard rows are increasing positions, so the keys some row sees are
        // the rows [lo, lim] of the shard and those every row sees
        // [flo, limf].
        const int lo = max(0, first_row_at_or_after(p.layout, p.L, p.N, it.j, x.wlo));
        const int lim = last_visible_row(p.layout, p.L, p.N, it.j, x.whi);
        const int flo = max(0, first_row_at_or_after(p.layout, p.L, p.N, it.j, x.flo));
        const int limf = last_visible_row(p.layout, p.L, p.N, it.j, x.fhi);
        it.c = lo >= p.L ? p.n_ktiles : lo / kTile;
        it.c_end = lim < 0 ? 0 : min(p.n_ktiles, lim / kTile + 1);
        it.c_fbeg = (flo + kTile - 1) / kTile;
        it.c_full = limf < kTile - 1 ? 0 : min(n_complete, (limf - (kTile - 1)) / kTile + 1);
        it.c_full = min(it.c_full, it.c_end);
      } else {
        it.c = 0;
        it.c_fbeg = 0;
        if (!p.causal) {
          it.c_end = p.n_ktiles;
          it.c_full = n_complete;
        } else {
          // keys visible to the latest query form a prefix [0, lim] of the
          // shard; keys visible to the earliest query form [0, limf].
          const int lim = last_visible_row(p.layout, p.L, p.N, it.j, x.qmax);
          const int limf = last_visible_row(p.layout, p.L, p.N, it.j, x.qmin);
          it.c_end = lim < 0 ? 0 : min(p.n_ktiles, lim / kTile + 1);
          it.c_full = limf < kTile - 1 ? 0 : min(n_complete, (limf - (kTile - 1)) / kTile + 1);
          it.c_full = min(it.c_full, it.c_end);
        }
      }
    }
    j = it.j;
    c = it.c;
    partial = it.c < it.c_fbeg || it.c >= it.c_full;
    ++it.c;
    return true;
  } else {
    if (!it.started) {  // first call: start at the split's first tile
      it.c = x.kc0;
      it.started = true;
    }
    if (kBNc || !p.causal) {
      if (it.c >= x.kc1) return false;
      c = it.c++;
      j = 0;
      partial = c >= n_complete || c == x.kbound;
      return true;
    } else {
      // classified once per CTA: bit t for tile kc0 + t
      const int nt = min(x.kc1 - x.kc0, kBlockKeyTiles);
      int t = it.c - x.kc0;
      while (t < nt) {
        const uint32_t w = x.kbits[t >> 5] >> (t & 31);
        if (w != 0) {
          t += __ffs(w) - 1;
          break;
        }
        t = (t | 31) + 1;
      }
      if (t >= nt) {
        it.c = x.kc1;
        return false;
      }
      c = x.kc0 + t;
      j = 0;
      partial = (x.kbits[kBitWords + (t >> 5)] >> (t & 31)) & 1u;
      it.c = c + 1;
      return true;
    }
  }
}

// Block mode: how many key tiles of [kc0, kc1), counted from kc0, every row
// of query tile a sees in full -- complete tiles whose key positions are all
// <= the tile's smallest query position (any positions, sorted or not).
// Warp w walks tiles kc0 + w, kc0 + w + nw, ... eight at a time (one 16-byte
// load per lane and tile when k_pos is 16-byte aligned) and stops at its
// first tile that fails; the prefix ends at the smallest of those.
// Block-collective; `scratch` holds 128 ints.
template <bool kVec>
__device__ __forceinline__ int first_failing_tile(const FwdParams &p, int kc0, int kc1, int qmin,
                                                  int warp, int lane, int nw) {
  constexpr int kBatch = 8;
  const int n_complete = p.Lk / kTile;
  int first = kc1;
  for (int c = kc0 + warp; c < kc1 && first == kc1; c += kBatch * nw) {
    int hi[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int t = c + u * nw;
      hi[u] = INT_MIN;
      if (t < kc1 && t < n_complete) {
        const int32_t *kp = p.k_pos + static_cast<size_t>(t) * kTile;
        if constexpr (kVec) {
          const int4 v4 = __ldg(reinterpret_cast<const int4 *>(kp) + lane);
          hi[u] = max(max(v4.x, v4.y), max(v4.z, v4.w));
        } else {
#pragma unroll
          for (int e = 0; e < kTile / 32; ++e) hi[u] = max(hi[u], __ldg(kp + e * 32 + lane));
        }
      } else if (t < kc1) {
        hi[u] = INT_MAX;  // the ragged last tile is masked
      }
    }
#pragma unroll
    for (int u = kBatch - 1; u >= 0; --u)
      if (__any_sync(kFull, hi[u] > qmin)) first = c + u * nw;
  }
  return first;
}

// Whether some key tile of [t0, kc1) has a key that a row of the query tile
// (latest position qmax) sees; warp-parallel like first_failing_tile, each
// warp stopping at its first such tile.
template <bool kVec>
__device__ __forceinline__ bool any_visible_tile(const FwdParams &p, int t0, int kc1, int qmax,
                                                 int warp, int lane, int nw) {
  constexpr int kBatch = 8;
  bool found = false;
  for (int c = t0 + warp; c < kc1 && !found; c += kBatch * nw) {
    int lo[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int t = c + u * nw;
      lo[u] = INT_MAX;
      if (t < kc1) {
        const int32_t *kp = p.k_pos + static_cast<size_t>(t) * kTile;
        if (kVec && (t + 1) * kTile <= p.Lk) {
          const int4 v4 = __ldg(reinterpret_cast<const int4 *>(kp) + lane);
          lo[u] = min(min(v4.x, v4.y), min(v4.z, v4.w));
        } else {
#pragma unroll
          for (int e = 0; e < kTile / 32; ++e)
            if (t * kTile + e * 32 + lane < p.Lk) lo[u] = min(lo[u], __ldg(kp + e * 32 + lane));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) found |= __any_sync(kFull, lo[u] <= qmax);
  }
  return found;
}

// The leading fully seen tiles (returned, counted from kc0) and, when
// `want_tail`, whether a key after the first tile that is not fully seen is
// visible to some row of the tile (tail_vis; left true otherwise).
__device__ __noinline__ int full_prefix_tiles(const FwdParams &p, int a, int kc0, int kc1,
                                              int *scratch, bool want_tail, bool &tail_vis) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int r1 = min((a + 1) * kTile, p.L);
  int qmin = INT_MAX, qmax = INT_MIN;
  for (int r = a * kTile + static_cast<int>(threadIdx.x); r < r1; r += blockDim.x) {
    const int v = __ldg(p.q_pos + r);
    qmin = min(qmin, v);
    qmax = max(qmax, v);
  }
  qmin = warp_min(qmin);
  qmax = warp_max(qmax);
  if (lane == 0) {
    scratch[warp] = qmin;
    scratch[32 + warp] = qmax;
  }
  __syncthreads();
  qmin = INT_MAX;
  qmax = INT_MIN;
  for (int w = 0; w < nw; ++w) {
    qmin = min(qmin, scratch[w]);
    qmax = max(qmax, scratch[32 + w]);
  }
  const bool vec = (reinterpret_cast<uintptr_t>(p.k_pos) & 15u) == 0;
  const int first = vec ? first_failing_tile<true>(p, kc0, kc1, qmin, warp, lane, nw)
                        : first_failing_tile<false>(p, kc0, kc1, qmin, warp, lane, nw);
  __syncthreads();  // every warp has read qmin / qmax
  if (lane == 0) scratch[64 + warp] = first;
  __syncthreads();
  int f = kc1;
  for (int w = 0; w < nw; ++w) f = min(f, scratch[64 + w]);
  tail_vis = true;
  if (want_tail) {
    const bool any = vec ? any_visible_tile<true>(p, f + 1, kc1, qmax, warp, lane, nw)
                         : any_visible_tile<false>(p, f + 1, kc1, qmax, warp, lane, nw);
    __syncthreads();  // every warp has read the firsts
    if (lane == 0) scratch[96 + warp] = any ? 1 : 0;
    __syncthreads();
    int v = 0;
    for (int w = 0; w < nw; ++w) v |= scratch[96 + w];
    tail_vis = v != 0;
  }
  __syncthreads();  // scratch is free again
  return f - kc0;
}

template <int D>
__device__ __forceinline__ void issue_s_mma(uint32_t tS, uint32_t q_saddr, uint32_t k_saddr,
                                            uint32_t idesc) {
  // S = Q K^T: A = Q (128 x D, K-major), B = K (128 keys x D, K-major).
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
    mma_ss(tS, smem_desc_sw128(q_saddr + off, 16, 1024), smem_desc_sw128(k_saddr + off, 16, 1024),
           idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv_mma(uint32_t tO, uint32_t tP, uint32_t v_saddr,
                                             uint32_t idesc, bool accumulate) {
  // O (+)= P V: A = P from TMEM (128 x 128 bf16, 2 per column),
  // B = V (128 keys x D, MN-major: 64-column atoms 16 KB apart, 8-key
  // groups 1 KB apart; 16 keys per instruction).
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk) {
    mma_ts(tO, tP + kk * 8, smem_desc_sw128(v_saddr + kk * 16 * 128, kTile * 128, 1024), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

// P = 2^(s * c - shift) for one 128-key row: writes P (bf16 pairs) to TMEM
// columns [0,64) -- and with kSplit the rounding residual to [64,128) --
// and accumulates the fp32 row sum into four paired accumulators.
template <bool kSplit>
__device__ __forceinline__ void exp_pack_store(const float (&s)[kTile], uint64_t sl2x2,
                                               uint64_t nbx2, uint64_t (&acc)[4], uint32_t tS) {
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = f2pack(0.f, 0.f);
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t pk[16];
    uint32_t lo[kSplit ? 16 : 1];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int cc = q4 * 32 + 2 * e;
      float x0, x1;
      f2unpack(ffma2(f2pack(s[cc], s[cc + 1]), sl2x2, nbx2), x0, x1);
      const float p0 = ex2(x0);
      const float p1 = ex2(x1);
      acc[e & 3] = fadd2(acc[e & 3], f2pack(p0, p1));
      pk[e] = pack_bf16x2(p0, p1);
      if constexpr (kSplit)
        lo[e] = pack_bf16x2(p0 - __uint_as_float(pk[e] << 16),
                            p1 - __uint_as_float(pk[e] & 0xffff0000u));
    }
    tmem_st16(tS + q4 * 16, pk);
    if constexpr (kSplit) tmem_st16(tS + 64 + q4 * 16, lo);
  }
}

template <int D, int NQ, bool kBlock, bool kDocs, bool kBNc>
__global__ void __launch_bounds__(FwdCfg<D, NQ>::kThreads, 1)
    fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using C = FwdCfg<D, NQ>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  int fp = 0;  // two-launch causal step: leading key tiles seen in full
  if constexpr (kBlock) {
    // a prefill pass that covers only part of each query tile's key range:
    // nothing to do when this CTA's split lies outside it
    if (p.kt_end != nullptr || p.kt_begin != nullptr) {
      const Unit y = decode_unit(p, blockIdx.x);
      int kc0 = y.kc0, kc1 = y.kc1;
      if (p.kt_end != nullptr) kc1 = min(kc1, __ldg(p.kt_end + y.a));
      if (p.kt_begin != nullptr) kc0 = max(kc0, __ldg(p.kt_begin + y.a));
      if (kc0 >= kc1) return;
    }
    if (p.full_prefix != 0) {
      const Unit y = decode_unit(p, blockIdx.x);
      bool tail_vis = true;
      fp = full_prefix_tiles(p, y.a, y.kc0, y.kc1, reinterpret_cast<int *>(smem + C::kBitsOff),
                             p.full_prefix == 2, tail_vis);
      // a CTA with work in both launches pays a second start and state
      // merge, which a short prefix does not earn back: it stays whole
      if (fp < y.kc1 - y.kc0 && fp < kMinPrefixTiles) fp = 0;
      // the first launch also takes the tile after the prefix, masked by
      // position: on a ring step that is the diagonal tile, and the second
      // launch is left with nothing
      if (p.full_prefix == 1 ? fp == 0 : (fp > 0 && (y.kc0 + fp + 1 >= y.kc1 || !tail_vis)))
        return;
    }
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);

  if (threadIdx.x == 0) {
    mbar_init(&bars[C::bQFull], 1);
    for (int s = 0; s < C::kKSt; ++s) {
      mbar_init(&bars[C::bKFull + s], 1);
      mbar_init(&bars[C::bKEmpty + s], 1);
    }
    for (int s = 0; s < C::kVSt; ++s) {
      mbar_init(&bars[C::bVFull + s], 1);
      mbar_init(&bars[C::bVEmpty + s], 1);
    }
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&bars[C::bSFull + t], 1);
      mbar_init(&bars[C::bPReady + t], 4);
      mbar_init(&bars[C::bODone + t], 1);
    }
    mbar_init(&bars[C::bDrain], 1);
    *abort_flag = 0;
    *reinterpret_cast<int *>(smem + C::kMiscOff + 8) = 0;  // block mode: visible-key count
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

  Unit x = decode_unit(p, blockIdx.x);
  // the first key tile of the CTA's whole range (a second launch of a
  // causal step starts later but takes its precision mode from all of it)
  int kc_all = x.kc0;
  if constexpr (kBlock) {
    if (p.kt_end != nullptr) x.kc1 = min(x.kc1, __ldg(p.kt_end + x.a));
    if (p.kt_begin != nullptr) x.kc0 = max(x.kc0, __ldg(p.kt_begin + x.a));
    kc_all = x.kc0;
    if (p.full_prefix == 1) {
      x.kc1 = min(x.kc1, x.kc0 + fp + 1);
      if (x.kc0 + fp < x.kc1) x.kbound = x.kc0 + fp;
    }
    if (p.full_prefix == 2 && fp > 0) x.kc0 += fp + 1;
  }
  unit_qrange<kBlock, kDocs, kBNc>(p, x);
  // Rows that see fewer than kSplitKeys keys take the hi + lo path.  On the
  // ring a row at position t sees t + 1 keys.  A block step counts, over the
  // CTA's key range, the keys its earliest query sees (every row of the tile
  // sees at least those).
  bool split;
  if constexpr (!kBlock) {
    split = x.minvis < kSplitKeys;
  } else {
    const int k0 = kc_all * kTile, k1 = min(p.Lk, x.kc1 * kTile);
    const int nt = x.kc1 - x.kc0;
    if (!kBNc && p.causal) {
      int *cnt = reinterpret_cast<int *>(smem + C::kMiscOff + 8);
      // Classify the CTA's key tiles once, a warp per tile: keep a tile
      // when a key precedes the unit's last query, mask it when a key
      // follows the first query (or the tile is ragged); count on the way
      // the keys every query sees.
      uint32_t *bits = reinterpret_cast<uint32_t *>(smem + C::kBitsOff);
      for (int w = threadIdx.x; w < 2 * kBitWords; w += blockDim.x) bits[w] = 0;
      __syncthreads();
      const int n_complete = p.Lk / kTile;
      int mine = 0;
      for (int t = warp; t < min(nt, kBlockKeyTiles); t += blockDim.x >> 5) {
        const int tile = x.kc0 + t;
        int lo = INT_MAX, hi = INT_MIN;
#pragma unroll
        for (int e = 0; e < kTile / 32; ++e) {
          const int kr = tile * kTile + e * 32 + lane;
          if (kr < p.Lk) {
            const int v = p.k_pos[kr];
            lo = min(lo, v);
            hi = max(hi, v);
            mine += v <= x.qmin ? 1 : 0;
          }
        }
        lo = warp_min(lo);
        hi = warp_max(hi);
        if (lane == 0 && lo <= x.qmax) {
          atomicOr(&bits[t >> 5], 1u << (t & 31));
          if (tile >= n_complete || hi > x.qmin) atomicOr(&bits[kBitWords + (t >> 5)], 1u << (t & 31));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(kFull, mine, o);
      if (lane == 0) atomicAdd(cnt, mine);
      __syncthreads();
      // keys of the fully seen tiles a first launch took (a lower bound)
      split = k1 - k0 < kSplitKeys || *cnt + fp * kTile < kSplitKeys;
      x.kbits = bits;
    } else {
      split = k1 - k0 < kSplitKeys;  // without the causal rule every row sees the range
    }
  }

  if (warp >= C::kSoftmaxWarps) {
    if constexpr (C::kResplit) regs_set<C::kOtherRegs, C::kLaunchRegs>();
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    int c2, c3;
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      mbar_arrive_expect_tx(&bars[C::bQFull], NQ * C::kTileBytes);
      map_coords(p.layout, p.L, p.N, x.i, x.a * kTile, c2, c3);
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        const int hq = x.kh * p.g + x.pr * NQ + t;
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_5d(smem + C::kQOff + t * C::kTileBytes + hf * C::kHalfBytes, &qmap,
                      &bars[C::bQFull], hf * 64, hq, c2, c3, x.bb);
      }
    }
    int k_par[C::kKSt], v_par[C::kVSt];
    for (int s = 0; s < C::kKSt; ++s) k_par[s] = -1;
    for (int s = 0; s < C::kVSt; ++s) v_par[s] = -1;
    KvIter it;
    int j, c, n = 0;
    bool partial;
    while (kv_next<kBlock, kDocs, kBNc>(p, x, it, j, c, partial)) {
      if (lane == 0) {
        map_coords(p.layout, p.L, p.N, j, c * kTile, c2, c3);
        const int ks = n % C::kKSt;
        const uint32_t kph = (n / C::kKSt) & 1;
        if (mbar_wait(&bars[C::bKEmpty + ks], kph ^ 1, abort_flag, kSiteProdK)) {
          mbar_arrive_expect_tx(&bars[C::bKFull + ks], C::kTileBytes);
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_5d(smem + C::kKOff + ks * C::kTileBytes + hf * C::kHalfBytes, &kmap,
                        &bars[C::bKFull + ks], hf * 64, x.kh, c2, c3, x.bb);
          k_par[ks] = static_cast<int>(kph);
          const int vs = n % C::kVSt;
          const uint32_t vph = (n / C::kVSt) & 1;
          if (mbar_wait(&bars[C::bVEmpty + vs], vph ^ 1, abort_flag, kSiteProdV)) {
            mbar_arrive_expect_tx(&bars[C::bVFull + vs], C::kTileBytes);
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_5d(smem + C::kVOff + vs * C::kTileBytes + hf * C::kHalfBytes, &vmap,
                          &bars[C::bVFull + vs], hf * 64, x.kh, c2, c3, x.bb);
            v_par[vs] = static_cast<int>(vph);
          }
        }
      }
      __syncwarp();
      if (*abort_flag) break;
      ++n;
    }
    if (lane == 0 && *abort_flag) {
      // Let every copy this warp started land before the CTA unwinds.
      mbar_wait_budget(&bars[C::bQFull], 0, kWaitBudgetCycles);
      for (int s = 0; s < C::kKSt; ++s)
        if (k_par[s] >= 0) mbar_wait_budget(&bars[C::bKFull + s], k_par[s], kWaitBudgetCycles);
      for (int s = 0; s < C::kVSt; ++s)
        if (v_par[s] >= 0) mbar_wait_budget(&bars[C::bVFull + s], v_par[s], kWaitBudgetCycles);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&bars[C::bQFull], 0, abort_flag, kSiteMmaQ);
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
    if (ok) {
      tc_fence_after();
      const uint32_t q_saddr = sbase + C::kQOff;
      const uint32_t k_saddr = sbase + C::kKOff;
      const uint32_t v_saddr = sbase + C::kVOff;
      KvIter it;
      int j, c, n = 0;
      bool partial;
      bool has = kv_next<kBlock, kDocs, kBNc>(p, x, it, j, c, partial);
      if (has && lane == 0) {
        if (mbar_wait(&bars[C::bKFull + 0], 0, abort_flag, kSiteMmaK)) {
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            issue_s_mma<D>(tmem + t * 128, q_saddr + t * C::kTileBytes, k_saddr, C::kIdescS);
            mma_commit(&bars[C::bSFull + t]);
          }
          mma_commit(&bars[C::bKEmpty + 0]);
        }
      }
      __syncwarp();
      while (has && !*abort_flag) {
        const bool has_next = kv_next<kBlock, kDocs, kBNc>(p, x, it, j, c, partial);
        if (lane == 0) {
          const int vs = n % C::kVSt;
          const uint32_t vph = (n / C::kVSt) & 1;
          const int ks = (n + 1) % C::kKSt;
          const uint32_t kph = ((n + 1) / C::kKSt) & 1;
          bool go = mbar_wait(&bars[C::bVFull + vs], vph, abort_flag, kSiteMmaV);
          if (go) tc_fence_after();
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (!go) break;
            go = mbar_wait(&bars[C::bPReady + t], n & 1, abort_flag, kSiteMmaP);
            if (!go) break;
            tc_fence_after();
            issue_pv_mma<D>(tmem + C::kOCol0 + t * 128, tmem + t * 128,
                            v_saddr + vs * C::kTileBytes, C::kIdescPV, n > 0);
            if (split)
              issue_pv_mma<D>(tmem + C::kOCol0 + t * 128, tmem + t * 128 + 64,
                              v_saddr + vs * C::kTileBytes, C::kIdescPV, true);
            if (t == NQ - 1) mma_commit(&bars[C::bVEmpty + vs]);
            if (has_next) {
              if (t == 0) {
                go = mbar_wait(&bars[C::bKFull + ks], kph, abort_flag, kSiteMmaK);
                if (!go) break;
                tc_fence_after();
              }
              issue_s_mma<D>(tmem + t * 128, q_saddr + t * C::kTileBytes,
                             k_saddr + ks * C::kTileBytes, C::kIdescS);
              mma_commit(&bars[C::bSFull + t]);
              if (t == NQ - 1) mma_commit(&bars[C::bKEmpty + ks]);
            } else {
              mma_commit(&bars[C::bODone + t]);
            }
          }
        }
        __syncwarp();
        ++n;
        has = has_next;
      }
    }
    if (lane == 0) {
      // Every MMA this thread issued has finished before TMEM is released.
      mma_commit(&bars[C::bDrain]);
      mbar_wait_budget(&bars[C::bDrain], 0, kWaitBudgetCycles);
    }
    __syncwarp();
  }
  } else {
    if constexpr (C::kResplit) regs_set<C::kSoftmaxRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // TMEM lane == tile row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + C::kOCol0 + t * 128;
    const int hq = x.kh * p.g + x.pr * NQ + t;
    const int r_abs = x.a * kTile + row;
    const bool row_exists = r_abs < p.L;
    const int r_cl = row_exists ? r_abs : p.L - 1;
    const int qp = kBlock ? ((!kBNc && p.causal) || (kBNc && x.kbound >= 0) ? p.q_pos[r_cl] : 0)
                                : token_at(p.layout, p.L, p.N, x.i, r_cl);
    // ring mode: this row sees key positions [q_wlo, q_whi]
    int q_wlo = 0, q_whi = 0;
    if constexpr (kDocs) key_window(p.cu, p.n_docs, x.bb, p.S, p.causal, qp, q_wlo, q_whi);
    const float sl2 = p.scale_log2;

    float m_run = -INFINITY;  // exponent shift (log2 units of the scaled logits)
    float m_max = -INFINITY;  // exact running row max (same units)
    float l_sum = 0.f;
    KvIter it;
    int j, c, n = 0;
    bool partial;
    bool aborted = false;
    // One copy of the tile loop per precision mode, chosen once per unit, so
    // the hot loop carries no branch on it.
    auto tile_loop = [&](auto split_tag) {
    constexpr bool kSplit = decltype(split_tag)::value;
    while (kv_next<kBlock, kDocs, kBNc>(p, x, it, j, c, partial)) {
      const bool got = mbar_wait(&bars[C::bSFull + t], n & 1, abort_flag, kSiteSmS);
      if (!__all_sync(kFull, got)) {  // tcgen05.ld/st below are warp-collective
        aborted = true;
        break;
      }
      tc_fence_after();
      uint32_t sr[kTile];
      tmem_ld128(tS, sr);
      float s[kTile];
#pragma unroll
      for (int e = 0; e < kTile; ++e) s[e] = __uint_as_float(sr[e]);
      if (partial) {
        if constexpr (!kBlock) {
          if constexpr (kDocs) {
            const int lim = min(p.Lk - 1, last_visible_row(p.layout, p.L, p.N, j, q_whi));
            const int lo = first_row_at_or_after(p.layout, p.L, p.N, j, q_wlo);
            const int climit = lim - c * kTile;
            const int cbase = lo - c * kTile;
#pragma unroll
            for (int e = 0; e < kTile; ++e)
              if (e > climit || e < cbase) s[e] = -INFINITY;
          } else {
            int lim = p.Lk - 1;
            if (p.causal) lim = min(lim, last_visible_row(p.layout, p.L, p.N, j, qp));
            const int climit = lim - c * kTile;
#pragma unroll
            for (int e = 0; e < kTile; ++e)
              if (e > climit) s[e] = -INFINITY;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kTile; ++e) {
            const int kr = c * kTile + e;
            const bool vis =
                kr < p.Lk && (kBNc ? (c != x.kbound || __ldg(p.k_pos + kr) <= qp)
                                   : (!p.causal || __ldg(p.k_pos + kr) <= qp));
            if (!vis) s[e] = -INFINITY;
          }
        }
      }
      // row max as eight short 3-input-max chains, then a small tree
      auto row_max = [&]() {
        float pm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = s[k];
#pragma unroll
        for (int e = 8; e + 16 <= kTile; e += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) pm[k] = fmax3(pm[k], s[e + k], s[e + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = fmaxf(pm[k], s[kTile - 8 + k]);
        return fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]),
                     fmaxf(pm[6], pm[7]));
      };
      // O_t row *= alpha.  The previous PV into O_t is complete: it was
      // issued before this tile's S MMA, whose commit we waited on.
      auto rescale_o = [&](float alpha) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tO + ch * 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tO + ch * 32, r);
        }
      };
      // P = 2^(s * scale * log2 e - shift): paired FMAs, four paired sums
      const uint64_t sl2x2 = f2pack(sl2, sl2);
      uint64_t acc[4];
      // When every row of the warp already has a shift, P is formed against
      // it while the row max is computed alongside; a row whose max passed
      // its shift by more than the threshold (rare after the first tiles)
      // takes a new shift and the warp forms the tile's P again.
      bool spec = __all_sync(kFull, m_run != -INFINITY);
      // a new shift: the max passed the old one by more than the threshold,
      // or by less but with a key that would dominate the row's sum so far
      auto needs_shift = [&](float mx2) {
        return mx2 > m_run + kRescaleThreshold ||
               (mx2 > m_run && ex2(mx2 - m_run) * kDominance > l_sum);
      };
      if (!spec) {
        const float mx2 = row_max() * sl2;
        m_max = fmaxf(m_max, mx2);
        const bool need = needs_shift(mx2);
        float alpha = 1.f;
        if (need) {
          alpha = ex2(m_run - mx2);  // 0 when m_run is still -inf
          m_run = mx2;
        }
        if (n > 0 && __any_sync(kFull, need)) rescale_o(alpha);
        l_sum *= alpha;
      }
      for (;;) {
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        exp_pack_store<kSplit>(s, sl2x2, f2pack(-base, -base), acc, tS);
        if (!spec) break;
        spec = false;
        if constexpr (!kBlock) {
          // The ring epilogue needs no exact max: when the tile's P sums to
          // at most min(2^8, l / 8) in the current shift's units, no P
          // passes either bound of needs_shift, and the warp skips the max.
          float b0, b1, b2, b3, b4, b5, b6, b7;
          f2unpack(acc[0], b0, b1);
          f2unpack(acc[1], b2, b3);
          f2unpack(acc[2], b4, b5);
          f2unpack(acc[3], b6, b7);
          const float ts = ((b0 + b1) + (b2 + b3)) + ((b4 + b5) + (b6 + b7));
          if (!__any_sync(kFull, ts > fminf(256.f, l_sum * (1.f / kDominance)))) break;
        }
        const float mx2 = row_max() * sl2;
        m_max = fmaxf(m_max, mx2);
        const bool need = needs_shift(mx2);
        if (!__any_sync(kFull, need)) break;
        float alpha = 1.f;
        if (need) {
          alpha = ex2(m_run - mx2);
          m_run = mx2;
        }
        rescale_o(alpha);
        l_sum *= alpha;
        tmem_st_wait();  // the first P stores have landed before they are overwritten
      }
      float a0, a1, a2, a3, a4, a5, a6, a7;
      f2unpack(acc[0], a0, a1);
      f2unpack(acc[1], a2, a3);
      f2unpack(acc[2], a4, a5);
      f2unpack(acc[3], a6, a7);
      l_sum += ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::bPReady + t]);
      ++n;
    }
    };
    if (split)
      tile_loop(std::true_type{});
    else
      tile_loop(std::false_type{});

    // ------------------------------------------------------------ epilogue
    bool have_o = n > 0 && !aborted;
    if (have_o) {
      if (!mbar_wait(&bars[C::bODone + t], 0, abort_flag, kSiteSmO)) have_o = false;
      tc_fence_after();
    }
    have_o = __all_sync(kFull, have_o && *abort_flag == 0);
    if constexpr (!kBlock) {
      const int tok = token_at(p.layout, p.L, p.N, x.i, r_cl);
      const size_t orow = ((static_cast<size_t>(x.bb) * p.S + tok) * p.h + hq) * D;
      const bool live = have_o && l_sum > 0.f;
      const float inv_l = live ? 1.f / l_sum : 0.f;
      if (row_exists && !*abort_flag)
        p.lse[(static_cast<size_t>(x.bb) * p.h + hq) * p.S + tok] =
            live ? (m_run + log2f(l_sum)) * kLn2 : -INFINITY;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        if (have_o) tmem_ld32(tO + ch * 32, r);
        if (row_exists && !*abort_flag) {
          float4 *dst = reinterpret_cast<float4 *>(p.out + orow + ch * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float4 v4;
            v4.x = live ? __uint_as_float(r[4 * e + 0]) * inv_l : 0.f;
            v4.y = live ? __uint_as_float(r[4 * e + 1]) * inv_l : 0.f;
            v4.z = live ? __uint_as_float(r[4 * e + 2]) * inv_l : 0.f;
            v4.w = live ? __uint_as_float(r[4 * e + 3]) * inv_l : 0.f;
            dst[e] = v4;
          }
        }
      }
    } else {
      // Fold the block result (shift m_run, sum l_sum, numerator in TMEM)
      // into the caller's state, re-referenced to the exact running max.
      // with a key split, each split folds into its own state slice
      const size_t z = p.split_tiles > 0 ? blockIdx.y : 0;
      const size_t si = z * p.b * p.h * static_cast<size_t>(p.L) +
                        (static_cast<size_t>(x.bb) * p.h + hq) * p.L + r_cl;
      const size_t oi = z * p.b * p.h * static_cast<size_t>(p.L) * D +
                        ((static_cast<size_t>(x.bb) * p.L + r_cl) * p.h + hq) * D;
      const float m_old2 = row_exists ? p.st_m[si] * kLog2e : -INFINITY;
      const float M = fmaxf(m_old2, have_o ? m_max : -INFINITY);
      const bool write = row_exists && !*abort_flag && have_o && M != -INFINITY;
      const float a_old = (m_old2 == -INFINITY) ? 0.f : ex2(m_old2 - M);
      const float a_blk = (!have_o || m_run == -INFINITY) ? 0.f : ex2(m_run - M);
      if (write) {
        p.st_l[si] = p.st_l[si] * a_old + l_sum * a_blk;
        p.st_m[si] = M * kLn2;
      }
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        if (have_o) tmem_ld32(tO + ch * 32, r);
        if (write) {
          float4 *dst = reinterpret_cast<float4 *>(p.st_o + oi + ch * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float4 v4 = dst[e];
            v4.x = v4.x * a_old + __uint_as_float(r[4 * e + 0]) * a_blk;
            v4.y = v4.y * a_old + __uint_as_float(r[4 * e + 1]) * a_blk;
            v4.z = v4.z * a_old + __uint_as_float(r[4 * e + 2]) * a_blk;
            v4.w = v4.w * a_old + __uint_as_float(r[4 * e + 3]) * a_blk;
            dst[e] = v4;
          }
        }
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

template <int D, int NQ, bool kBlock, bool kDocs = false>
cudaError_t launch_fwd_t(const FwdParams &p, const CUtensorMap &qmap, const CUtensorMap &kmap,
                         const CUtensorMap &vmap, long long n_units, cudaStream_t stream) {
  using C = FwdCfg<D, NQ>;
  // A block step without the causal rule runs an instantiation that has no
  // causal code at all: the position classification and masks of the causal
  // one made the same non-causal work 20 % slower (1211 against 1458 useful
  // TFLOP/s at 64K x 64K).  Causal block steps keep the general one.
  auto kern = fwd_kernel<D, NQ, kBlock, kDocs, false>;
  if constexpr (kBlock) {
    if (!p.causal) kern = fwd_kernel<D, NQ, kBlock, kDocs, true>;
  }
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  if (e != cudaSuccess) return e;
  if constexpr (C::kResplit) {
    // The register increase in the kernel waits until the pool covers it.
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    // The re-split assumes each warpgroup starts from exactly kLaunchRegs.
    if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  }
  const unsigned int splits = (kBlock && p.split_tiles > 0)
                                  ? static_cast<unsigned int>((p.n_ktiles + p.split_tiles - 1) /
                                                              p.split_tiles)
                                  : 1u;
  kern<<<dim3(static_cast<unsigned int>(n_units), splits), dim3(C::kThreads), C::kSmemAlloc,
         stream>>>(
      p, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdParams &p, int d, int nq, const CUtensorMap &qmap,
                       const CUtensorMap &kmap, const CUtensorMap &vmap, long long n_units,
                       cudaStream_t stream) {
  if (n_units <= 0) return cudaSuccess;
  const bool blk = p.block_mode != 0;
  const bool docs = !blk && p.cu != nullptr;
  if (d == 128 && nq == 2)
    return blk ? launch_fwd_t<128, 2, true>(p, qmap, kmap, vmap, n_units, stream)
           : docs ? launch_fwd_t<128, 2, false, true>(p, qmap, kmap, vmap, n_units, stream)
                  : launch_fwd_t<128, 2, false>(p, qmap, kmap, vmap, n_units, stream);
  if (d == 128 && nq == 1)
    return blk ? launch_fwd_t<128, 1, true>(p, qmap, kmap, vmap, n_units, stream)
           : docs ? launch_fwd_t<128, 1, false, true>(p, qmap, kmap, vmap, n_units, stream)
                  : launch_fwd_t<128, 1, false>(p, qmap, kmap, vmap, n_units, stream);
  if (d == 64 && nq == 2)
    return blk ? launch_fwd_t<64, 2, true>(p, qmap, kmap, vmap, n_units, stream)
           : docs ? launch_fwd_t<64, 2, false, true>(p, qmap, kmap, vmap, n_units, stream)
                  : launch_fwd_t<64, 2, false>(p, qmap, kmap, vmap, n_units, stream);
  if (d == 64 && nq == 1)
    return blk ? launch_fwd_t<64, 1, true>(p, qmap, kmap, vmap, n_units, stream)
           : docs ? launch_fwd_t<64, 1, false, true>(p, qmap, kmap, vmap, n_units, stream)
                  : launch_fwd_t<64, 1, false>(p, qmap, kmap, vmap, n_units, stream);
  return cudaErrorInvalidValue;
}

RA_DEFINE_ERROR_WORD_READER(read_error_word_fwd)

}  // namespace ra
