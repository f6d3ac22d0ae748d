// ra_bwd.cu -- blockwise backward of ring attention for sm_103a.
//
// Recomputation backward (the first page's "The Backward Pass and Gradient
// Exchange"; the fourth page's "The Backward Pass: Symmetric Ring
// Operation"): with the saved LSE and D = rowsum(dO * O),
//     P  = exp(S - LSE),      S = scale Q K^T
//     dV_j += P^T dO,         dP = dO V^T,       dS = P * (dP - D)
//     dK_j += scale dS^T Q,   dQ_i += scale dS K
// One CTA owns one 128-key tile of one KV head and keeps K, V in shared
// memory and dK, dV in tensor memory.  Like the key/value block that carries
// its gradient accumulators around the ring, the tile meets the query shards
// in ring order: shard (j + s) mod N at step s, and inside each shard every
// query tile the causal rule does not mask completely, for each of the g
// query heads of its GQA group.  dQ partial tiles are added into the fp32 dq
// output with vector reductions.
//
// Precision: bf16 operands with fp32 accumulation lose up to 2^-9 of each
// product term, which on query rows with few visible keys (large weights)
// reaches the 1e-2 parity budget.  dS is always formed from the fp32 P; on
// steps whose query tile has a row seeing fewer than kSplitKeys keys, P and
// dS also go to the tensor cores as a bf16 pair hi + lo (lo = the rounding
// residual): dV += P_hi^T dO + P_lo^T dO, dK += dS_hi^T Q + dS_lo^T Q,
// dQ = dS_hi K + dS_lo K.
//
// Warp roles (12 warps):
//   warps 0-3  "softmax": thread = key row; P^T = exp2(S^T - LSE2), written to
//              TMEM as bf16 (and its residual on split steps); dS^T =
//              P^T (dP^T - D) to shared memory (residual over the step's dO
//              tile once dV is done with it, on split steps)
//   warps 4-7  dQ drain: TMEM -> registers -> red.global.add.v4.f32; at the
//              end the dK / dV epilogue
//   warp 8     TMA producer: K, V once; Q and dO tiles into a 2-deep ring
//   warp 9     TMEM allocator and MMA issuer (lane 0)
//   warps 10-11 idle
// TMEM columns: S^T then P_hi^T [0,64) + P_lo^T [64,128); dP^T then dQ
// [128,256); dV [256,..); dK [384,..).
// MMAs per step: S^T = K Q^T, dP^T = V dO^T (SS, both K-major);
// dV += P^T dO (A from TMEM, dO MN-major); dK += dS^T Q (dS^T K-major, Q
// MN-major); dQ = dS K (dS^T read MN-major, K MN-major).
#include <climits>
#include <cmath>

#include "ra_internal.cuh"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr unsigned int kFull = 0xffffffffu;

template <int D>
struct BwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kTile * 128;
  static constexpr int kTileBytes = kHalves * kHalfBytes;  // 128 rows x D bf16
  static constexpr int kDsBytes = 2 * kHalfBytes;          // 128 keys x 128 queries bf16
  static constexpr int kQSt = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kDoOff = kQOff + kQSt * kTileBytes;
  static constexpr int kDsOff = kDoOff + kQSt * kTileBytes;
  // dS_lo^T (split steps): over the step's dO tile when that is as large as
  // a dS tile (D = 128), else a buffer of its own.
  static constexpr bool kDsLoInDo = kTileBytes >= kDsBytes;
  static constexpr int kDsLoOff = kDsOff + kDsBytes;
  static constexpr int kBarOff = kDsLoOff + (kDsLoInDo ? 0 : kDsBytes);
  static constexpr int bKV = 0;
  static constexpr int bQFull = 1;
  static constexpr int bQEmpty = bQFull + kQSt;
  static constexpr int bSFull = bQEmpty + kQSt;
  static constexpr int bDpFull = bSFull + 1;
  static constexpr int bPReady = bDpFull + 1;
  static constexpr int bDsReady = bPReady + 1;
  static constexpr int bDsEmpty = bDsReady + 1;
  static constexpr int bDqFull = bDsEmpty + 1;
  static constexpr int bDqEmpty = bDqFull + 1;
  static constexpr int bDvDone = bDqEmpty + 1;
  static constexpr int bDone = bDvDone + 1;
  static constexpr int bDrain = bDone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static constexpr int kThreads = 384;
  // 168 registers per thread at launch = 128 x (232 softmax + 160 dQ drain
  // + 112 producer / MMA) re-split per warpgroup.
  static constexpr int kLaunchRegs = 168;
  static constexpr int kSoftmaxRegs = 232;
  static constexpr int kDrainRegs = 160;
  static constexpr int kOtherRegs = 112;
  static_assert(128 * (kSoftmaxRegs + kDrainRegs + kOtherRegs) == kThreads * kLaunchRegs,
                "register re-split must use exactly the launch pool");
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384;
  static constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t kIdescDv = idesc_bf16_f32(128, D, false, true);     // dV, dK
  static constexpr uint32_t kIdescDq = idesc_bf16_f32(128, D, true, true);      // dQ
};

enum : unsigned int {
  kSiteBProdKV = 0x51, kSiteBProdQ = 0x52,
  kSiteBMmaKV = 0x61, kSiteBMmaQ = 0x62, kSiteBMmaP = 0x63, kSiteBMmaDs = 0x64, kSiteBMmaDq = 0x65,
  kSiteBSmS = 0x71, kSiteBSmDp = 0x72, kSiteBSmDs = 0x73, kSiteBSmDv = 0x74,
  kSiteBDq = 0x81, kSiteBDone = 0x82,
};

struct KvUnit {
  int bb, kh, j, c;   // batch, kv head, kv shard, kv tile
  int kmin, kmax;     // token positions of the tile's first and last existing key
};

// Units: groups of (batch, kv head, kv shard); inside a group the key tiles
// run first to last (under a causal mask the first tiles meet the most query
// tiles), so long units start first and neighbours share query tiles in L2.
__device__ __forceinline__ KvUnit decode_kv_unit(const BwdParams &p, long long u) {
  KvUnit x;
  x.c = static_cast<int>(u % p.n_ktiles);
  long long g = u / p.n_ktiles;
  x.j = static_cast<int>(g % p.N);
  g /= p.N;
  x.kh = static_cast<int>(g % p.n_kv);
  x.bb = static_cast<int>(g / p.n_kv);
  const int r0 = x.c * kTile;
  const int r1 = min(r0 + kTile, p.L) - 1;
  x.kmin = token_at(p.layout, p.L, p.N, x.j, r0);
  x.kmax = token_at(p.layout, p.L, p.N, x.j, r1);
  return x;
}

// First local row of query shard i whose token position is >= pos.
__device__ __forceinline__ int first_row_at_or_after(const BwdParams &p, int i, int pos) {
  if (p.layout == RA_LAYOUT_STRIPED) return -floordiv(i - pos, p.N);  // ceil((pos - i) / N)
  return pos - i * p.L;
}

struct QIter {
  int s = -1, i = 0, a = 0, a_full = 0, hh = 0;
};

// Next (query shard i, query tile a, query head hq) that meets this key
// tile, in ring order.  `partial` marks steps that need the causal element
// mask.
__device__ __forceinline__ bool q_next(const BwdParams &p, const KvUnit &x, QIter &it, int &i,
                                       int &a, int &hq, bool &partial, bool &split) {
  bool have = false;
  if (it.s >= 0) {
    if (++it.hh < p.g) {
      have = true;
    } else {
      it.hh = 0;
      if (++it.a < p.n_qtiles) have = true;
    }
  }
  while (!have) {
    if (++it.s >= p.N) return false;
    it.i = (x.j + it.s) % p.N;
    it.hh = 0;
    if (!p.causal) {
      it.a = 0;
      it.a_full = 0;
    } else {
      // visible query tiles: those whose last row sees the tile's first key
      const int r_vis = max(0, first_row_at_or_after(p, it.i, x.kmin));
      it.a = r_vis >= p.L ? p.n_qtiles : r_vis / kTile;
      // unmasked query tiles: every row sees the tile's last key
      const int r_full = max(0, first_row_at_or_after(p, it.i, x.kmax));
      it.a_full = min(p.n_qtiles, (r_full + kTile - 1) / kTile);
    }
    have = it.a < p.n_qtiles;
  }
  i = it.i;
  a = it.a;
  hq = x.kh * p.g + it.hh;
  partial = it.a < it.a_full;
  split = p.causal ? (token_at(p.layout, p.L, p.N, it.i, it.a * kTile) + 1 < kSplitKeys)
                   : (p.S < kSplitKeys);
  return true;
}

__device__ __forceinline__ void shard_coords_b(int layout, int p, int r, int &c2, int &c3) {
  if (layout == RA_LAYOUT_STRIPED) {
    c2 = p;
    c3 = r;
  } else {
    c2 = r;
    c3 = p;
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

// P^T row (fp32) to TMEM as bf16 pairs in columns [0,64); with kSplit the
// rounding residual too, in columns [64,128).
template <bool kSplit>
__device__ __forceinline__ void store_p_pair(const float (&pf)[kTile], uint32_t tS) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t hi[16];
    uint32_t lo[kSplit ? 16 : 1];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int c = q4 * 32 + 2 * e;
      hi[e] = pack_bf16x2(pf[c], pf[c + 1]);
      if constexpr (kSplit)
        lo[e] = pack_bf16x2(pf[c] - __uint_as_float(hi[e] << 16),
                            pf[c + 1] - __uint_as_float(hi[e] & 0xffff0000u));
    }
    tmem_st16(tS + q4 * 16, hi);
    if constexpr (kSplit) tmem_st16(tS + 64 + q4 * 16, lo);
  }
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    bwd_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap domap) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
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
    mbar_init(&bars[C::bSFull], 1);
    mbar_init(&bars[C::bDpFull], 1);
    mbar_init(&bars[C::bPReady], 4);
    mbar_init(&bars[C::bDsReady], 4);
    mbar_init(&bars[C::bDsEmpty], 1);
    mbar_init(&bars[C::bDqFull], 1);
    mbar_init(&bars[C::bDqEmpty], 4);
    mbar_init(&bars[C::bDvDone], 1);
    mbar_init(&bars[C::bDone], 1);
    mbar_init(&bars[C::bDrain], 1);
    *abort_flag = 0;
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
  const KvUnit x = decode_kv_unit(p, blockIdx.x);

  if (warp >= 8) {
    regs_set<C::kOtherRegs, C::kLaunchRegs>();
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    int q_par[C::kQSt] = {-1, -1};
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      prefetch_tmap(&domap);
      int c2, c3;
      shard_coords_b(p.layout, x.j, x.c * kTile, c2, c3);
      mbar_arrive_expect_tx(&bars[C::bKV], 2 * C::kTileBytes);
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf) {
        tma_load_5d(smem + C::kKOff + hf * C::kHalfBytes, &kmap, &bars[C::bKV], hf * 64, x.kh, c2,
                    c3, x.bb);
        tma_load_5d(smem + C::kVOff + hf * C::kHalfBytes, &vmap, &bars[C::bKV], hf * 64, x.kh, c2,
                    c3, x.bb);
      }
    }
    QIter it;
    int i, a, hq, n = 0;
    bool partial, split;
    while (q_next(p, x, it, i, a, hq, partial, split)) {
      if (lane == 0) {
        const int st = n % C::kQSt;
        const uint32_t ph = (n / C::kQSt) & 1;
        if (mbar_wait(&bars[C::bQEmpty + st], ph ^ 1, abort_flag, kSiteBProdQ)) {
          int c2, c3;
          shard_coords_b(p.layout, i, a * kTile, c2, c3);
          mbar_arrive_expect_tx(&bars[C::bQFull + st], 2 * C::kTileBytes);
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf) {
            tma_load_5d(smem + C::kQOff + st * C::kTileBytes + hf * C::kHalfBytes, &qmap,
                        &bars[C::bQFull + st], hf * 64, hq, c2, c3, x.bb);
            tma_load_5d(smem + C::kDoOff + st * C::kTileBytes + hf * C::kHalfBytes, &domap,
                        &bars[C::bQFull + st], hf * 64, hq, c2, c3, x.bb);
          }
          q_par[st] = static_cast<int>(ph);
        }
      }
      __syncwarp();
      if (*abort_flag) break;
      ++n;
    }
    if (lane == 0 && *abort_flag) {
      mbar_wait_budget(&bars[C::bKV], 0, kWaitBudgetCycles);
      for (int s = 0; s < C::kQSt; ++s)
        if (q_par[s] >= 0) mbar_wait_budget(&bars[C::bQFull + s], q_par[s], kWaitBudgetCycles);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&bars[C::bKV], 0, abort_flag, kSiteBMmaKV);
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
    if (ok) {
      tc_fence_after();
      const uint32_t k_s = sbase + C::kKOff;
      const uint32_t v_s = sbase + C::kVOff;
      const uint32_t ds_s = sbase + C::kDsOff;
      QIter it;
      int i, a, hq, n = 0;
      bool partial, split;
      bool has = q_next(p, x, it, i, a, hq, partial, split);
      if (has && lane == 0) {
        if (mbar_wait(&bars[C::bQFull + 0], 0, abort_flag, kSiteBMmaQ)) {
          tc_fence_after();
          mma_kk<D>(tmem + C::kColS, k_s, sbase + C::kQOff, C::kIdescKK);
          mma_commit(&bars[C::bSFull]);
        }
      }
      __syncwarp();
      while (has && !*abort_flag) {
        const bool cur_split = split;
        const bool has_next = q_next(p, x, it, i, a, hq, partial, split);
        if (lane == 0) {
          const int st = n % C::kQSt;
          const uint32_t q_s = sbase + C::kQOff + st * C::kTileBytes;
          const uint32_t do_s = sbase + C::kDoOff + st * C::kTileBytes;
          const uint32_t dslo_s = C::kDsLoInDo ? do_s : sbase + C::kDsLoOff;
          bool go = true;
          if (n > 0) go = mbar_wait(&bars[C::bDqEmpty], (n - 1) & 1, abort_flag, kSiteBMmaDq);
          if (go) {
            tc_fence_after();
            // dP^T = V dO^T
            mma_kk<D>(tmem + C::kColDp, v_s, do_s, C::kIdescKK);
            mma_commit(&bars[C::bDpFull]);
            go = mbar_wait(&bars[C::bPReady], n & 1, abort_flag, kSiteBMmaP);
          }
          if (go) {
            tc_fence_after();
            // dV += P_hi^T dO + P_lo^T dO: A from TMEM (bf16 pairs), B = dO MN-major
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + C::kColDv, tmem + C::kColS + kk * 8,
                     smem_desc_sw128(do_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv,
                     (n > 0 || kk > 0) ? 1u : 0u);
            if (cur_split)
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ts(tmem + C::kColDv, tmem + C::kColS + 64 + kk * 8,
                       smem_desc_sw128(do_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv,
                       1u);
            mma_commit(&bars[C::bDvDone]);
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
            // dK += dS^T Q: A = dS^T (keys x queries, K-major), B = Q MN-major
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tmem + C::kColDk,
                     smem_desc_sw128(ds_s + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024),
                     smem_desc_sw128(q_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv,
                     (n > 0 || kk > 0) ? 1u : 0u);
            if (cur_split)  // dK += dS_lo^T Q
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ss(tmem + C::kColDk,
                       smem_desc_sw128(dslo_s + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16,
                                       1024),
                       smem_desc_sw128(q_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDv, 1u);
            // dQ = dS K: A = dS (queries x keys) read from dS^T MN-major, B = K MN-major
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tmem + C::kColDp, smem_desc_sw128(ds_s + kk * 16 * 128, kTile * 128, 1024),
                     smem_desc_sw128(k_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDq,
                     kk > 0 ? 1u : 0u);
            if (cur_split)  // dQ += dS_lo K
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_ss(tmem + C::kColDp,
                       smem_desc_sw128(dslo_s + kk * 16 * 128, kTile * 128, 1024),
                       smem_desc_sw128(k_s + kk * 16 * 128, kTile * 128, 1024), C::kIdescDq, 1u);
            mma_commit(&bars[C::bDqFull]);
            mma_commit(&bars[C::bDsEmpty]);
            mma_commit(&bars[C::bQEmpty + st]);
          }
        }
        __syncwarp();
        ++n;
        has = has_next;
      }
      if (lane == 0) mma_commit(&bars[C::bDone]);
    }
    if (lane == 0) {
      mma_commit(&bars[C::bDrain]);
      mbar_wait_budget(&bars[C::bDrain], 0, kWaitBudgetCycles);
    }
    __syncwarp();
  }
  } else if (warp < 4) {
    regs_set<C::kSoftmaxRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------ softmax (thread = key)
    const int row = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS;
    const uint32_t tDp = tmem + lane_off + C::kColDp;
    const int kr = x.c * kTile + row;
    const bool key_exists = kr < p.L;
    const int kp = token_at(p.layout, p.L, p.N, x.j, key_exists ? kr : p.L - 1);
    const float sl2 = p.scale_log2;
    uint8_t *ds_row = smem + C::kDsOff + row * 128;
    QIter it;
    int i, a, hq, n = 0;
    bool partial, split;
    while (q_next(p, x, it, i, a, hq, partial, split)) {
      const size_t qrow0 = ((static_cast<size_t>(x.bb) * p.h + hq) * p.N + i) * p.Lpad + a * kTile;
      const float4 *lse4 = reinterpret_cast<const float4 *>(p.lse2 + qrow0);
      const float4 *d4 = reinterpret_cast<const float4 *>(p.dvec + qrow0);
      // query columns c < c0 are masked for this key
      int c0 = 0;
      if (partial) c0 = first_row_at_or_after(p, i, kp) - a * kTile;
      if (!key_exists) c0 = kTile;
      if (!__all_sync(kFull, mbar_wait(&bars[C::bSFull], n & 1, abort_flag, kSiteBSmS))) break;
      tc_fence_after();
      float pf[kTile];  // P^T row of this key, fp32
      {
        uint32_t sr[kTile];
        tmem_ld128(tS, sr);
#pragma unroll
        for (int e4 = 0; e4 < kTile / 4; ++e4) {
          const float4 l4 = __ldg(lse4 + e4);
          const int c = e4 * 4;
          pf[c + 0] = ex2(fmaf(__uint_as_float(sr[c + 0]), sl2, -l4.x));
          pf[c + 1] = ex2(fmaf(__uint_as_float(sr[c + 1]), sl2, -l4.y));
          pf[c + 2] = ex2(fmaf(__uint_as_float(sr[c + 2]), sl2, -l4.z));
          pf[c + 3] = ex2(fmaf(__uint_as_float(sr[c + 3]), sl2, -l4.w));
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + u < c0) pf[c + u] = 0.f;
        }
      }
      // P_hi^T to columns [0,64) (and P_lo^T to [64,128) on split steps)
      if (split)
        store_p_pair<true>(pf, tS);
      else
        store_p_pair<false>(pf, tS);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::bPReady]);

      bool go = mbar_wait(&bars[C::bDpFull], n & 1, abort_flag, kSiteBSmDp);
      if (go) go = mbar_wait(&bars[C::bDsEmpty], (n & 1) ^ 1, abort_flag, kSiteBSmDs);
      // the residual goes over this step's dO tile once dV has read it
      if (go && split && C::kDsLoInDo)
        go = mbar_wait(&bars[C::bDvDone], n & 1, abort_flag, kSiteBSmDv);
      if (!__all_sync(kFull, go)) break;
      tc_fence_after();
      uint8_t *dslo_row = (C::kDsLoInDo ? smem + C::kDoOff + (n % C::kQSt) * C::kTileBytes
                                        : smem + C::kDsLoOff) +
                          row * 128;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        tmem_ld32(tDp + ch * 32, r);
        uint32_t whi[16], wlo[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 dd = __ldg(d4 + ch * 8 + e4);
          const int c = ch * 32 + e4 * 4;
          const float s0 = pf[c + 0] * (__uint_as_float(r[e4 * 4 + 0]) - dd.x);
          const float s1 = pf[c + 1] * (__uint_as_float(r[e4 * 4 + 1]) - dd.y);
          const float s2 = pf[c + 2] * (__uint_as_float(r[e4 * 4 + 2]) - dd.z);
          const float s3 = pf[c + 3] * (__uint_as_float(r[e4 * 4 + 3]) - dd.w);
          const uint32_t h01 = pack_bf16x2(s0, s1);
          const uint32_t h23 = pack_bf16x2(s2, s3);
          whi[e4 * 2 + 0] = h01;
          whi[e4 * 2 + 1] = h23;
          wlo[e4 * 2 + 0] = pack_bf16x2(s0 - __uint_as_float(h01 << 16),
                                        s1 - __uint_as_float(h01 & 0xffff0000u));
          wlo[e4 * 2 + 1] = pack_bf16x2(s2 - __uint_as_float(h23 << 16),
                                        s3 - __uint_as_float(h23 & 0xffff0000u));
        }
        // dS_hi^T: 32 queries = four 16-byte chunks of this key's row, 128-byte swizzled
        uint8_t *half = ds_row + (ch >> 1) * (kTile * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((ch & 1) * 4 + u) ^ (row & 7);
          *reinterpret_cast<uint4 *>(half + chunk * 16) =
              make_uint4(whi[u * 4 + 0], whi[u * 4 + 1], whi[u * 4 + 2], whi[u * 4 + 3]);
        }
        if (split) {
          uint8_t *half_lo = dslo_row + (ch >> 1) * (kTile * 128);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int chunk = ((ch & 1) * 4 + u) ^ (row & 7);
            *reinterpret_cast<uint4 *>(half_lo + chunk * 16) =
                make_uint4(wlo[u * 4 + 0], wlo[u * 4 + 1], wlo[u * 4 + 2], wlo[u * 4 + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::bDsReady]);
      ++n;
    }
  } else if (warp < 8) {
    regs_set<C::kDrainRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------ dQ drain, then dK/dV
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDq = tmem + lane_off + C::kColDp;
    QIter it;
    int i, a, hq, n = 0;
    bool partial, split;
    bool aborted = false;
    while (q_next(p, x, it, i, a, hq, partial, split)) {
      if (!__all_sync(kFull, mbar_wait(&bars[C::bDqFull], n & 1, abort_flag, kSiteBDq))) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const int qr = a * kTile + row;
      const bool exists = qr < p.L;
      float *dst = p.dq + ((static_cast<size_t>(x.bb) * p.S +
                            token_at(p.layout, p.L, p.N, i, exists ? qr : 0)) *
                               p.h +
                           hq) *
                              D;
      uint32_t r[D / 32][32];
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tDq + ch * 32, r[ch]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::bDqEmpty]);
      if (exists) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float *ptr = dst + ch * 32 + u * 4;
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(ptr),
                         "f"(__uint_as_float(r[ch][u * 4 + 0]) * p.scale),
                         "f"(__uint_as_float(r[ch][u * 4 + 1]) * p.scale),
                         "f"(__uint_as_float(r[ch][u * 4 + 2]) * p.scale),
                         "f"(__uint_as_float(r[ch][u * 4 + 3]) * p.scale)
                         : "memory");
          }
      }
      ++n;
    }
    // dK, dV of this key tile
    bool have = n > 0 && !aborted;
    if (have) have = mbar_wait(&bars[C::bDone], 0, abort_flag, kSiteBDone);
    have = __all_sync(kFull, have && *abort_flag == 0);
    if (have) tc_fence_after();
    const int kr = x.c * kTile + row;
    const bool write = kr < p.L && !*abort_flag && (n == 0 || have);
    const size_t off =
        ((static_cast<size_t>(x.bb) * p.S +
          token_at(p.layout, p.L, p.N, x.j, kr < p.L ? kr : 0)) *
             p.n_kv +
         x.kh) *
        D;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? C::kColDk : C::kColDv;
      float *dst = (which == 0 ? p.dk : p.dv) + off;
      const float mul = which == 0 ? p.scale : 1.f;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        if (have) tmem_ld32(tmem + lane_off + col + ch * 32, r);
        if (write) {
          float4 *d4 = reinterpret_cast<float4 *>(dst + ch * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            d4[u] = have ? make_float4(__uint_as_float(r[u * 4 + 0]) * mul,
                                       __uint_as_float(r[u * 4 + 1]) * mul,
                                       __uint_as_float(r[u * 4 + 2]) * mul,
                                       __uint_as_float(r[u * 4 + 3]) * mul)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
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

// D = rowsum(dO * O) and LSE2 = LSE * log2(e) per (batch, head, query row),
// written in shard-local order [b, h, N, Lpad]; padding rows get D = 0 and
// LSE2 = +inf (their P is exactly 0).  One warp per row.
template <int D>
__global__ void bwd_pre_kernel(BwdParams p, const float *out, const float *lse,
                               const uint16_t *dout) {
  const long long rows = static_cast<long long>(p.b) * p.h * p.N * p.Lpad;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < rows;
       w += warps) {
    const int r = static_cast<int>(w % p.Lpad);
    long long t = w / p.Lpad;
    const int i = static_cast<int>(t % p.N);
    t /= p.N;
    const int hq = static_cast<int>(t % p.h);
    const long long bb = t / p.h;
    float dsum = 0.f, l2 = INFINITY;
    if (r < p.L) {
      const int tok = token_at(p.layout, p.L, p.N, i, r);
      const size_t row = ((bb * p.S + tok) * p.h + hq) * D;
      const float4 *o4 = reinterpret_cast<const float4 *>(out + row);
      const uint2 *g4 = reinterpret_cast<const uint2 *>(dout + row);
      for (int e = lane; e < D / 4; e += 32) {
        const float4 o = o4[e];
        const uint2 gg = g4[e];
        dsum += o.x * __uint_as_float(gg.x << 16) + o.y * __uint_as_float(gg.x & 0xffff0000u) +
                o.z * __uint_as_float(gg.y << 16) + o.w * __uint_as_float(gg.y & 0xffff0000u);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(kFull, dsum, o);
      const float lv = lse[(bb * p.h + hq) * p.S + tok];
      l2 = (lv == -INFINITY) ? INFINITY : lv * kLog2e;
    }
    if (lane == 0) {
      p.dvec[w] = dsum;
      p.lse2[w] = l2;
    }
  }
}

template <int D>
cudaError_t launch_bwd_t(const BwdParams &p, const float *out, const float *lse,
                         const uint16_t *dout, const CUtensorMap &qmap, const CUtensorMap &kmap,
                         const CUtensorMap &vmap, const CUtensorMap &domap, long long n_units,
                         int n_sm, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const long long pre_rows = static_cast<long long>(p.b) * p.h * p.N * p.Lpad;
  long long pre_blocks = (pre_rows * 32 + 255) / 256;
  if (pre_blocks > static_cast<long long>(n_sm) * 8) pre_blocks = static_cast<long long>(n_sm) * 8;
  if (pre_blocks < 1) pre_blocks = 1;
  bwd_pre_kernel<D><<<static_cast<unsigned int>(pre_blocks), 256, 0, stream>>>(p, out, lse, dout);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = bwd_kernel<D>;
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
      p, qmap, kmap, vmap, domap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdParams &p, int d, const float *out, const float *lse,
                       const uint16_t *dout, const CUtensorMap &qmap, const CUtensorMap &kmap,
                       const CUtensorMap &vmap, const CUtensorMap &domap, long long n_units,
                       int n_sm, cudaStream_t stream) {
  if (n_units <= 0) return cudaSuccess;
  if (d == 128)
    return launch_bwd_t<128>(p, out, lse, dout, qmap, kmap, vmap, domap, n_units, n_sm, stream);
  if (d == 64)
    return launch_bwd_t<64>(p, out, lse, dout, qmap, kmap, vmap, domap, n_units, n_sm, stream);
  return cudaErrorInvalidValue;
}

RA_DEFINE_ERROR_WORD_READER(read_error_word_bwd)

}  // namespace ra
