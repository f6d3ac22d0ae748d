// ra_internal.cuh -- declarations shared by the kernels and the C-ABI layer:
// token placement, ring visit order, tile classification, kernel parameter
// blocks and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ra.h"

namespace ra {

constexpr int kTile = 128;   // query rows per Q tile, keys per K/V tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Rows that see fewer keys than this put large weights on single keys, so
// their P (and dS) go to the tensor cores as a bf16 pair hi + lo instead of
// one bf16 value: a bf16 operand keeps 8 significant bits, and on such rows
// the dropped 2^-9 of each weight alone approaches the 1e-2 parity budget
// (a row with two keys: dQ off by up to 1.3e-2 in a model of the rounding,
// 2e-3 at 256 keys, 1.6e-3 at 512).  Longer rows spread the weights and keep
// plain bf16; a longer row that still puts a large weight on a few keys is
// caught by the peaked-P rules of the forward and backward kernels.
constexpr int kSplitKeys = 512;

// Causal block steps: one CTA classifies its whole key range once (keep and
// mask bits in shared memory), so a range holds at most this many key tiles
// (8,388,608 keys); the host refuses longer causal ranges.
constexpr int kBlockKeyTiles = 65536;

// ------------------------------------------------------------ placement
// Token held at local row r of shard p.  Contiguous: shard p holds
// [p*L, (p+1)*L).  Striped: token t lives on shard t mod N at row t div N
// (the first page's "Striped Attention"; the third page's section 6 example).
// Zig-zag (the first page's "Zig-Zag Ring Attention"): 2N half-blocks of
// C = L/2 tokens, shard p holding half-block p at rows [0, C) and half-block
// 2N-1-p at rows [C, L).  Under every layout a shard's tokens increase with
// the local row, so the keys of a shard that a query sees form a prefix.
__host__ __device__ __forceinline__ int token_at(int layout, int L, int N, int p, int r) {
  if (layout == RA_LAYOUT_STRIPED) return r * N + p;
  if (layout == RA_LAYOUT_ZIGZAG) {
    const int C = L >> 1;
    return r < C ? p * C + r : (2 * N - 1 - p) * C + (r - C);
  }
  return p * L + r;
}

// Key/value shard that query shard i meets at ring step s: (i - s) mod N
// (the fourth page's "The Ring Communication Protocol", k_block_idx).
__host__ __device__ __forceinline__ int kv_shard_at(int i, int s, int N) {
  int j = (i - s) % N;
  return j < 0 ? j + N : j;
}

__host__ __device__ __forceinline__ int floordiv(int a, int b) {  // b > 0
  int q = a / b;
  return (q * b > a) ? q - 1 : q;
}

// Largest local key row of shard j visible to a query at position qp, under
// the inclusive causal rule (key position <= query position); may be < 0
// (nothing visible) or >= L (the whole shard).
__host__ __device__ __forceinline__ int last_visible_row(int layout, int L, int N, int j, int qp) {
  if (layout == RA_LAYOUT_STRIPED) return floordiv(qp - j, N);
  if (layout == RA_LAYOUT_ZIGZAG) {
    const int C = L >> 1;
    const int early = j * C, late = (2 * N - 1 - j) * C;
    if (qp < early + C) return qp - early;
    return qp < late ? C - 1 : C + (qp - late);
  }
  return qp - j * L;
}

// First local row of shard i whose token is >= pos; <= 0 when every row is,
// >= L when none is.
__host__ __device__ __forceinline__ int first_row_at_or_after(int layout, int L, int N, int i,
                                                              int pos) {
  if (layout == RA_LAYOUT_STRIPED) return -floordiv(i - pos, N);  // ceil((pos - i) / N)
  if (layout == RA_LAYOUT_ZIGZAG) {
    const int C = L >> 1;
    const int early = i * C, late = (2 * N - 1 - i) * C;
    if (pos < early + C) return pos - early;
    return pos <= late ? C : C + (pos - late);
  }
  return pos - i * L;
}

// Coordinates (c2, c3) of local row r of shard p in the 5-D tensor-map view
// of a [b, S, heads, d] tensor: striped maps are (x, head, shard, row, batch),
// the others (x, head, row, shard, batch) over contiguous blocks of L tokens.
// A zig-zag row is addressed through its token in the contiguous view (a
// tile never straddles a half-block, so its rows stay consecutive tokens).
__host__ __device__ __forceinline__ void map_coords(int layout, int L, int N, int p, int r,
                                                    int &c2, int &c3) {
  if (layout == RA_LAYOUT_STRIPED) {
    c2 = p;
    c3 = r;
  } else if (layout == RA_LAYOUT_ZIGZAG) {
    const int t = token_at(layout, L, N, p, r);
    c2 = t % L;
    c3 = t / L;
  } else {
    c2 = r;
    c3 = p;
  }
}

// ------------------------------------------------------------ packed documents
// Documents packed end to end into one sequence (the third page's section
// 5): cu [b][n_docs + 1] holds each batch row's document offsets, from 0 to
// S, non-decreasing.  A query sees only keys of its own document (and, under
// the causal rule, none after itself), so the keys a query at position t
// sees are the positions [ds, causal ? t : de - 1] of its document [ds, de).
// Without documents (cu == nullptr) the document is the whole sequence.
__device__ __forceinline__ void doc_of(const int32_t *cu, int n_docs, int bb, int S, int t,
                                       int &ds, int &de) {
  if (cu == nullptr) {
    ds = 0;
    de = S;
    return;
  }
  const int32_t *c = cu + static_cast<size_t>(bb) * (n_docs + 1);
  int lo = 0, hi = n_docs - 1;  // the last document that starts at or before t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  ds = c[lo];
  de = c[lo + 1];
}

// Keys visible to the query at position t form the position window
// [win_lo, win_hi] (inclusive).
__device__ __forceinline__ void key_window(const int32_t *cu, int n_docs, int bb, int S,
                                           int causal, int t, int &win_lo, int &win_hi) {
  int ds, de;
  doc_of(cu, n_docs, bb, S, t, ds, de);
  win_lo = ds;
  win_hi = causal ? t : de - 1;
}

// ------------------------------------------------------------ parameters
struct FwdParams {
  int b, h, n_kv, g;        // g = h / n_kv
  int N;                    // shards (1 for a block step)
  int L;                    // query rows per shard
  int Lk;                   // key rows per shard (== L on the ring)
  int S;                    // tokens per sequence (ring) or Lq (block step)
  int layout;               // ra_layout
  int causal;
  float scale_log2;         // scale * log2(e)
  int n_qtiles;             // ceil(L / 128)
  int n_ktiles;             // ceil(Lk / 128)
  int pairs;                // g / NQ query-head groups per KV head
  int block_mode;           // 0: ring + finalize, 1: block step with state merge
  int split_tiles;          // block mode: key tiles per split (0: one split of all)
  const int32_t *cu;        // ring: packed-document offsets [b][n_docs + 1], or null
  int n_docs;
  const int32_t *q_pos;     // block mode: [Lq]
  const int32_t *k_pos;     // block mode: [Lk]
  float *out;               // ring: [b, S, h, d]
  float *lse;               // ring: [b, h, S]
  float *st_m;              // block: [b, h, Lq]
  float *st_l;              // block: [b, h, Lq]
  float *st_o;              // block: [b, Lq, h, d]
  // block mode, chunked prefill: per query tile, the key tiles before
  // kt_end[a] are seen in full by every row of the tile; a pass may stop its
  // key range there (kt_end) or start it there (kt_begin)
  const int32_t *kt_end;
  const int32_t *kt_begin;
  // block mode, causal step in two launches: each CTA finds the leading key
  // tiles of its range that every row of its query tile sees in full; 1: the
  // launch (without the causal rule) covers only those, 2: the launch (with
  // it) covers the rest.  0: the whole range.
  int full_prefix;
};

struct BwdParams {
  int b, h, n_kv, g;
  const int32_t *cu;        // packed-document offsets [b][n_docs + 1], or null
  int n_docs;
  int N, L, S;              // shards, rows per shard, tokens per sequence
  // block mode: one query block of L rows (N = 1, S = L) against one key
  // block of Lk rows, token positions from q_pos / k_pos (increasing)
  int block;
  int Lk;
  // unpacked ring: each unit meets qgroup consecutive query shards (n_groups
  // groups of them), so that short shards still make long units
  int qgroup, n_groups;
  const int32_t *q_pos;     // [L]
  const int32_t *k_pos;     // [Lk]
  int layout, causal;
  float scale;              // dQ, dK multiplier
  float scale_log2;         // scale * log2(e)
  int n_qtiles, n_ktiles;   // ceil(L / 128)
  int Lpad;                 // n_qtiles * 128
  float *dvec;              // [b, h, N, Lpad] -rowsum(dO * O), shard-local order
  float *lse2;              // [b, h, N, Lpad] -LSE * log2(e), -inf on padding rows
  float *dq;                // [b, S, h, d], accumulated (zeroed before the launch)
  float *dk, *dv;           // [b, S, n_kv, d]
};

// Forward launch (ra_fwd.cu).  Tensor maps view Q/K/V as 5-D tensors whose
// coordinates are (x, head, shard-or-row, row-or-shard, batch); see
// make_qkv_maps() in ra_api.cu.
cudaError_t launch_fwd(const FwdParams &p, int d, int nq, const CUtensorMap &qmap,
                       const CUtensorMap &kmap, const CUtensorMap &vmap, long long n_units,
                       cudaStream_t stream);

// Backward launch (ra_bwd.cu): the D / LSE2 pre-pass, then the main kernel.
cudaError_t launch_bwd(const BwdParams &p, int d, const float *out, const float *lse,
                       const uint16_t *dout, const CUtensorMap &qmap, const CUtensorMap &kmap,
                       const CUtensorMap &vmap, const CUtensorMap &domap,
                       const CUtensorMap &dqmap, const CUtensorMap &dkmap,
                       const CUtensorMap &dvmap, long long n_units, int n_sm,
                       cudaStream_t stream);

// Element-wise kernels (ra_small.cu).
cudaError_t launch_finalize(float *o, const float *l, const float *m, float *lse, int b,
                            long long Lq, int h, int d, cudaStream_t stream);
cudaError_t launch_merge(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, float *o, float *lse, int b, long long Lq, int h,
                         int d, cudaStream_t stream);
cudaError_t launch_position_map(int layout, int S, int N, int32_t *shard_of, int32_t *local_of,
                                int32_t *token_of, cudaStream_t stream);
cudaError_t launch_ring_order(int N, int32_t *order, cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(long long budget, cudaStream_t stream);
cudaError_t launch_state_init(float *m, float *l, float *o, long long m_rows, int d,
                              cudaStream_t stream);
cudaError_t launch_combine(const float *m, const float *l, const float *o, int splits, float *out,
                           float *lse, int b, long long Lq, int h, int d, cudaStream_t stream);
cudaError_t launch_prefill_visible(const int32_t *q_pos, const int32_t *k_pos, long long Lq,
                                   long long Lk, int32_t *kmax, int32_t *kt_end,
                                   cudaStream_t stream);
cudaError_t launch_ex2_probe(long long iters, float *sink, int blocks, int threads,
                             cudaStream_t stream);
// Record a message for ra_last_error() on this thread and return `st`.
ra_status report_error(ra_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// The calling thread's last error message, and a way to put back a saved one
// (for a call that runs another entry point only to validate its arguments).
const char *last_error_text();
void restore_last_error(const char *text);

// Read-and-clear of each translation unit's device error word.
cudaError_t read_error_word_fwd(unsigned int *word);
cudaError_t read_error_word_small(unsigned int *word);
cudaError_t read_error_word_bwd(unsigned int *word);

}  // namespace ra
