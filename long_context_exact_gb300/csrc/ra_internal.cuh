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
// the dropped 2^-9 of each weight alone approaches the 1e-2 parity budget.
// Longer rows spread the weights and keep plain bf16.
constexpr int kSplitKeys = 4096;

// ------------------------------------------------------------ placement
// Token held at local row r of shard p.  Contiguous: shard p holds
// [p*L, (p+1)*L).  Striped: token t lives on shard t mod N at row t div N
// (the first page's "Striped Attention"; the third page's section 6 example).
__host__ __device__ __forceinline__ int token_at(int layout, int L, int N, int p, int r) {
  return layout == RA_LAYOUT_STRIPED ? r * N + p : p * L + r;
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
// the inclusive causal rule (key position <= query position); may be < 0.
__host__ __device__ __forceinline__ int last_visible_row(int layout, int L, int N, int j, int qp) {
  return layout == RA_LAYOUT_STRIPED ? floordiv(qp - j, N) : qp - j * L;
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
  const int32_t *q_pos;     // block mode: [Lq]
  const int32_t *k_pos;     // block mode: [Lk]
  float *out;               // ring: [b, S, h, d]
  float *lse;               // ring: [b, h, S]
  float *st_m;              // block: [b, h, Lq]
  float *st_l;              // block: [b, h, Lq]
  float *st_o;              // block: [b, Lq, h, d]
};

struct BwdParams {
  int b, h, n_kv, g;
  int N, L, S;              // shards, rows per shard, tokens per sequence
  int layout, causal;
  float scale;              // dQ, dK multiplier
  float scale_log2;         // scale * log2(e)
  int n_qtiles, n_ktiles;   // ceil(L / 128)
  int Lpad;                 // n_qtiles * 128
  float *dvec;              // [b, h, N, Lpad] rowsum(dO * O), shard-local order
  float *lse2;              // [b, h, N, Lpad] LSE * log2(e), +inf on padding rows
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
                       const CUtensorMap &dqmap, long long n_units, int n_sm,
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
// Record a message for ra_last_error() on this thread and return `st`.
ra_status report_error(ra_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

// Read-and-clear of each translation unit's device error word.
cudaError_t read_error_word_fwd(unsigned int *word);
cudaError_t read_error_word_small(unsigned int *word);
cudaError_t read_error_word_bwd(unsigned int *word);

}  // namespace ra
