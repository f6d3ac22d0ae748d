// ra_small.cu -- the HBM-bound and bookkeeping kernels: finalize, the
// two-sided rescale-merge, the token-placement and ring-order maps, and the
// bounded-wait self test.  Also home of the device error word.
#include <cmath>

#include <climits>

#include "ra_internal.cuh"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr int kEwThreads = 256;

// Grid size for a grid-stride loop over `work` items: enough CTAs to fill
// every SM several times, never more than the work needs.
inline unsigned int ew_grid(long long work) {
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n_sm <= 0)
      n_sm = 152;
  }
  const long long want = (work + kEwThreads - 1) / kEwThreads;
  const long long cap = static_cast<long long>(n_sm) * 8;
  return static_cast<unsigned int>(want < 1 ? 1 : (want < cap ? want : cap));
}

// Grid for the row kernels below: blockIdx.y walks the (batch, head) pairs,
// blockIdx.x the rows of one pair, so no thread divides a row index; about
// eight CTAs per SM in all.
inline dim3 rows_grid(long long pairs, long long rows_per_pair, int rows_per_warp) {
  const long long ctas = static_cast<long long>(ew_grid(1LL << 40));
  const long long gy = pairs < 65535 ? pairs : 65535;
  const long long per_cta = static_cast<long long>(kEwThreads / 32) * rows_per_warp;
  long long gx = (rows_per_pair + per_cta - 1) / per_cta;
  const long long cap = (ctas + gy - 1) / gy;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  return dim3(static_cast<unsigned int>(gx), static_cast<unsigned int>(gy < 1 ? 1 : gy));
}

// Rows handled per warp and loop trip by the two HBM-bound kernels below:
// their loads are all issued before any result is formed, so each warp keeps
// kRowsPerTrip rows of every operand in flight (one float4 per lane and row).
constexpr int kRowsPerTrip = 4;

// One warp per (batch, head, row), lane e holding columns 4e..4e+3 (d = 64
// uses half the warp).  o <- o / l, lse = m + ln l; rows with l == 0 get 0
// and -inf.
__global__ void finalize_kernel(float *o, const float *l, const float *m, float *lse, int b,
                                long long Lq, int h, int d) {
  const int lane = threadIdx.x & 31;
  const bool col = lane < d / 4;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const size_t ostride = static_cast<size_t>(h) * d;  // floats between rows of one head
  for (long long bh = blockIdx.y; bh < static_cast<long long>(b) * h; bh += gridDim.y) {
    const long long bb = bh / h;
    float *orow = o + (static_cast<size_t>(bb) * Lq * h + (bh - bb * h)) * d;
    const float *lrow = l + bh * Lq, *mrow = m + bh * Lq;
    float *lserow = lse + bh * Lq;
    for (long long base = w0; base < Lq; base += kRowsPerTrip * warps) {
      float4 v[kRowsPerTrip];
      float lr[kRowsPerTrip], mr[kRowsPerTrip];
#pragma unroll
      for (int k = 0; k < kRowsPerTrip; ++k) {
        const long long r = base + k * warps;
        if (r < Lq) {
          lr[k] = lrow[r];
          mr[k] = mrow[r];
          if (col) v[k] = reinterpret_cast<const float4 *>(orow + r * ostride)[lane];
        }
      }
#pragma unroll
      for (int k = 0; k < kRowsPerTrip; ++k) {
        const long long r = base + k * warps;
        if (r < Lq) {
          const bool live = lr[k] > 0.f;
          const float inv = live ? 1.f / lr[k] : 0.f;
          if (lane == 0) lserow[r] = live ? mr[k] + logf(lr[k]) : -INFINITY;
          if (col) {
            float4 x = v[k];
            x.x *= inv;
            x.y *= inv;
            x.z *= inv;
            x.w *= inv;
            reinterpret_cast<float4 *>(orow + r * ostride)[lane] = x;
          }
        }
      }
    }
  }
}

// Rescale-merge of two normalised partial results over disjoint keys.
// o (and lse) may alias side a: each element is read before it is written.
__global__ void merge_kernel(const float *o_a, const float *lse_a, const float *o_b,
                             const float *lse_b, float *o, float *lse, int b, long long Lq, int h,
                             int d) {
  const int lane = threadIdx.x & 31;
  const bool col = lane < d / 4;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const size_t ostride = static_cast<size_t>(h) * d;  // floats between rows of one head
  for (long long bh = blockIdx.y; bh < static_cast<long long>(b) * h; bh += gridDim.y) {
    const long long bb = bh / h;
    const size_t obase = (static_cast<size_t>(bb) * Lq * h + (bh - bb * h)) * d;
    for (long long base = w0; base < Lq; base += kRowsPerTrip * warps) {
      float4 va[kRowsPerTrip], vb[kRowsPerTrip];
      float la[kRowsPerTrip], lb[kRowsPerTrip];
#pragma unroll
      for (int k = 0; k < kRowsPerTrip; ++k) {
        const long long r = base + k * warps;
        if (r < Lq) {
          la[k] = lse_a[bh * Lq + r];
          lb[k] = lse_b[bh * Lq + r];
          if (col) {
            const size_t off = obase + r * ostride;
            va[k] = reinterpret_cast<const float4 *>(o_a + off)[lane];
            vb[k] = reinterpret_cast<const float4 *>(o_b + off)[lane];
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kRowsPerTrip; ++k) {
        const long long r = base + k * warps;
        if (r < Lq) {
          const float mx = fmaxf(la[k], lb[k]);
          float wa = 0.f, wb = 0.f, out_lse = -INFINITY;
          if (mx != -INFINITY) {
            wa = (la[k] == -INFINITY) ? 0.f : expf(la[k] - mx);
            wb = (lb[k] == -INFINITY) ? 0.f : expf(lb[k] - mx);
            const float den = wa + wb;
            out_lse = mx + logf(den);
            wa /= den;
            wb /= den;
          }
          if (col) {
            const float4 a = va[k], c = vb[k];
            float4 x;
            x.x = (wa == 0.f ? 0.f : wa * a.x) + (wb == 0.f ? 0.f : wb * c.x);
            x.y = (wa == 0.f ? 0.f : wa * a.y) + (wb == 0.f ? 0.f : wb * c.y);
            x.z = (wa == 0.f ? 0.f : wa * a.z) + (wb == 0.f ? 0.f : wb * c.z);
            x.w = (wa == 0.f ? 0.f : wa * a.w) + (wb == 0.f ? 0.f : wb * c.w);
            reinterpret_cast<float4 *>(o + obase + r * ostride)[lane] = x;
          }
          __syncwarp();
          if (lane == 0) lse[bh * Lq + r] = out_lse;
        }
      }
    }
  }
}

// Empty online-softmax states for `splits` key splits: m = -inf, l = 0,
// O = 0 (m_rows = splits * b * h * Lq entries, o_vals = m_rows * d; l may be
// null).
__global__ void state_init_kernel(float *m, float *l, float *o, long long m_rows,
                                  long long o_vals) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < o_vals / 4;
       t += stride) {
    reinterpret_cast<float4 *>(o)[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < m_rows) {
      m[t] = -INFINITY;
      if (l) l[t] = 0.f;
    }
  }
}

// Combination of the unnormalised states of `splits` disjoint key ranges
// (the second page's rescale-merge, over any number of parts):
//   M = max_s m_s,  L = sum_s l_s e^(m_s - M),
//   out = sum_s e^(m_s - M) O_s / L,  lse = M + ln L;
// rows no key reaches (L = 0) get 0 and -inf.  One warp per (batch, head,
// row); lane e holds columns 4e..4e+3.  State slices are split_rows =
// b * h * Lq rows apart (m, l) and split_rows * d floats apart (O).
__global__ void combine_kernel(const float *m, const float *l, const float *o, int splits,
                               float *out, float *lse, int b, long long Lq, int h, int d) {
  const long long rows = static_cast<long long>(b) * h * Lq;
  const int lane = threadIdx.x & 31;
  const bool col = lane < d / 4;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long r0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const size_t ostride = static_cast<size_t>(h) * d;  // floats between rows of one head
  for (long long bh = blockIdx.y; bh < static_cast<long long>(b) * h; bh += gridDim.y) {
    const long long bb = bh / h;
    const size_t obase = (static_cast<size_t>(bb) * Lq * h + (bh - bb * h)) * d;
    for (long long r = r0; r < Lq; r += warps) {
      const long long w = bh * Lq + r;
      float mx = -INFINITY;
      for (int z = lane; z < splits; z += 32) mx = fmaxf(mx, m[z * rows + w]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float den = 0.f;
      for (int z = lane; z < splits; z += 32) {
        const float mz = m[z * rows + w];
        if (mz != -INFINITY) den += l[z * rows + w] * expf(mz - mx);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      const bool live = mx != -INFINITY && den > 0.f;
      const size_t orow = obase + r * ostride;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (live && col) {
        for (int z = 0; z < splits; ++z) {
          const float mz = m[z * rows + w];
          if (mz == -INFINITY) continue;
          const float wz = expf(mz - mx) / den;
          const float4 v = reinterpret_cast<const float4 *>(o + z * rows * d + orow)[lane];
          acc.x += wz * v.x;
          acc.y += wz * v.y;
          acc.z += wz * v.z;
          acc.w += wz * v.w;
        }
      }
      if (col) reinterpret_cast<float4 *>(out + orow)[lane] = acc;
      if (lane == 0) lse[w] = live ? mx + logf(den) : -INFINITY;
    }
  }
}

__global__ void position_map_kernel(int layout, int S, int N, int32_t *shard_of,
                                    int32_t *local_of, int32_t *token_of) {
  const int L = S / N;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < S;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    // idx enumerates (shard p, local row r); the token is where it lands.
    const int p = static_cast<int>(idx / L);
    const int r = static_cast<int>(idx % L);
    const int t = token_at(layout, L, N, p, r);
    if (shard_of) shard_of[t] = p;
    if (local_of) local_of[t] = r;
    if (token_of) token_of[idx] = t;
  }
}

__global__ void ring_order_kernel(int N, int32_t *order) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < N * N) order[idx] = kv_shard_at(idx / N, idx % N, N);
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait
// runs out and the timeout is recorded in the error word.
__global__ void wait_timeout_selftest_kernel(long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_budget(&bar, 0, budget)) raise_error(kErrTimeout, 0xF0);
  }
}

// Throughput probe for the exp2 unit: each thread runs eight independent
// chains x <- 2^(-x) (values stay in [1/2, 1]), so the SFU pipes, not
// latency, bound it.  The chains' sum is written so nothing is elided.
__global__ void ex2_probe_kernel(long long iters, float *sink) {
  float x0 = 0.1f, x1 = 0.2f, x2 = 0.3f, x3 = 0.4f, x4 = 0.5f, x5 = 0.6f, x6 = 0.7f, x7 = 0.8f;
  for (long long i = 0; i < iters; ++i) {
    x0 = ex2(-x0);
    x1 = ex2(-x1);
    x2 = ex2(-x2);
    x3 = ex2(-x3);
    x4 = ex2(-x4);
    x5 = ex2(-x5);
    x6 = ex2(-x6);
    x7 = ex2(-x7);
  }
  sink[static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x] =
      x0 + x1 + x2 + x3 + x4 + x5 + x6 + x7;
}

}  // namespace

cudaError_t launch_finalize(float *o, const float *l, const float *m, float *lse, int b,
                            long long Lq, int h, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(b) * h * Lq;
  if (rows == 0) return cudaSuccess;
  finalize_kernel<<<rows_grid(static_cast<long long>(b) * h, Lq, kRowsPerTrip), kEwThreads, 0,
                    stream>>>(o, l, m, lse, b, Lq, h, d);
  return cudaGetLastError();
}

cudaError_t launch_merge(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, float *o, float *lse, int b, long long Lq, int h,
                         int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(b) * h * Lq;
  if (rows == 0) return cudaSuccess;
  merge_kernel<<<rows_grid(static_cast<long long>(b) * h, Lq, kRowsPerTrip), kEwThreads, 0,
                 stream>>>(o_a, lse_a, o_b, lse_b, o, lse, b, Lq, h, d);
  return cudaGetLastError();
}

cudaError_t launch_state_init(float *m, float *l, float *o, long long m_rows, int d,
                              cudaStream_t stream) {
  const long long o_vals = m_rows * d;
  if (o_vals == 0) return cudaSuccess;
  state_init_kernel<<<ew_grid(o_vals / 4), kEwThreads, 0, stream>>>(m, l, o, m_rows, o_vals);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *m, const float *l, const float *o, int splits, float *out,
                           float *lse, int b, long long Lq, int h, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(b) * h * Lq;
  if (rows == 0) return cudaSuccess;
  combine_kernel<<<rows_grid(static_cast<long long>(b) * h, Lq, 1), kEwThreads, 0, stream>>>(
      m, l, o, splits, out, lse, b, Lq, h, d);
  return cudaGetLastError();
}

// Causal chunked prefill, first pass: the largest key position of every
// 128-key tile (a warp per tile).
__global__ void tile_kmax_kernel(const int32_t *k_pos, int Lk, int n_ktiles, int32_t *kmax) {
  const int lane = threadIdx.x & 31;
  const int c = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (c >= n_ktiles) return;  // whole warps: 32 lanes share c
  int mx = INT_MIN;
  for (int e = lane; e < 128; e += 32) {
    const int kr = c * 128 + e;
    if (kr < Lk) mx = max(mx, k_pos[kr]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) kmax[c] = mx;
}

// Second pass: for query tile a, the number of leading key tiles whose
// largest key position is at most the tile's smallest query position --
// the key tiles every row of the tile sees in full.  A block per query tile.
__global__ void prefill_visible_kernel(const int32_t *q_pos, int Lq, const int32_t *kmax,
                                       int n_ktiles, int32_t *kt_end) {
  __shared__ int qmin_s;
  __shared__ int first_s;
  const int a = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) first_s = n_ktiles;
  if (warp == 0) {
    int mn = INT_MAX;
    for (int r = a * 128 + lane; r < min(Lq, a * 128 + 128); r += 32) mn = min(mn, q_pos[r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    if (lane == 0) qmin_s = mn;
  }
  __syncthreads();
  const int qmin = qmin_s;
  int first = n_ktiles;
  for (int c = threadIdx.x; c < n_ktiles; c += blockDim.x)
    if (kmax[c] > qmin) {
      first = c;
      break;
    }
  if (first < n_ktiles) atomicMin(&first_s, first);
  __syncthreads();
  if (threadIdx.x == 0) kt_end[a] = first_s;
}

cudaError_t launch_prefill_visible(const int32_t *q_pos, const int32_t *k_pos, long long Lq,
                                   long long Lk, int32_t *kmax, int32_t *kt_end,
                                   cudaStream_t stream) {
  const long long n_qtiles = (Lq + 127) / 128;
  const int n_ktiles = static_cast<int>((Lk + 127) / 128);
  if (n_qtiles <= 0 || n_ktiles <= 0) return cudaSuccess;
  tile_kmax_kernel<<<(n_ktiles + 7) / 8, 256, 0, stream>>>(k_pos, static_cast<int>(Lk), n_ktiles,
                                                           kmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prefill_visible_kernel<<<static_cast<unsigned int>(n_qtiles), 512, 0, stream>>>(
      q_pos, static_cast<int>(Lq), kmax, n_ktiles, kt_end);
  return cudaGetLastError();
}

cudaError_t launch_position_map(int layout, int S, int N, int32_t *shard_of, int32_t *local_of,
                                int32_t *token_of, cudaStream_t stream) {
  if (S == 0) return cudaSuccess;
  position_map_kernel<<<ew_grid(S), kEwThreads, 0, stream>>>(layout, S, N, shard_of, local_of,
                                                             token_of);
  return cudaGetLastError();
}

cudaError_t launch_ring_order(int N, int32_t *order, cudaStream_t stream) {
  const int n = N * N;
  ring_order_kernel<<<(n + kEwThreads - 1) / kEwThreads, kEwThreads, 0, stream>>>(N, order);
  return cudaGetLastError();
}

cudaError_t launch_ex2_probe(long long iters, float *sink, int blocks, int threads,
                             cudaStream_t stream) {
  ex2_probe_kernel<<<blocks, threads, 0, stream>>>(iters, sink);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(long long budget, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(budget);
  return cudaGetLastError();
}

RA_DEFINE_ERROR_WORD_READER(read_error_word_small)

}  // namespace ra
