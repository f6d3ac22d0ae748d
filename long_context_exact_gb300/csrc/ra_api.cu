// ra_api.cu -- the extern "C" boundary declared in include/ra.h: argument
// validation, TMA tensor-map construction, kernel launches and error
// reporting.  No device memory is allocated here.
#include <cmath>
#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "ra_internal.cuh"

namespace ra {
namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

// Count one kernel launch that the runtime accepted.
cudaError_t counted(cudaError_t e, uint64_t n = 1) {
  if (e == cudaSuccess) g_launches.fetch_add(n, std::memory_order_relaxed);
  return e;
}

ra_status fail(ra_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
ra_status fail(ra_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

ra_status cuda_fail(cudaError_t e, const char *what) {
  return fail(RA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  }
  return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pointers must be non-null and 16-byte aligned (TMA and float4 access).
#define RA_CHECK_PTR(p)                                                                   \
  do {                                                                                    \
    if ((p) == nullptr) return fail(RA_ERR_INVALID_ARG, "%s is NULL", #p);                \
    if (!aligned16(p)) return fail(RA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p);  \
  } while (0)

bool known_layout(int layout) {
  return layout == RA_LAYOUT_CONTIGUOUS || layout == RA_LAYOUT_STRIPED ||
         layout == RA_LAYOUT_ZIGZAG;
}

// Packed documents: offsets [b][n_docs + 1] on the device (contents are the
// caller's contract and are not read on the host).
ra_status check_docs(const int32_t *cu, int n_docs) {
  if (cu == nullptr) return n_docs == 0 ? RA_OK : fail(RA_ERR_INVALID_ARG, "n_docs without cu_seqlens");
  if (n_docs < 1 || n_docs > (1 << 30))
    return fail(RA_ERR_INVALID_ARG, "n_docs must be in 1 .. 2^30 (got %d)", n_docs);
  return RA_OK;
}

// Zig-zag shards are two half-blocks of S / 2N tokens each; the attention
// kernels need every 128-row tile inside one half-block.
ra_status check_zigzag_tiles(int layout, int64_t S, int n_shards) {
  if (layout != RA_LAYOUT_ZIGZAG) return RA_OK;
  if (S % (2LL * n_shards) != 0 || (S / (2LL * n_shards)) % kTile != 0)
    return fail(RA_ERR_UNSUPPORTED,
                "zig-zag needs half-blocks (S / 2N = %lld / %d) of whole %d-token tiles",
                (long long)S, 2 * n_shards, kTile);
  return RA_OK;
}

ra_status check_dims(const ra_dims &dm) {
  if (dm.b < 0 || dm.h <= 0 || dm.n_kv <= 0 || dm.d <= 0)
    return fail(RA_ERR_INVALID_ARG, "dims must be positive (b >= 0): b=%d h=%d n_kv=%d d=%d",
                dm.b, dm.h, dm.n_kv, dm.d);
  if (dm.h % dm.n_kv != 0)
    return fail(RA_ERR_UNSUPPORTED, "h=%d is not a multiple of n_kv=%d", dm.h, dm.n_kv);
  if (dm.d != 64 && dm.d != 128) return fail(RA_ERR_UNSUPPORTED, "d=%d (supported: 64, 128)", dm.d);
  return RA_OK;
}

ra_status resolve_scale(float scale, int d, float *out) {
  if (std::isnan(scale) || std::isinf(scale)) return fail(RA_ERR_INVALID_ARG, "scale is not finite");
  *out = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  return RA_OK;
}

// ------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// View a bf16 tensor [b, N*L, heads, d] whose rows are spread over N shards
// of L rows each as a 5-D tensor with coordinates
//   striped   : (x, head, shard, row, batch)   token = row * N + shard
//   contiguous: (x, head, row, shard, batch)   token = shard * L + row
// and a box of 64 columns x 128 rows of one head, 128-byte swizzled.
ra_status make_map(CUtensorMap *map, const void *base, int layout, int b, int N, int L, int heads,
                   int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t tok = static_cast<cuuint64_t>(heads) * d * 2;  // bytes per token
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  dims[0] = static_cast<cuuint64_t>(d);
  dims[1] = static_cast<cuuint64_t>(heads);
  strides[0] = static_cast<cuuint64_t>(d) * 2;
  if (layout == RA_LAYOUT_STRIPED) {
    dims[2] = static_cast<cuuint64_t>(N);
    dims[3] = static_cast<cuuint64_t>(L);
    strides[1] = tok;
    strides[2] = tok * N;
    box[2] = 1;
    box[3] = kTile;
  } else {
    dims[2] = static_cast<cuuint64_t>(L);
    dims[3] = static_cast<cuuint64_t>(N);
    strides[1] = tok;
    strides[2] = tok * L;
    box[2] = kTile;
    box[3] = 1;
  }
  dims[4] = static_cast<cuuint64_t>(b < 1 ? 1 : b);
  strides[3] = tok * N * L;
  box[0] = 64;
  box[1] = 1;
  box[4] = 1;
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return RA_OK;
}

// fp32 dq [b, N*L, h, d] for the backward's bulk reductions: same 5-D view
// as make_map, 32-column (128-byte) boxes of 32 rows, 128-byte swizzled.
ra_status make_dq_map(CUtensorMap *map, const float *base, int layout, int b, int N, int L,
                      int heads, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t tok = static_cast<cuuint64_t>(heads) * d * 4;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), 0, 0,
                        static_cast<cuuint64_t>(b < 1 ? 1 : b)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(d) * 4, tok, 0, tok * N * L};
  cuuint32_t box[5] = {32, 1, 1, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (layout == RA_LAYOUT_STRIPED) {
    dims[2] = static_cast<cuuint64_t>(N);
    dims[3] = static_cast<cuuint64_t>(L);
    strides[2] = tok * N;
    box[3] = 32;
  } else {
    dims[2] = static_cast<cuuint64_t>(L);
    dims[3] = static_cast<cuuint64_t>(N);
    strides[2] = tok * L;
    box[2] = 32;
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled (dq) failed (%d)", (int)r);
  return RA_OK;
}

ra_status launch_attention(const FwdParams &p, int d, const void *q, const void *k,
                           const void *v, long long q_rows_per_shard, long long k_rows_per_shard,
                           cudaStream_t stream) {
  CUtensorMap qm, km, vm;
  ra_status st;
  if ((st = make_map(&qm, q, p.layout, p.b, p.N, static_cast<int>(q_rows_per_shard), p.h, d)) != RA_OK)
    return st;
  if ((st = make_map(&km, k, p.layout, p.b, p.N, static_cast<int>(k_rows_per_shard), p.n_kv, d)) != RA_OK)
    return st;
  if ((st = make_map(&vm, v, p.layout, p.b, p.N, static_cast<int>(k_rows_per_shard), p.n_kv, d)) != RA_OK)
    return st;
  const int nq = (p.g % 2 == 0) ? 2 : 1;
  FwdParams pp = p;
  pp.pairs = p.g / nq;
  const long long n_units =
      static_cast<long long>(p.b) * p.n_kv * pp.pairs * p.N * static_cast<long long>(p.n_qtiles);
  if (n_units > 0x7fffffffLL) return fail(RA_ERR_UNSUPPORTED, "too many work units (%lld)", n_units);
  cudaError_t e = counted(launch_fwd(pp, d, nq, qm, km, vm, n_units, stream));
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return RA_OK;
}

// A causal block step over at least this many key tiles (16,384 keys) runs
// in two launches (the fully seen leading tiles of each query tile unmasked,
// the rest masked).  Below it the second launch's fixed cost -- every CTA
// starts and scans the positions once more -- and the tails of two short
// launches outweigh the faster tiles: 8K x 8K diagonal steps lost 6-11 %,
// 16K ones gained 2 %, 32K ones 13 % (off the diagonal 25 %).
constexpr int kTwoLaunchKeyTiles = 128;

// Key splits for a chunked prefill: n_splits if given (capped by the key
// tiles and kMaxSplits), else enough splits for about eight waves of CTAs
// (so the last, partly filled wave costs little) with at least four key
// tiles each, and at most kBlockKeyTiles tiles each.
constexpr int kMaxSplits = 64;

int resolve_splits(int64_t Lq, int64_t Lk, int n_splits, const ra_dims &dims) {
  const int n_ktiles = static_cast<int>((Lk + kTile - 1) / kTile);
  int s = n_splits;
  if (s <= 0) {
    const int g = dims.h / dims.n_kv;
    const long long units = static_cast<long long>(dims.b) * dims.n_kv * (g % 2 == 0 ? g / 2 : g) *
                            ((Lq + kTile - 1) / kTile);
    const long long want = (8LL * sm_count() + units - 1) / units;
    s = static_cast<int>(want < 1 ? 1 : (want > kMaxSplits ? kMaxSplits : want));
    s = std::min(s, std::max(1, (n_ktiles + 3) / 4));
    s = std::max(s, (n_ktiles + kBlockKeyTiles - 1) / kBlockKeyTiles);
  }
  s = std::min(std::min(s, kMaxSplits), std::max(1, n_ktiles));
  // splits of equal whole tiles: the last may be shorter, none empty
  const int per = (n_ktiles + s - 1) / s;
  return (n_ktiles + per - 1) / per;
}

}  // namespace

ra_status report_error(ra_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

const char *last_error_text() { return g_last_error.c_str(); }

void restore_last_error(const char *text) { g_last_error = text; }

}  // namespace ra

using namespace ra;

extern "C" {

int ra_version(void) { return 100; }

uint64_t ra_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *ra_last_error(void) { return g_last_error.c_str(); }

ra_status ra_block_step(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *m,
                        float *l, float *o, const int32_t *q_pos, const int32_t *k_pos,
                        int64_t Lq, int64_t Lk, ra_dims dims, int causal, float scale,
                        void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (Lq < 0 || Lk < 0) return fail(RA_ERR_INVALID_ARG, "negative length Lq=%lld Lk=%lld",
                                    (long long)Lq, (long long)Lk);
  if (Lq >= (1LL << 31) || Lk >= (1LL << 31))
    return fail(RA_ERR_UNSUPPORTED, "Lq/Lk must be below 2^31");
  if (Lq == 0 || Lk == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(q);
  RA_CHECK_PTR(k);
  RA_CHECK_PTR(v);
  RA_CHECK_PTR(m);
  RA_CHECK_PTR(l);
  RA_CHECK_PTR(o);
  if (causal) {
    if (!q_pos || !k_pos) return fail(RA_ERR_INVALID_ARG, "causal block step needs q_pos and k_pos");
    if ((Lk + kTile - 1) / kTile > kBlockKeyTiles)
      return fail(RA_ERR_UNSUPPORTED, "a causal block step takes at most %lld keys (Lk=%lld)",
                  static_cast<long long>(kBlockKeyTiles) * kTile, (long long)Lk);
  }
  float sc = 0.f;
  if ((st = resolve_scale(scale, dims.d, &sc)) != RA_OK) return st;
  FwdParams p{};
  p.b = dims.b;
  p.h = dims.h;
  p.n_kv = dims.n_kv;
  p.g = dims.h / dims.n_kv;
  p.N = 1;
  p.L = static_cast<int>(Lq);
  p.Lk = static_cast<int>(Lk);
  p.S = static_cast<int>(Lq);
  p.layout = RA_LAYOUT_CONTIGUOUS;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = sc * kLog2e;
  p.n_qtiles = static_cast<int>((Lq + kTile - 1) / kTile);
  p.n_ktiles = static_cast<int>((Lk + kTile - 1) / kTile);
  p.block_mode = 1;
  p.q_pos = q_pos;
  p.k_pos = k_pos;
  p.st_m = m;
  p.st_l = l;
  p.st_o = o;
  if (causal && p.n_ktiles >= kTwoLaunchKeyTiles) {
    // Two launches that fold into the same state: the leading key tiles each
    // query tile sees in full (on a ring step, all tiles off the diagonal)
    // through the kernel without the causal rule, ~25 % faster per tile;
    // then the rest through the causal one.  Each CTA finds its own split.
    FwdParams pv = p;
    pv.causal = 0;
    pv.full_prefix = 1;
    if ((st = launch_attention(pv, dims.d, q, k, v, Lq, Lk, static_cast<cudaStream_t>(stream))) !=
        RA_OK)
      return st;
    p.full_prefix = 2;
  }
  return launch_attention(p, dims.d, q, k, v, Lq, Lk, static_cast<cudaStream_t>(stream));
}

ra_status ra_finalize(float *o, const float *l, const float *m, float *lse, int64_t Lq,
                      ra_dims dims, void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (Lq < 0) return fail(RA_ERR_INVALID_ARG, "negative Lq");
  if (Lq == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(o);
  RA_CHECK_PTR(l);
  RA_CHECK_PTR(m);
  RA_CHECK_PTR(lse);
  cudaError_t e = counted(launch_finalize(o, l, m, lse, dims.b, Lq, dims.h, dims.d,
                                  static_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "finalize launch");
}

ra_status ra_merge(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                   float *o, float *lse, int64_t Lq, ra_dims dims, void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (Lq < 0) return fail(RA_ERR_INVALID_ARG, "negative Lq");
  if (Lq == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(o_a);
  RA_CHECK_PTR(lse_a);
  RA_CHECK_PTR(o_b);
  RA_CHECK_PTR(lse_b);
  RA_CHECK_PTR(o);
  RA_CHECK_PTR(lse);
  cudaError_t e = counted(launch_merge(o_a, lse_a, o_b, lse_b, o, lse, dims.b, Lq, dims.h, dims.d,
                                       static_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "merge launch");
}

// ints of the per-query-tile array in the prefill workspace (16-byte padded)
static inline int64_t p_qtiles_rounded(int64_t Lq) { return ((Lq + kTile - 1) / kTile + 3) / 4 * 4; }

size_t ra_prefill_workspace_size(int64_t Lq, int64_t Lk, int n_splits, ra_dims dims) {
  if (Lq <= 0 || Lk <= 0 || dims.b <= 0 || dims.h <= 0 || dims.n_kv <= 0 ||
      dims.h % dims.n_kv != 0 || dims.d <= 0 || Lq >= (1LL << 31) || Lk >= (1LL << 31))
    return 0;
  const int s = resolve_splits(Lq, Lk, n_splits, dims);
  const size_t rows = static_cast<size_t>(dims.b) * dims.h * static_cast<size_t>(Lq);
  // states of the s key splits, then one int per query tile (a causal
  // prefill's split point between its two passes) and one per key tile (the
  // tile's largest key position)
  const size_t n_qtiles = static_cast<size_t>((Lq + kTile - 1) / kTile);
  const size_t n_ktiles = static_cast<size_t>((Lk + kTile - 1) / kTile);
  return static_cast<size_t>(s) * rows * (2 + static_cast<size_t>(dims.d)) * sizeof(float) +
         (n_qtiles * sizeof(int32_t) + 15) / 16 * 16 + (n_ktiles * sizeof(int32_t) + 15) / 16 * 16;
}

ra_status ra_chunked_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *out,
                             float *lse, const int32_t *q_pos, const int32_t *k_pos, int64_t Lq,
                             int64_t Lk, int n_splits, ra_dims dims, int causal, float scale,
                             void *workspace, size_t workspace_bytes, void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (Lq < 0 || Lk < 0) return fail(RA_ERR_INVALID_ARG, "negative length Lq=%lld Lk=%lld",
                                    (long long)Lq, (long long)Lk);
  if (Lq >= (1LL << 31) || Lk >= (1LL << 31))
    return fail(RA_ERR_UNSUPPORTED, "Lq/Lk must be below 2^31");
  if (n_splits < 0 || n_splits > kMaxSplits)
    return fail(RA_ERR_INVALID_ARG, "n_splits must be 0 (automatic) .. %d", kMaxSplits);
  if (Lq == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(q);
  RA_CHECK_PTR(out);
  RA_CHECK_PTR(lse);
  if (Lk > 0) {
    RA_CHECK_PTR(k);
    RA_CHECK_PTR(v);
  }
  if (causal && (!q_pos || (Lk > 0 && !k_pos)))
    return fail(RA_ERR_INVALID_ARG, "causal prefill needs q_pos and k_pos");
  if (causal && Lk > 0) {
    const int splits = resolve_splits(Lq, Lk, n_splits, dims);
    const long long n_ktiles = (Lk + kTile - 1) / kTile;
    if ((n_ktiles + splits - 1) / splits > kBlockKeyTiles)
      return fail(RA_ERR_UNSUPPORTED,
                  "a causal key split covers at most %lld keys: %lld keys need more than %d "
                  "splits",
                  static_cast<long long>(kBlockKeyTiles) * kTile, (long long)Lk, splits);
  }
  float sc = 0.f;
  if ((st = resolve_scale(scale, dims.d, &sc)) != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const long long rows = static_cast<long long>(dims.b) * dims.h * Lq;
  if (Lk == 0) {  // nothing to attend to: O = 0, LSE = -inf
    cudaError_t e = counted(launch_state_init(lse, nullptr, out, rows, dims.d, cs));
    return e == cudaSuccess ? RA_OK : cuda_fail(e, "empty prefill");
  }
  const size_t need = ra_prefill_workspace_size(Lq, Lk, n_splits, dims);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(RA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(RA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  const int splits = resolve_splits(Lq, Lk, n_splits, dims);
  float *m = static_cast<float *>(workspace);
  float *l = m + static_cast<size_t>(splits) * rows;
  float *o = l + static_cast<size_t>(splits) * rows;
  int32_t *kt_end = reinterpret_cast<int32_t *>(o + static_cast<size_t>(splits) * rows * dims.d);
  int32_t *kmax = kt_end + (p_qtiles_rounded(Lq));
  FwdParams p{};
  p.b = dims.b;
  p.h = dims.h;
  p.n_kv = dims.n_kv;
  p.g = dims.h / dims.n_kv;
  p.N = 1;
  p.L = static_cast<int>(Lq);
  p.Lk = static_cast<int>(Lk);
  p.S = static_cast<int>(Lq);
  p.layout = RA_LAYOUT_CONTIGUOUS;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = sc * kLog2e;
  p.n_qtiles = static_cast<int>((Lq + kTile - 1) / kTile);
  p.n_ktiles = static_cast<int>((Lk + kTile - 1) / kTile);
  p.split_tiles = (p.n_ktiles + splits - 1) / splits;
  p.block_mode = 1;
  p.q_pos = q_pos;
  p.k_pos = k_pos;
  p.st_m = m;
  p.st_l = l;
  p.st_o = o;
  cudaError_t e = counted(launch_state_init(m, l, o, static_cast<long long>(splits) * rows,
                                            dims.d, cs));
  if (e != cudaSuccess) return cuda_fail(e, "state init");
  if (causal) {
    // The key tiles every row of a query tile sees in full (for the usual
    // prefill, all but the last few) go through the block kernel without the
    // causal rule, which runs them ~25 % faster; then the rest through the
    // causal one, whose block steps merge into the same split states.
    e = counted(launch_prefill_visible(q_pos, k_pos, Lq, Lk, kmax, kt_end, cs), 2);
    if (e != cudaSuccess) return cuda_fail(e, "prefill pre-pass");
    FwdParams pv = p;
    pv.causal = 0;
    pv.q_pos = nullptr;
    pv.k_pos = nullptr;
    pv.kt_end = kt_end;
    if ((st = launch_attention(pv, dims.d, q, k, v, Lq, Lk, cs)) != RA_OK) return st;
    p.kt_begin = kt_end;
  }
  if ((st = launch_attention(p, dims.d, q, k, v, Lq, Lk, cs)) != RA_OK) return st;
  e = counted(launch_combine(m, l, o, splits, out, lse, dims.b, Lq, dims.h, dims.d, cs));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "combine launch");
}

ra_status ra_ring_attention_packed(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   float *out, float *lse, int64_t S, int n_shards,
                                   ra_layout layout, int causal, float scale, ra_dims dims,
                                   const int32_t *cu_seqlens, int n_docs, void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (!known_layout(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
  if (S < 0) return fail(RA_ERR_INVALID_ARG, "negative S");
  if (n_shards < 1) return fail(RA_ERR_INVALID_ARG, "n_shards must be >= 1");
  if (S >= (1LL << 31)) return fail(RA_ERR_UNSUPPORTED, "S must be below 2^31");
  if (S % n_shards != 0)
    return fail(RA_ERR_UNSUPPORTED, "S=%lld is not a multiple of n_shards=%d", (long long)S, n_shards);
  if ((st = check_zigzag_tiles(layout, S, n_shards)) != RA_OK) return st;
  if (S == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(q);
  RA_CHECK_PTR(k);
  RA_CHECK_PTR(v);
  RA_CHECK_PTR(out);
  RA_CHECK_PTR(lse);
  if ((st = check_docs(cu_seqlens, n_docs)) != RA_OK) return st;
  float sc = 0.f;
  if ((st = resolve_scale(scale, dims.d, &sc)) != RA_OK) return st;
  const long long L = S / n_shards;
  FwdParams p{};
  p.b = dims.b;
  p.h = dims.h;
  p.n_kv = dims.n_kv;
  p.g = dims.h / dims.n_kv;
  p.N = n_shards;
  p.L = static_cast<int>(L);
  p.Lk = static_cast<int>(L);
  p.S = static_cast<int>(S);
  p.layout = layout;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = sc * kLog2e;
  p.n_qtiles = static_cast<int>((L + kTile - 1) / kTile);
  p.n_ktiles = p.n_qtiles;
  p.block_mode = 0;
  p.out = out;
  p.lse = lse;
  p.cu = cu_seqlens;
  p.n_docs = n_docs;
  return launch_attention(p, dims.d, q, k, v, L, L, static_cast<cudaStream_t>(stream));
}

ra_status ra_ring_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *out,
                            float *lse, int64_t S, int n_shards, ra_layout layout, int causal,
                            float scale, ra_dims dims, void *stream) {
  return ra_ring_attention_packed(q, k, v, out, lse, S, n_shards, layout, causal, scale, dims,
                                  nullptr, 0, stream);
}

size_t ra_bwd_workspace_size(int64_t S, int n_shards, ra_dims dims) {
  if (S <= 0 || n_shards < 1 || S % n_shards != 0 || dims.b <= 0 || dims.h <= 0) return 0;
  const int64_t L = S / n_shards;
  const int64_t Lpad = (L + kTile - 1) / kTile * kTile;
  return static_cast<size_t>(2) * dims.b * dims.h * static_cast<size_t>(n_shards) *
         static_cast<size_t>(Lpad) * sizeof(float);
}

ra_status ra_ring_attention_packed_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                       const float *out, const float *lse, const uint16_t *dout,
                                       float *dq, float *dk, float *dv, void *workspace,
                                       size_t workspace_bytes, int64_t S, int n_shards,
                                       ra_layout layout, int causal, float scale, ra_dims dims,
                                       const int32_t *cu_seqlens, int n_docs, void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (!known_layout(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
  if (S < 0) return fail(RA_ERR_INVALID_ARG, "negative S");
  if (n_shards < 1) return fail(RA_ERR_INVALID_ARG, "n_shards must be >= 1");
  if (S >= (1LL << 31)) return fail(RA_ERR_UNSUPPORTED, "S must be below 2^31");
  if (S % n_shards != 0)
    return fail(RA_ERR_UNSUPPORTED, "S=%lld is not a multiple of n_shards=%d", (long long)S, n_shards);
  if ((st = check_zigzag_tiles(layout, S, n_shards)) != RA_OK) return st;
  if (S == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(q);
  RA_CHECK_PTR(k);
  RA_CHECK_PTR(v);
  RA_CHECK_PTR(out);
  RA_CHECK_PTR(lse);
  RA_CHECK_PTR(dout);
  RA_CHECK_PTR(dq);
  RA_CHECK_PTR(dk);
  RA_CHECK_PTR(dv);
  if ((st = check_docs(cu_seqlens, n_docs)) != RA_OK) return st;
  const size_t need = ra_bwd_workspace_size(S, n_shards, dims);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(RA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(RA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  float sc = 0.f;
  if ((st = resolve_scale(scale, dims.d, &sc)) != RA_OK) return st;
  const int64_t L = S / n_shards;
  BwdParams p{};
  p.cu = cu_seqlens;
  p.n_docs = n_docs;
  p.b = dims.b;
  p.h = dims.h;
  p.n_kv = dims.n_kv;
  p.g = dims.h / dims.n_kv;
  p.N = n_shards;
  p.L = static_cast<int>(L);
  p.S = static_cast<int>(S);
  p.layout = layout;
  p.causal = causal ? 1 : 0;
  p.scale = sc;
  p.scale_log2 = sc * kLog2e;
  p.n_qtiles = static_cast<int>((L + kTile - 1) / kTile);
  p.n_ktiles = p.n_qtiles;
  p.Lpad = p.n_qtiles * kTile;
  const size_t rows = static_cast<size_t>(dims.b) * dims.h * n_shards * p.Lpad;
  p.dvec = static_cast<float *>(workspace);
  p.lse2 = p.dvec + rows;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  CUtensorMap qm, km, vm, dom, dqm, dkm, dvm;
  if ((st = make_map(&qm, q, layout, dims.b, n_shards, p.L, dims.h, dims.d)) != RA_OK) return st;
  if ((st = make_map(&km, k, layout, dims.b, n_shards, p.L, dims.n_kv, dims.d)) != RA_OK) return st;
  if ((st = make_map(&vm, v, layout, dims.b, n_shards, p.L, dims.n_kv, dims.d)) != RA_OK) return st;
  if ((st = make_map(&dom, dout, layout, dims.b, n_shards, p.L, dims.h, dims.d)) != RA_OK) return st;
  if ((st = make_dq_map(&dqm, dq, layout, dims.b, n_shards, p.L, dims.h, dims.d)) != RA_OK) return st;
  if ((st = make_dq_map(&dkm, dk, layout, dims.b, n_shards, p.L, dims.n_kv, dims.d)) != RA_OK) return st;
  if ((st = make_dq_map(&dvm, dv, layout, dims.b, n_shards, p.L, dims.n_kv, dims.d)) != RA_OK) return st;
  // one unit per (key tile, group of query shards, query head), the group
  // covering ~32K query rows (one shard when shards are that long); packed
  // documents: one per (key tile, query shard), the KV head's query heads
  // inside
  p.qgroup = cu_seqlens != nullptr ? 1 : std::max(1, std::min(n_shards, 32768 / p.Lpad));
  p.n_groups = (n_shards + p.qgroup - 1) / p.qgroup;
  const long long n_units =
      cu_seqlens != nullptr
          ? static_cast<long long>(dims.b) * dims.n_kv * n_shards * n_shards * p.n_ktiles
          : static_cast<long long>(dims.b) * dims.h * n_shards * p.n_groups * p.n_ktiles;
  if (n_units > 0x7fffffffLL) return fail(RA_ERR_UNSUPPORTED, "too many work units (%lld)", n_units);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(dq, 0, static_cast<size_t>(dims.b) * S * dims.h * dims.d * 4, cs);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(dk, 0, static_cast<size_t>(dims.b) * S * dims.n_kv * dims.d * 4, cs);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(dv, 0, static_cast<size_t>(dims.b) * S * dims.n_kv * dims.d * 4, cs);
  if (e != cudaSuccess) return cuda_fail(e, "gradient clear");
  e = counted(launch_bwd(p, dims.d, out, lse, dout, qm, km, vm, dom, dqm, dkm, dvm, n_units,
                         sm_count(), cs), 2);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "backward launch");
}

size_t ra_block_bwd_workspace_size(int64_t Lq, ra_dims dims) {
  return ra_bwd_workspace_size(Lq, 1, dims);
}

ra_status ra_block_step_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *out, const float *lse, const uint16_t *dout, float *dq,
                            float *dk, float *dv, const int32_t *q_pos, const int32_t *k_pos,
                            int64_t Lq, int64_t Lk, ra_dims dims, int causal, float scale,
                            void *workspace, size_t workspace_bytes, void *stream) {
  ra_status st;
  if ((st = check_dims(dims)) != RA_OK) return st;
  if (Lq < 0 || Lk < 0) return fail(RA_ERR_INVALID_ARG, "negative length Lq=%lld Lk=%lld",
                                    (long long)Lq, (long long)Lk);
  if (Lq >= (1LL << 31) || Lk >= (1LL << 31))
    return fail(RA_ERR_UNSUPPORTED, "Lq/Lk must be below 2^31");
  if (Lq == 0 || Lk == 0 || dims.b == 0) return RA_OK;
  RA_CHECK_PTR(q);
  RA_CHECK_PTR(k);
  RA_CHECK_PTR(v);
  RA_CHECK_PTR(out);
  RA_CHECK_PTR(lse);
  RA_CHECK_PTR(dout);
  RA_CHECK_PTR(dq);
  RA_CHECK_PTR(dk);
  RA_CHECK_PTR(dv);
  if (causal && (!q_pos || !k_pos))
    return fail(RA_ERR_INVALID_ARG, "causal block backward needs q_pos and k_pos");
  const size_t need = ra_block_bwd_workspace_size(Lq, dims);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(RA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(RA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  float sc = 0.f;
  if ((st = resolve_scale(scale, dims.d, &sc)) != RA_OK) return st;
  BwdParams p{};
  p.cu = nullptr;
  p.n_docs = 0;
  p.b = dims.b;
  p.h = dims.h;
  p.n_kv = dims.n_kv;
  p.g = dims.h / dims.n_kv;
  p.N = 1;
  p.L = static_cast<int>(Lq);
  p.S = static_cast<int>(Lq);
  p.layout = RA_LAYOUT_CONTIGUOUS;
  p.causal = causal ? 1 : 0;
  p.scale = sc;
  p.scale_log2 = sc * kLog2e;
  p.n_qtiles = static_cast<int>((Lq + kTile - 1) / kTile);
  p.n_ktiles = static_cast<int>((Lk + kTile - 1) / kTile);
  p.Lpad = p.n_qtiles * kTile;
  p.block = 1;
  p.Lk = static_cast<int>(Lk);
  p.qgroup = 1;
  p.n_groups = 1;
  p.q_pos = causal ? q_pos : nullptr;
  p.k_pos = causal ? k_pos : nullptr;
  const size_t rows = static_cast<size_t>(dims.b) * dims.h * p.Lpad;
  p.dvec = static_cast<float *>(workspace);
  p.lse2 = p.dvec + rows;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  CUtensorMap qm, km, vm, dom, dqm, dkm, dvm;
  const int Lqi = p.L, Lki = p.Lk;
  if ((st = make_map(&qm, q, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lqi, dims.h, dims.d)) != RA_OK) return st;
  if ((st = make_map(&km, k, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lki, dims.n_kv, dims.d)) != RA_OK) return st;
  if ((st = make_map(&vm, v, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lki, dims.n_kv, dims.d)) != RA_OK) return st;
  if ((st = make_map(&dom, dout, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lqi, dims.h, dims.d)) != RA_OK) return st;
  if ((st = make_dq_map(&dqm, dq, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lqi, dims.h, dims.d)) != RA_OK) return st;
  if ((st = make_dq_map(&dkm, dk, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lki, dims.n_kv, dims.d)) != RA_OK) return st;
  if ((st = make_dq_map(&dvm, dv, RA_LAYOUT_CONTIGUOUS, dims.b, 1, Lki, dims.n_kv, dims.d)) != RA_OK) return st;
  // one unit per (key tile, query head); dq, dk and dv are added to, not cleared
  const long long n_units = static_cast<long long>(dims.b) * dims.h * p.n_ktiles;
  if (n_units > 0x7fffffffLL) return fail(RA_ERR_UNSUPPORTED, "too many work units (%lld)", n_units);
  cudaError_t e = counted(launch_bwd(p, dims.d, out, lse, dout, qm, km, vm, dom, dqm, dkm, dvm,
                                     n_units, sm_count(), static_cast<cudaStream_t>(stream)), 2);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "block backward launch");
}

ra_status ra_ring_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                const float *out, const float *lse, const uint16_t *dout,
                                float *dq, float *dk, float *dv, void *workspace,
                                size_t workspace_bytes, int64_t S, int n_shards, ra_layout layout,
                                int causal, float scale, ra_dims dims, void *stream) {
  return ra_ring_attention_packed_bwd(q, k, v, out, lse, dout, dq, dk, dv, workspace,
                                      workspace_bytes, S, n_shards, layout, causal, scale, dims,
                                      nullptr, 0, stream);
}

ra_status ra_position_map(ra_layout layout, int64_t S, int n_shards, int32_t *shard_of,
                          int32_t *local_of, int32_t *token_of, void *stream) {
  if (!known_layout(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
  if (S < 0 || n_shards < 1) return fail(RA_ERR_INVALID_ARG, "S >= 0 and n_shards >= 1 required");
  if (S >= (1LL << 31)) return fail(RA_ERR_UNSUPPORTED, "S must be below 2^31");
  if (S % n_shards != 0) return fail(RA_ERR_UNSUPPORTED, "S is not a multiple of n_shards");
  if (layout == RA_LAYOUT_ZIGZAG && S % (2LL * n_shards) != 0)
    return fail(RA_ERR_UNSUPPORTED, "zig-zag needs S to be a multiple of 2 * n_shards");
  if (S == 0) return RA_OK;
  cudaError_t e = counted(launch_position_map(layout, static_cast<int>(S), n_shards, shard_of,
                                              local_of, token_of, static_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "position map launch");
}

ra_status ra_ring_order(int n_shards, int32_t *order, void *stream) {
  if (n_shards < 1 || n_shards > 46340) return fail(RA_ERR_INVALID_ARG, "n_shards out of range");
  if (!order) return fail(RA_ERR_INVALID_ARG, "order is NULL");
  cudaError_t e = counted(launch_ring_order(n_shards, order, static_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "ring order launch");
}

ra_status ra_stream_check(void *stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int words[3] = {0u, 0u, 0u};
  if ((e = read_error_word_fwd(&words[0])) != cudaSuccess) return cuda_fail(e, "error word read");
  if ((e = read_error_word_small(&words[1])) != cudaSuccess) return cuda_fail(e, "error word read");
  if ((e = read_error_word_bwd(&words[2])) != cudaSuccess) return cuda_fail(e, "error word read");
  for (unsigned int w : words) {
    if (w == 0u) continue;
    if ((w & 0xffu) == 2u)
      return fail(RA_ERR_UNSUPPORTED,
                  "kernel refused to run: dynamic shared memory base misaligned (site 0x%x)",
                  w >> 8);
    return fail(RA_ERR_DEVICE_TIMEOUT, "device wait ran out (code %u, site 0x%x)", w & 0xffu,
                w >> 8);
  }
  return RA_OK;
}

ra_status ra_ex2_probe(int64_t iters, float *sink, int64_t sink_floats, void *stream) {
  if (iters < 1 || iters > (1LL << 24)) return fail(RA_ERR_INVALID_ARG, "iters out of range");
  RA_CHECK_PTR(sink);
  const int threads = 256;
  const long long blocks = static_cast<long long>(sm_count()) * 4;
  if (sink_floats < blocks * threads)
    return fail(RA_ERR_INVALID_ARG, "sink holds %lld floats, %lld needed", (long long)sink_floats,
                blocks * threads);
  cudaError_t e = counted(launch_ex2_probe(iters, sink, static_cast<int>(blocks), threads,
                                           static_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "ex2 probe launch");
}

int64_t ra_ex2_probe_threads(void) { return static_cast<int64_t>(sm_count()) * 4 * 256; }

ra_status ra_selftest_wait_timeout(long long budget_cycles, void *stream) {
  if (budget_cycles < 1 || budget_cycles > (1LL << 31))
    return fail(RA_ERR_INVALID_ARG, "budget_cycles out of range");
  cudaError_t e = counted(launch_wait_timeout_selftest(budget_cycles, static_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "self-test launch");
}

}  // extern "C"
