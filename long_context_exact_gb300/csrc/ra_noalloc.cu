// ra_noalloc.cu -- the backward without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run
// the backward: code running inside a CUDA-graph capture (cudaMalloc is not
// capturable), plug-ins and runtimes that only receive pre-allocated tensors
// from a host framework that owns the allocator, and real-time loops that
// forbid allocator traffic.  For them this file keeps the backward's scratch
// (per query row: D = rowsum(dO * O) and the log2-domain LSE) in a fixed
// array in the library's own device memory, and passes its address to the
// ordinary backward launch.  The caller still passes every input and output.
//
// The array is a file-scope static __device__ array, so every GPU that loads
// the library holds it until the process exits.  Its host-side name is only
// a stand-in for the symbol: host code must ask the runtime for the device
// address (cudaGetSymbolAddress) with the device current, once per device.
#include <mutex>
#include <string>

#include "ra_internal.cuh"

namespace ra {
namespace {

constexpr size_t kNoAllocScratchBytes = RA_BWD_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device, looked up on the
// first call for that device.
cudaError_t scratch_for_current_device(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace ra

extern "C" {

// See include/ra.h.  Validation and the launch are those of
// ra_ring_attention_bwd; only the scratch comes from the static array.
ra_status ra_ring_attention_bwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                        const float *out, const float *lse, const uint16_t *dout,
                                        float *dq, float *dk, float *dv, int64_t S, int n_shards,
                                        ra_layout layout, int causal, float scale, ra_dims dims,
                                        void *stream) {
  // First pass: the ordinary entry point without a workspace.  It checks the
  // shape (dims, layout, S against n_shards and the zig-zag tile rule) and
  // every pointer (null, 16-byte alignment), launches nothing, and answers
  // RA_ERR_WORKSPACE when those are good (RA_OK for an empty problem).  The
  // scale and the tensor-map encodings are checked by the second call below,
  // before it launches anything.  The first pass's expected workspace
  // complaint is not left behind as this thread's last error.
  const std::string before = ra::last_error_text();
  const ra_status st = ra_ring_attention_bwd(q, k, v, out, lse, dout, dq, dk, dv, nullptr, 0, S,
                                             n_shards, layout, causal, scale, dims, stream);
  if (st != RA_ERR_WORKSPACE) return st;
  ra::restore_last_error(before.c_str());
  const size_t need = ra_bwd_workspace_size(S, n_shards, dims);
  if (need > ra::kNoAllocScratchBytes)
    return ra::report_error(RA_ERR_WORKSPACE,
                            "the allocation-free backward holds %zu bytes of scratch; this "
                            "problem needs %zu (b * h * n_shards * rows per shard rounded up "
                            "to 128, times 8 bytes)",
                            ra::kNoAllocScratchBytes, need);
  void *scratch = nullptr;
  cudaError_t e = ra::scratch_for_current_device(&scratch);
  if (e != cudaSuccess)
    return ra::report_error(RA_ERR_CUDA, "scratch address lookup: %s", cudaGetErrorString(e));
  // The scratch needs no clearing: the pre-pass writes every word the main
  // kernel reads before it runs (and dq is cleared on the stream as usual).
  return ra_ring_attention_bwd(q, k, v, out, lse, dout, dq, dk, dv, scratch,
                               ra::kNoAllocScratchBytes, S, n_shards, layout, causal, scale, dims,
                               stream);
}

}  // extern "C"
