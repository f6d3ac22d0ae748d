// ra_host.cu -- entry points that take host buffers.
//
// ra_host_alloc places pinned host memory on the NUMA node the driver names
// as nearest to the current GPU: on a Grace machine with two CPU sockets a
// buffer on the far socket crosses the socket link on every copy, which on
// one machine slowed host-to-device copies from ~210 GB/s to ~26 GB/s.
//
// ra_pipeline runs ring-attention steps (forward, optionally followed by the
// backward) on host buffers with two device buffer sets and three streams,
// so that step n+1's inputs go up and step n's results come down while step
// n computes:
//   up:      [wait: set free] H2D q, k, v -> qkv_in; H2D dout -> do_in
//   compute: [wait: qkv_in, set read back] forward -> fwd_done;
//            [wait: do_in] backward -> all_done
//   down:    [wait: fwd_done] D2H out, lse; [wait: all_done] D2H dq, dk, dv
//            -> read_back
// The pages have no counterpart: on one GPU there is no ring transfer, and
// this is the host-side plumbing around the computation they describe.
#include <pthread.h>
#include <sched.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "ra_internal.cuh"

namespace ra {
namespace {

// CPUs of NUMA node `node` from sysfs (a list such as "0-71,144-215").
bool node_cpus(int node, cpu_set_t *set) {
  char path[96];
  snprintf(path, sizeof path, "/sys/devices/system/node/node%d/cpulist", node);
  FILE *f = fopen(path, "r");
  if (f == nullptr) return false;
  char buf[4096];
  const size_t n = fread(buf, 1, sizeof buf - 1, f);
  fclose(f);
  buf[n] = 0;
  CPU_ZERO(set);
  int count = 0;
  const char *p = buf;
  while (*p != 0) {
    char *end = nullptr;
    const long a = strtol(p, &end, 10);
    if (end == p) break;
    long b = a;
    p = end;
    if (*p == '-') {
      ++p;
      b = strtol(p, &end, 10);
      if (end == p) break;
      p = end;
    }
    for (long c = a; c <= b && c < CPU_SETSIZE; ++c)
      if (c >= 0) {
        CPU_SET(static_cast<int>(c), set);
        ++count;
      }
    if (*p != ',') break;
    ++p;
  }
  return count > 0;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace
}  // namespace ra

struct ra_pipeline {
  int device = 0;
  ra_dims dims{};
  int64_t S = 0;
  int n_shards = 0;
  ra_layout layout = RA_LAYOUT_STRIPED;
  int causal = 0;
  float scale = 0.f;
  int backward = 0;
  size_t q_bytes = 0, kv_bytes = 0, o_bytes = 0, lse_bytes = 0, dkv_bytes = 0;
  cudaStream_t up = nullptr, compute = nullptr, down = nullptr;
  struct Set {
    uint16_t *q = nullptr, *k = nullptr, *v = nullptr, *dout = nullptr;
    float *out = nullptr, *lse = nullptr, *dq = nullptr, *dk = nullptr, *dv = nullptr;
    cudaEvent_t qkv_in = nullptr, do_in = nullptr, fwd_done = nullptr, all_done = nullptr,
                read_back = nullptr;
    bool used = false;
  } set[2];
  void *block = nullptr;  // one device allocation holding both sets and the workspace
  void *ws = nullptr;
  size_t ws_bytes = 0;
  uint64_t steps = 0;
};

namespace {

void destroy_pipeline(ra_pipeline *pl) {
  if (pl == nullptr) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(pl->device);
  for (cudaStream_t s : {pl->up, pl->compute, pl->down})
    if (s != nullptr) cudaStreamSynchronize(s);
  for (auto &st : pl->set)
    for (cudaEvent_t e : {st.qkv_in, st.do_in, st.fwd_done, st.all_done, st.read_back})
      if (e != nullptr) cudaEventDestroy(e);
  for (cudaStream_t s : {pl->up, pl->compute, pl->down})
    if (s != nullptr) cudaStreamDestroy(s);
  if (pl->block != nullptr) cudaFree(pl->block);
  if (prev >= 0) cudaSetDevice(prev);
  delete pl;
}

}  // namespace

extern "C" {

ra_status ra_host_alloc(size_t bytes, void **ptr) {
  if (ptr == nullptr) return ra::report_error(RA_ERR_INVALID_ARG, "ptr is NULL");
  *ptr = nullptr;
  if (bytes == 0) return RA_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ra::report_error(RA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  int node = -1;
  if (cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, dev) != cudaSuccess) {
    cudaGetLastError();
    node = -1;
  }
  // The driver takes the pages when it pins them, on the node of the CPU the
  // calling thread runs on: run on the GPU's node for the call.
  cpu_set_t old_set, node_set;
  bool moved = false;
  if (node >= 0 && pthread_getaffinity_np(pthread_self(), sizeof old_set, &old_set) == 0 &&
      ra::node_cpus(node, &node_set))
    moved = pthread_setaffinity_np(pthread_self(), sizeof node_set, &node_set) == 0;
  void *p = nullptr;
  e = cudaHostAlloc(&p, bytes, cudaHostAllocPortable);
  if (moved) pthread_setaffinity_np(pthread_self(), sizeof old_set, &old_set);
  if (e != cudaSuccess)
    return ra::report_error(RA_ERR_CUDA, "cudaHostAlloc(%zu): %s", bytes, cudaGetErrorString(e));
  *ptr = p;
  return RA_OK;
}

ra_status ra_host_free(void *ptr) {
  if (ptr == nullptr) return RA_OK;
  const cudaError_t e = cudaFreeHost(ptr);
  if (e != cudaSuccess) return ra::report_error(RA_ERR_CUDA, "cudaFreeHost: %s", cudaGetErrorString(e));
  return RA_OK;
}

int ra_host_numa_node(void) {
  int dev = 0, node = -1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return node;
}

ra_status ra_pipeline_create(int64_t S, int n_shards, ra_layout layout, int causal, float scale,
                             ra_dims dims, int backward, ra_pipeline **pipeline) {
  if (pipeline == nullptr) return ra::report_error(RA_ERR_INVALID_ARG, "pipeline is NULL");
  *pipeline = nullptr;
  if (S <= 0 || n_shards <= 0 || n_shards > S)
    return ra::report_error(RA_ERR_INVALID_ARG, "need 1 <= n_shards <= S (S=%lld, n_shards=%d)",
                            static_cast<long long>(S), n_shards);
  if (dims.b <= 0 || dims.h <= 0 || dims.n_kv <= 0 || (dims.d != 64 && dims.d != 128) ||
      dims.h % dims.n_kv != 0)
    return ra::report_error(RA_ERR_UNSUPPORTED, "dims b=%d h=%d n_kv=%d d=%d", dims.b, dims.h,
                            dims.n_kv, dims.d);
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_STRIPED && layout != RA_LAYOUT_ZIGZAG)
    return ra::report_error(RA_ERR_INVALID_ARG, "unknown layout %d", static_cast<int>(layout));
  ra_pipeline *pl = new (std::nothrow) ra_pipeline;
  if (pl == nullptr) return ra::report_error(RA_ERR_INVALID_ARG, "out of host memory");
  cudaError_t e = cudaGetDevice(&pl->device);
  pl->dims = dims;
  pl->S = S;
  pl->n_shards = n_shards;
  pl->layout = layout;
  pl->causal = causal;
  pl->scale = scale;
  pl->backward = backward != 0;
  const size_t rows = static_cast<size_t>(dims.b) * S;
  pl->q_bytes = rows * dims.h * dims.d * 2;
  pl->kv_bytes = rows * dims.n_kv * dims.d * 2;
  pl->o_bytes = rows * dims.h * dims.d * 4;
  pl->lse_bytes = rows * dims.h * 4;
  pl->dkv_bytes = rows * dims.n_kv * dims.d * 4;
  pl->ws_bytes = pl->backward ? ra_bwd_workspace_size(S, n_shards, dims) : 0;
  constexpr size_t kAlign = 256;
  size_t per_set = ra::round_up(pl->q_bytes, kAlign) + 2 * ra::round_up(pl->kv_bytes, kAlign) +
                   ra::round_up(pl->o_bytes, kAlign) + ra::round_up(pl->lse_bytes, kAlign);
  if (pl->backward)
    per_set += ra::round_up(pl->q_bytes, kAlign) + ra::round_up(pl->o_bytes, kAlign) +
               2 * ra::round_up(pl->dkv_bytes, kAlign);
  const size_t total = 2 * per_set + ra::round_up(pl->ws_bytes, kAlign);
  if (e == cudaSuccess) e = cudaMalloc(&pl->block, total);
  for (cudaStream_t *s : {&pl->up, &pl->compute, &pl->down})
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  if (e == cudaSuccess) {
    char *cur = static_cast<char *>(pl->block);
    auto take = [&](size_t n) {
      char *r = cur;
      cur += ra::round_up(n, kAlign);
      return r;
    };
    for (auto &st : pl->set) {
      st.q = reinterpret_cast<uint16_t *>(take(pl->q_bytes));
      st.k = reinterpret_cast<uint16_t *>(take(pl->kv_bytes));
      st.v = reinterpret_cast<uint16_t *>(take(pl->kv_bytes));
      st.out = reinterpret_cast<float *>(take(pl->o_bytes));
      st.lse = reinterpret_cast<float *>(take(pl->lse_bytes));
      if (pl->backward) {
        st.dout = reinterpret_cast<uint16_t *>(take(pl->q_bytes));
        st.dq = reinterpret_cast<float *>(take(pl->o_bytes));
        st.dk = reinterpret_cast<float *>(take(pl->dkv_bytes));
        st.dv = reinterpret_cast<float *>(take(pl->dkv_bytes));
      }
      for (cudaEvent_t *ev : {&st.qkv_in, &st.do_in, &st.fwd_done, &st.all_done, &st.read_back})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    }
    pl->ws = pl->ws_bytes > 0 ? take(pl->ws_bytes) : nullptr;
  }
  if (e != cudaSuccess) {
    destroy_pipeline(pl);
    return ra::report_error(RA_ERR_CUDA, "pipeline setup (%zu device bytes): %s", total,
                            cudaGetErrorString(e));
  }
  *pipeline = pl;
  return RA_OK;
}

ra_status ra_pipeline_submit(ra_pipeline *pl, const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, const uint16_t *dout, float *out, float *lse,
                             float *dq, float *dk, float *dv) {
  if (pl == nullptr) return ra::report_error(RA_ERR_INVALID_ARG, "pipeline is NULL");
  if (q == nullptr || k == nullptr || v == nullptr || (pl->backward && dout == nullptr))
    return ra::report_error(RA_ERR_INVALID_ARG, "an input host buffer is NULL");
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != pl->device) cudaSetDevice(pl->device);
  auto &st = pl->set[pl->steps % 2];
  cudaError_t e = cudaSuccess;
  auto enq = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
  };
  // inputs up, once the compute that last read this set has finished
  if (st.used) enq(cudaStreamWaitEvent(pl->up, st.all_done, 0));
  enq(cudaMemcpyAsync(st.q, q, pl->q_bytes, cudaMemcpyHostToDevice, pl->up));
  enq(cudaMemcpyAsync(st.k, k, pl->kv_bytes, cudaMemcpyHostToDevice, pl->up));
  enq(cudaMemcpyAsync(st.v, v, pl->kv_bytes, cudaMemcpyHostToDevice, pl->up));
  enq(cudaEventRecord(st.qkv_in, pl->up));
  if (pl->backward) {
    enq(cudaMemcpyAsync(st.dout, dout, pl->q_bytes, cudaMemcpyHostToDevice, pl->up));
    enq(cudaEventRecord(st.do_in, pl->up));
  }
  // compute, once the inputs are in and this set's last results are read back
  enq(cudaStreamWaitEvent(pl->compute, st.qkv_in, 0));
  if (st.used) enq(cudaStreamWaitEvent(pl->compute, st.read_back, 0));
  if (e != cudaSuccess) {
    if (prev >= 0 && prev != pl->device) cudaSetDevice(prev);
    return ra::report_error(RA_ERR_CUDA, "pipeline copies: %s", cudaGetErrorString(e));
  }
  ra_status rs = ra_ring_attention(st.q, st.k, st.v, st.out, st.lse, pl->S, pl->n_shards,
                                   pl->layout, pl->causal, pl->scale, pl->dims, pl->compute);
  if (rs == RA_OK) {
    enq(cudaEventRecord(st.fwd_done, pl->compute));
    if (pl->backward) {
      enq(cudaStreamWaitEvent(pl->compute, st.do_in, 0));
      rs = ra_ring_attention_bwd(st.q, st.k, st.v, st.out, st.lse, st.dout, st.dq, st.dk, st.dv,
                                 pl->ws, pl->ws_bytes, pl->S, pl->n_shards, pl->layout, pl->causal,
                                 pl->scale, pl->dims, pl->compute);
    }
  }
  if (rs != RA_OK) {
    if (prev >= 0 && prev != pl->device) cudaSetDevice(prev);
    return rs;
  }
  enq(cudaEventRecord(st.all_done, pl->compute));
  // results down: out and lse while the backward runs, the gradients after it
  enq(cudaStreamWaitEvent(pl->down, st.fwd_done, 0));
  if (out != nullptr) enq(cudaMemcpyAsync(out, st.out, pl->o_bytes, cudaMemcpyDeviceToHost, pl->down));
  if (lse != nullptr)
    enq(cudaMemcpyAsync(lse, st.lse, pl->lse_bytes, cudaMemcpyDeviceToHost, pl->down));
  if (pl->backward) {
    enq(cudaStreamWaitEvent(pl->down, st.all_done, 0));
    if (dq != nullptr) enq(cudaMemcpyAsync(dq, st.dq, pl->o_bytes, cudaMemcpyDeviceToHost, pl->down));
    if (dk != nullptr)
      enq(cudaMemcpyAsync(dk, st.dk, pl->dkv_bytes, cudaMemcpyDeviceToHost, pl->down));
    if (dv != nullptr)
      enq(cudaMemcpyAsync(dv, st.dv, pl->dkv_bytes, cudaMemcpyDeviceToHost, pl->down));
  }
  enq(cudaEventRecord(st.read_back, pl->down));
  st.used = true;
  ++pl->steps;
  if (prev >= 0 && prev != pl->device) cudaSetDevice(prev);
  if (e != cudaSuccess)
    return ra::report_error(RA_ERR_CUDA, "pipeline copies: %s", cudaGetErrorString(e));
  return RA_OK;
}

ra_status ra_pipeline_sync(ra_pipeline *pl) {
  if (pl == nullptr) return ra::report_error(RA_ERR_INVALID_ARG, "pipeline is NULL");
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != pl->device) cudaSetDevice(pl->device);
  cudaError_t e = cudaStreamSynchronize(pl->up);
  const cudaError_t e2 = cudaStreamSynchronize(pl->down);
  if (e == cudaSuccess) e = e2;
  // the compute stream last: this also reads and clears the device error word
  ra_status rs = ra_stream_check(pl->compute);
  if (prev >= 0 && prev != pl->device) cudaSetDevice(prev);
  if (rs != RA_OK) return rs;
  if (e != cudaSuccess)
    return ra::report_error(RA_ERR_CUDA, "pipeline sync: %s", cudaGetErrorString(e));
  return RA_OK;
}

ra_status ra_pipeline_destroy(ra_pipeline *pl) {
  destroy_pipeline(pl);
  return RA_OK;
}

}  // extern "C"
