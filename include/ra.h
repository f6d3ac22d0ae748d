/*
 * ra.h -- C ABI of the GB300 blockwise ring-attention engine.
 *
 * The engine computes exact softmax attention, O = softmax(scale * Q K^T) V,
 * the way Ring Attention does: a resident query shard meets the key/value
 * shards one after another in ring order and keeps an online-softmax state
 * per query row (running max m, running sum l, unnormalised output O), then
 * divides by l.  On one GPU the N devices of the ring are N virtual shards of
 * one sequence.
 *
 * Sources (page title, then section):
 *  - "Ring Attention with Blockwise Transformers: Mathematical Foundations,
 *    Circular KV Passing, Overlapped Communication-Computation, and Linear
 *    Context Scaling": "Blockwise Attention and Online Softmax Formulations"
 *    (the update of m, l, O and the final division by l), "The Ring Attention
 *    Protocol" (query block resident, key/value blocks rotate), "Causal
 *    Masking Dynamics" (striped placement t -> t mod N; zig-zag half-blocks
 *    p and 2N-1-p), "The Backward Pass and Gradient Exchange" (P recomputed
 *    from saved statistics), and its closing remark on inference (a short
 *    query chunk against a long resident key/value cache).
 *  - "Ring Attention for Infinite Context": "FlashAttention Integration" (the
 *    rescale-merge of a running output with a block output).
 *  - summary of "Ring Attention with Blockwise Transformers for Near-Infinite
 *    Context": "The Ring Communication Protocol" (host i holds block
 *    (i - idx) mod N on iteration idx), "The Backward Pass: Symmetric Ring
 *    Operation".
 *  - the magicnetworld.com article on ring attention's communication budget,
 *    causal triangle and load imbalance: section 2 (symbols, GQA with h query
 *    heads sharing n_kv KV heads), section 5 (documents packed into one window
 *    with a block-diagonal mask), section 6 (causal mask; contiguous versus
 *    striped placement).
 *
 * Conventions for every call:
 *  - Tensors are dense, row-major, in DEVICE memory, and owned by the caller
 *    (the host-buffer pipeline at the end takes host memory).  The calls
 *    allocate no device memory, except ra_pipeline_create (its buffer sets)
 *    and the allocation-free backward's one fixed array in the library's own
 *    device memory.  Base pointers must be 16-byte aligned.
 *  - bf16 tensors are passed as raw 16-bit patterns (uint16_t).
 *  - Query-side tensors are [b, rows, h, d]; key/value-side tensors are
 *    [b, rows, n_kv, d].  Per-row statistics are [b, h, rows] float.
 *  - GQA: query head hq reads KV head hq / (h / n_kv).
 *  - Causal masking is inclusive: key position <= query position.
 *  - `m` and `lse` are in natural-log units of the scaled logits
 *    scale * <q, k>.  LSE = m + ln(l).  A row that sees no key has l = 0,
 *    O = 0 and LSE = -inf.
 *  - scale <= 0 selects 1/sqrt(d).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues work on it and returns; nothing synchronises.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call launches nothing and leaves every output untouched.
 *  - Device-side waits are bounded; a wait that runs out sets a device error
 *    word, and the kernel unwinds.  ra_stream_check() reports it.
 *  - Supported: d in {64, 128}; h % n_kv == 0; the row counts of one call
 *    below 2^31; n_shards >= 1 with S % n_shards == 0 (zig-zag: S / 2N a
 *    multiple of 128).
 *  - The backward's dq, dk and dv are sums of fp32 partial tiles added in
 *    arrival order: two runs agree to fp32 rounding, not bit for bit.  The
 *    forward calls are deterministic.
 *  - Precision: P (and in the backward dS) reaches the tensor cores as bf16
 *    with fp32 accumulation.  Where that rounding could carry a large share
 *    of a result it goes as a bf16 pair hi + lo (the second term the
 *    rounding residual): in query tiles whose earliest row sees fewer than
 *    512 keys, and in the backward on steps whose P holds an entry above
 *    1/16.  The forward re-references a row's exponent shift to the exact
 *    row max when a key would hold more than 1/9 of the row's weight so far,
 *    so that key's P is exactly 1.
 */
#ifndef RA_H
#define RA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, negative size, bad enum */
  RA_ERR_UNSUPPORTED = 2,     /* shape the kernels do not handle */
  RA_ERR_CUDA = 3,            /* a CUDA runtime call or launch failed */
  RA_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device-side wait ran out */
  RA_ERR_WORKSPACE = 5        /* workspace missing or too small */
} ra_status;

typedef enum {
  RA_LAYOUT_CONTIGUOUS = 0,   /* shard p holds tokens [p*L, (p+1)*L) */
  RA_LAYOUT_STRIPED = 1,      /* shard p holds tokens p, p+N, p+2N, ... */
  RA_LAYOUT_ZIGZAG = 2        /* 2N half-blocks of C = L/2 tokens; shard p holds
                                 half-block p (local rows [0, C)) and half-block
                                 2N-1-p (rows [C, L)): the first page's "Zig-Zag
                                 Ring Attention".  Needs S % (2N) == 0, and for
                                 the attention calls C % 128 == 0. */
} ra_layout;

typedef struct {
  int b;      /* batch */
  int h;      /* query heads */
  int n_kv;   /* key/value heads (h % n_kv == 0) */
  int d;      /* head dimension: 64 or 128 */
} ra_dims;

/* One ring step: fold one key/value block into the online-softmax state of a
 * query block ("Blockwise Attention and Online Softmax Formulations"; the
 * fourth page's "Incremental Blockwise Attention" steps 1-5):
 *   m~ = rowmax(S), m' = max(m, m~), P = exp(S - m'),
 *   l' = exp(m - m') l + rowsum(P),  O' = exp(m - m') O + P V,
 * with S = scale * Q K^T over the visible keys.  The block's contribution is
 * computed on the tensor cores and merged into the state with the second
 * page's rescale-merge, so `m` is the exact running row max afterwards.
 *   q      [b, Lq, h, d] bf16         k, v [b, Lk, n_kv, d] bf16
 *   m, l   [b, h, Lq] float, in/out   o    [b, Lq, h, d] float, in/out
 *   q_pos  [Lq] int32, k_pos [Lk] int32: token positions, used only when
 *          causal != 0 (key c visible to query r iff k_pos[c] <= q_pos[r]).
 * Initial state: m = -inf, l = 0, o = 0.  Rows with no visible key in this
 * block are left unchanged.  Lq or Lk == 0 is a no-op.  A causal step takes
 * at most 8,388,608 keys (each CTA classifies its whole key range once, in
 * shared memory); RA_ERR_UNSUPPORTED above that.  A causal step over at
 * least 16,384 keys is two kernel launches on `stream`: per 128-query tile,
 * the leading key tiles every row sees in full (at least 32 of them, or
 * all) and the one tile after them go through a kernel with only a
 * per-element position mask on that one tile, the rest (if any key of it
 * is visible) through the kernel with the full causal classification;
 * both fold into the state, so no workspace is needed.  Should the second
 * launch fail (RA_ERR_CUDA), the state already holds the first one's part. */
ra_status ra_block_step(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *m,
                        float *l, float *o, const int32_t *q_pos, const int32_t *k_pos,
                        int64_t Lq, int64_t Lk, ra_dims dims, int causal, float scale,
                        void *stream);

/* Finalize ("Blockwise Attention and Online Softmax Formulations": the
 * output is the unnormalised O divided by the row sum l):
 * o <- o / l in place, lse = m + ln(l).  Rows with l == 0 get o = 0 and
 * lse = -inf.  o [b, Lq, h, d]; l, m, lse [b, h, Lq]. */
ra_status ra_finalize(float *o, const float *l, const float *m, float *lse, int64_t Lq,
                      ra_dims dims, void *stream);

/* Rescale-merge of two normalised partial results over disjoint key sets
 * ("FlashAttention Integration" on the second page, with each side's own LSE
 * as its reference value):
 *   mx = max(lse_a, lse_b), w_x = exp(lse_x - mx),
 *   o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = mx + ln(w_a + w_b).
 * A side with lse = -inf contributes nothing.  o_* [b, Lq, h, d] float;
 * lse_* [b, h, Lq] float.  Outputs may alias side a. */
ra_status ra_merge(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                   float *o, float *lse, int64_t Lq, ra_dims dims, void *stream);

/* The whole ring on one GPU: every query shard i visits key/value shards
 * (i - s) mod N for s = 0..N-1 ("The Ring Communication Protocol"), with
 * causal tiles that are fully masked skipped, and finalizes.  One fused
 * launch; the online-softmax state stays in tensor memory.
 *   q [b, S, h, d] bf16, k, v [b, S, n_kv, d] bf16, in natural token order
 *   out [b, S, h, d] float, lse [b, h, S] float, in natural token order.
 * The layout only changes which tokens form a shard (and so the visit order
 * and the masked-tile pattern), never the result.  RA_ERR_UNSUPPORTED for a
 * zig-zag layout whose half-blocks are not whole 128-token tiles. */
ra_status ra_ring_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *out,
                            float *lse, int64_t S, int n_shards, ra_layout layout, int causal,
                            float scale, ra_dims dims, void *stream);

/* Packed documents (the third page's section 5: documents packed end to end
 * into one window, a block-diagonal mask keeping each to itself): as
 * ra_ring_attention / ra_ring_attention_bwd, but a query sees only keys of
 * its own document (and, causal, none after itself).  Key tiles no query of
 * a tile can see are skipped, as causal ones are.
 *   cu_seqlens: device int32 [b][n_docs + 1], document offsets of each batch
 *   row, from 0 to S, non-decreasing (empty documents allowed); the contents
 *   are not checked on the host.  n_docs >= 1.
 * Precision: query tiles with a row that sees fewer than 512 keys (a row
 * near the start of a document) take the hi + lo bf16 path. */
ra_status ra_ring_attention_packed(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   float *out, float *lse, int64_t S, int n_shards,
                                   ra_layout layout, int causal, float scale, ra_dims dims,
                                   const int32_t *cu_seqlens, int n_docs, void *stream);
ra_status ra_ring_attention_packed_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                       const float *out, const float *lse, const uint16_t *dout,
                                       float *dq, float *dk, float *dv, void *workspace,
                                       size_t workspace_bytes, int64_t S, int n_shards,
                                       ra_layout layout, int causal, float scale, ra_dims dims,
                                       const int32_t *cu_seqlens, int n_docs, void *stream);

/* Chunked prefill: Lq new query tokens (positions q_pos) attend to Lk
 * resident keys (positions k_pos) -- the first page's inference remark, a
 * block step with Lq much smaller than Lk.  The keys are cut into n_splits
 * ranges of whole 128-key tiles that run as concurrent block steps, each into
 * its own online-softmax state in the workspace, and the states are combined
 * with the second page's rescale-merge generalised to n parts:
 *   M = max_s m_s, L = sum_s l_s e^(m_s - M), out = sum_s e^(m_s - M) O_s / L,
 *   lse = M + ln L  (rows no key reaches: 0 and -inf).
 *   q [b, Lq, h, d] bf16; k, v [b, Lk, n_kv, d] bf16; q_pos [Lq], k_pos [Lk]
 *   int32 (needed when causal: key visible iff k_pos <= q_pos);
 *   out [b, Lq, h, d] float; lse [b, h, Lq] float (overwritten).
 *   n_splits: 0 picks enough splits to fill the GPU; at most 64.  Under the
 *   causal rule a split covers at most 8,388,608 keys (RA_ERR_UNSUPPORTED
 *   when n_splits leaves more; 0 picks enough).
 *   workspace: device memory of ra_prefill_workspace_size() bytes (same
 *   n_splits), 16-byte aligned, scratch after the call.
 * Under the causal rule the key tiles that every row of a 128-query tile sees
 * in full (all keys at or before the tile's earliest query position) run
 * without the causal mask, and then only the remaining tiles with it, merged
 * into the same split states; the results do not depend on this.
 * Launches three kernels on `stream` (five under the causal rule);
 * RA_ERR_WORKSPACE if the workspace is missing or small.  The pages give no
 * kernel for this case; splitting the keys is this library's way to fill
 * the GPU when Lq is short. */
size_t ra_prefill_workspace_size(int64_t Lq, int64_t Lk, int n_splits, ra_dims dims);
ra_status ra_chunked_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, float *out,
                             float *lse, const int32_t *q_pos, const int32_t *k_pos, int64_t Lq,
                             int64_t Lk, int n_splits, ra_dims dims, int causal, float scale,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace ra_ring_attention_bwd needs: per query row,
 * D = rowsum(dO * O) and the log2-domain LSE, both float, stored per shard
 * with each shard's rows padded to a multiple of 128.  0 if the arguments
 * are invalid or the problem is empty. */
size_t ra_bwd_workspace_size(int64_t S, int n_shards, ra_dims dims);

/* Blockwise backward with recomputation ("The Backward Pass and Gradient
 * Exchange"; "The Backward Pass: Symmetric Ring Operation"):
 *   P = exp(scale Q K^T - LSE), D = rowsum(dO * O),
 *   dV_j += P^T dO, dP = dO V^T, dS = P * (dP - D),
 *   dQ_i += scale dS K,  dK_j += scale dS^T Q.
 * Each key/value tile is visited by the query shards in ring order; dK/dV sum
 * over the g query heads of a KV head.
 *   q, dout [b, S, h, d] bf16; k, v [b, S, n_kv, d] bf16;
 *   out [b, S, h, d] float and lse [b, h, S] float from ra_ring_attention;
 *   dq [b, S, h, d] float, dk, dv [b, S, n_kv, d] float (overwritten).
 *   workspace: device memory of at least ra_bwd_workspace_size() bytes. */
ra_status ra_ring_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                const float *out, const float *lse, const uint16_t *dout,
                                float *dq, float *dk, float *dv, void *workspace,
                                size_t workspace_bytes, int64_t S, int n_shards, ra_layout layout,
                                int causal, float scale, ra_dims dims, void *stream);
/* (dq is zeroed on the stream and then accumulated; the workspace contents
 * need no initialisation and are scratch after the call.) */

/* Bytes of device workspace ra_block_step_bwd needs for Lq query rows:
 * D and the log2-domain LSE per row, rows padded to a multiple of 128. */
size_t ra_block_bwd_workspace_size(int64_t Lq, ra_dims dims);

/* One ring step of the backward ("The Backward Pass and Gradient Exchange":
 * the key/value block travels with its gradient accumulators dK_j, dV_j while
 * dQ_i stays with its query block; "The Backward Pass: Symmetric Ring
 * Operation"): the contribution of one key/value block to the gradients of
 * one query block, with P recomputed from the query rows' final LSE,
 *   P = exp(scale Q K^T - LSE), D = rowsum(dO * O), dS = P * (dP - D),
 *   dq += scale dS K,  dk += scale dS^T Q,  dv += P^T dO
 * (dk, dv summed over the g query heads of each KV head).
 *   q, dout [b, Lq, h, d] bf16;  k, v [b, Lk, n_kv, d] bf16;
 *   out [b, Lq, h, d] float, lse [b, h, Lq] float: the query rows' results
 *     over the WHOLE sequence (ra_finalize after every ring step, or the
 *     matching rows of ra_ring_attention);
 *   dq [b, Lq, h, d], dk, dv [b, Lk, n_kv, d] float: ADDED TO, not
 *     overwritten, so a ring walk accumulates into them step by step;
 *   q_pos [Lq], k_pos [Lk] int32 token positions, increasing along each
 *     block, used only when causal != 0 (key c visible to query r iff
 *     k_pos[c] <= q_pos[r]); a causal row at position t counts as seeing
 *     t + 1 keys for the precision rule below;
 *   workspace: device memory of at least ra_block_bwd_workspace_size(Lq)
 *     bytes, scratch (D and LSE are recomputed by every call).
 * Precision as in ra_ring_attention_bwd: query tiles whose earliest row sees
 * fewer than 512 keys (without the causal rule: Lk < 512) and steps whose
 * P holds an entry above 1/16 go to the tensor cores as bf16 hi + lo pairs.
 * Lq or Lk == 0 is a no-op.  Positions that do not increase give undefined
 * gradients (they are not checked). */
ra_status ra_block_step_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *out, const float *lse, const uint16_t *dout, float *dq,
                            float *dk, float *dv, const int32_t *q_pos, const int32_t *k_pos,
                            int64_t Lq, int64_t Lk, ra_dims dims, int causal, float scale,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Size of the fixed scratch array behind ra_ring_attention_bwd_noalloc. */
#define RA_BWD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* The backward above without a caller-supplied workspace, for callers that
 * cannot allocate device memory where they run it: inside a CUDA-graph
 * capture (cudaMalloc cannot be captured), in plug-ins that only receive
 * tensors from a host framework owning the allocator, or in loops that must
 * not touch an allocator.  The pages have no counterpart to this call; it is
 * a deployment convenience, not part of the method.
 *   Arguments, results and error behaviour are those of
 *   ra_ring_attention_bwd.  The scratch (D and the log2-domain LSE, see
 *   ra_bwd_workspace_size) lives in a file-scope device array of
 *   RA_BWD_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU loading the library
 *   holds until the process exits; problems needing more return
 *   RA_ERR_WORKSPACE with the sizes in ra_last_error(), e.g. b * h * S above
 *   8M query rows when S / n_shards is a multiple of 128.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current): make that first call
 *   outside any stream capture.  The call allocates nothing.
 *   All calls on one device share its array: calls whose work overlaps on
 *   that GPU (for example on two streams) race on it, so order them on one
 *   stream or with events.  Nothing in the array needs to start at zero;
 *   each call writes every word it later reads. */
ra_status ra_ring_attention_bwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                        const float *out, const float *lse, const uint16_t *dout,
                                        float *dq, float *dk, float *dv, int64_t S, int n_shards,
                                        ra_layout layout, int causal, float scale, ra_dims dims,
                                        void *stream);

/* ---- Host buffers.  The pages have no counterpart to these calls: on one
 * GPU there is no ring transfer, and they are the host-side plumbing that
 * moves a step's inputs in and its results out. */

/* Pinned (page-locked) host memory of `bytes`, allocated while the calling
 * thread runs on the CPUs of the NUMA node nearest the current device
 * (cudaDevAttrHostNumaId), so copies do not cross a CPU socket link.  *ptr is
 * NULL for bytes == 0.  Free with ra_host_free.  RA_ERR_CUDA if the pinned
 * allocation fails. */
ra_status ra_host_alloc(size_t bytes, void **ptr);
ra_status ra_host_free(void *ptr);
/* NUMA node nearest the current device, or -1 when unknown. */
int ra_host_numa_node(void);

/* A pipeline of ring-attention steps on host buffers: each submitted step
 * copies q, k, v (and dout) in, runs ra_ring_attention (and
 * ra_ring_attention_bwd), and copies out, lse (and dq, dk, dv) back.  Two
 * device buffer sets and three streams overlap step n+1's input copies and
 * step n's result copies with step n's compute; out and lse leave while the
 * backward runs.  Shapes, dtypes and layouts are those of ra_ring_attention
 * and ra_ring_attention_bwd, in host memory (pinned memory from
 * ra_host_alloc overlaps; pageable memory works but its copies do not).
 * Opaque; one pipeline serves one thread at a time. */
typedef struct ra_pipeline ra_pipeline;

/* Allocates both buffer sets and the backward workspace on the current
 * device (about 2 x (2 + 2 + 4 + 4) x b S h d bytes with the backward).
 * RA_ERR_UNSUPPORTED for dims the kernels do not take, RA_ERR_CUDA if the
 * device allocation fails. */
ra_status ra_pipeline_create(int64_t S, int n_shards, ra_layout layout, int causal, float scale,
                             ra_dims dims, int backward, ra_pipeline **pipeline);

/* Enqueue one step and return.  Inputs: q [b,S,h,d], k, v [b,S,n_kv,d],
 * dout [b,S,h,d] bf16 (dout only with the backward).  Outputs (any may be
 * NULL to skip that copy): out [b,S,h,d], lse [b,h,S], dq [b,S,h,d],
 * dk, dv [b,S,n_kv,d] float.  Every host buffer must stay valid, and the
 * inputs unchanged, until ra_pipeline_sync returns.  Errors of the attention
 * calls are returned as they are; after a non-OK status destroy the
 * pipeline. */
ra_status ra_pipeline_submit(ra_pipeline *pipeline, const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, const uint16_t *dout, float *out, float *lse,
                             float *dq, float *dk, float *dv);

/* Wait for every submitted step (its results are then in the host buffers);
 * reports device timeouts and CUDA errors as ra_stream_check does. */
ra_status ra_pipeline_sync(ra_pipeline *pipeline);

/* Wait, then free the pipeline's device memory, streams and events. */
ra_status ra_pipeline_destroy(ra_pipeline *pipeline);

/* Token placement maps (the third page's section 6 example; "Striped
 * Attention" and "Zig-Zag Ring Attention" on the first page), computed on the
 * device by the same functions the attention kernels use:
 *   shard_of[t], local_of[t] for t in [0, S);  token_of[p * L + r] inverse.
 * Any of the three device pointers may be NULL to skip that map. */
ra_status ra_position_map(ra_layout layout, int64_t S, int n_shards, int32_t *shard_of,
                          int32_t *local_of, int32_t *token_of, void *stream);

/* Ring visit order on the device: order[i * N + s] = key/value shard that
 * query shard i meets at ring step s, (i - s) mod N ("The Ring Communication
 * Protocol", k_block_idx). */
ra_status ra_ring_order(int n_shards, int32_t *order, void *stream);

/* Synchronise `stream`, then read and clear the device error word.  Returns
 * RA_ERR_DEVICE_TIMEOUT if a bounded device wait ran out since the last
 * check, RA_ERR_CUDA on a CUDA error, RA_OK otherwise. */
ra_status ra_stream_check(void *stream);

/* Measurement probe for the second roof of the forward: the exp2 rate of
 * the special-function units (every attention element needs one exp2 beside
 * its two multiply-adds on the tensor cores).  Launches
 * ra_ex2_probe_threads() threads, 4 CTAs of 256 per SM, each evaluating
 * 8 * iters dependent-chain exp2 (ex2.approx) and writing one float to
 * sink[thread]; the caller times the launch.  iters in 1 .. 2^24;
 * sink_floats must be at least ra_ex2_probe_threads().  The pages have no
 * counterpart to this call; it supports the roofline report only. */
ra_status ra_ex2_probe(int64_t iters, float *sink, int64_t sink_floats, void *stream);
int64_t ra_ex2_probe_threads(void);

/* Failure-detection self test: launches one CTA that waits on an mbarrier
 * nothing will ever arrive on, with a wait budget of `budget_cycles` SM
 * clocks (1 .. 2^31).  The wait runs out, the kernel records a timeout and
 * returns; ra_stream_check() must then report RA_ERR_DEVICE_TIMEOUT. */
ra_status ra_selftest_wait_timeout(long long budget_cycles, void *stream);

/* Number of kernels this library has launched in this process (all entry
 * points, all threads).  Lets a caller count the device work a region did. */
uint64_t ra_launch_count(void);

/* Message for the last non-OK status returned on the calling thread. */
const char *ra_last_error(void);

/* Library ABI version (major * 100 + minor). */
int ra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H */
