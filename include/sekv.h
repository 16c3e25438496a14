/*
 * sekv.h -- C ABI of libsekv, a GB300 (sm_103a) implementation of the
 * decode hot path of SeKV ("SeKV: Resolution-Adaptive KV Cache with
 * Hierarchical Semantic Memory for Long-Context LLM Inference"), and of the
 * prefill build of its span cache.
 *
 * Sources, cited per call as "page, section":
 *   [DE] gist.science, German explainer of the paper, "Technisches Resuemee":
 *        Methodik 1 (entropy-guided span segmentation), 2 (dual-resolution
 *        span representation), 3 (trained zoom-in, mixed-resolution
 *        attention); Problemstellung (the problem statement).
 *   [ZH] gist.science, Chinese explainer, "技术摘要": 方法论 1, 2, 3; 问题陈述.
 *   [EN] the paper's English abstract.
 *
 * General rules
 *   - Every pointer is caller-owned.  Device pointers are CUDA device
 *     memory of the current device unless a field says "host".  The library
 *     keeps no pointer after a call returns.
 *   - No call allocates device memory.  Scratch comes from a caller-owned
 *     workspace of sekv_workspace_size() bytes that must be zeroed once with
 *     sekv_workspace_init(); every call leaves it ready for the next call.
 *     One workspace serves one stream at a time: two calls that use the same
 *     workspace must not overlap on the GPU.
 *   - Calls are asynchronous on the given stream.  Argument errors are
 *     detected on the host before any launch and returned; nothing is
 *     launched then.  Errors the GPU detects (a bad index in a list, a
 *     capacity overflow, a wait that ran out) set a status word in the
 *     workspace; sekv_workspace_status() synchronises and reports it.
 *   - Sizes are fixed: head_dim == 128, route_dim == 64, at most 8 query
 *     heads per KV head, ranks at most 64.  Other values give
 *     SEKV_ERR_UNSUPPORTED.
 *   - bf16 means IEEE bfloat16 stored as 16-bit patterns.
 */
#ifndef SEKV_H_
#define SEKV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SEKV_HEAD_DIM 128
#define SEKV_ROUTE_DIM 64
#define SEKV_MAX_GROUP 8
#define SEKV_MAX_RANK 64
#define SEKV_MAX_QUERY_TOKENS 64 /* query tokens per sequence of sekv_decode_step_multi */

typedef enum sekv_status {
  SEKV_OK = 0,
  SEKV_ERR_INVALID = -1,      /* bad argument (null pointer, negative size, misalignment) */
  SEKV_ERR_CAPACITY = -2,     /* a caller buffer or the workspace is too small */
  SEKV_ERR_CUDA = -3,         /* a CUDA runtime call failed */
  SEKV_ERR_TIMEOUT = -4,      /* a bounded wait ran out (host or device) */
  SEKV_ERR_UNSUPPORTED = -5,  /* a size the library does not implement */
  SEKV_ERR_DEVICE = -6        /* the GPU flagged bad data (see sekv_workspace_status) */
} sekv_status;

/* Shapes and hyper-parameters shared by every call. */
typedef struct sekv_config {
  int32_t batch;       /* B: sequences */
  int32_t n_q_heads;   /* Hq: query heads; a multiple of n_kv_heads, Hq/Hkv <= 8 */
  int32_t n_kv_heads;  /* Hkv */
  int32_t head_dim;    /* must be 128 */
  int32_t route_dim;   /* must be 64 */
  int32_t n_sink;      /* full-resolution tokens at the start of the context */
  int32_t n_recent;    /* full-resolution tokens at the end of the context */
  int32_t max_spans;   /* capacity of every per-sequence span array; a multiple of 64 */
  int32_t rank_cap;    /* R: largest rank a span basis may keep (<= 64) */
  int32_t len_min;     /* segmentation: shortest span (anchor included) unless cut by the end */
  int32_t len_max;     /* segmentation: longest span (anchor included) */
  float tau;           /* segmentation: surprisal threshold (strict >) */
  int32_t flags;       /* SEKV_FLAG_* bits, 0 for none */
} sekv_config;

/* sekv_decode_step may start streaming this layer's cache and its routing
 * weights W_r (never q or theta) before the kernel that precedes it on the
 * stream has finished (programmatic dependent launch).  Set it only when no
 * preceding kernel on the stream writes this layer's cache or W_r; it hides
 * launch gaps between layers. */
#define SEKV_FLAG_OVERLAP_PREVIOUS 1

/* Fault-path testing only: every wait of a decode kernel for a copy to land
 * gives up at once if the copy has not landed when it is first tested
 * (normally it waits up to about two seconds).  Some wait then runs out, the
 * call's results are unreliable and sekv_workspace_status reports
 * SEKV_ERR_TIMEOUT (code 2); the kernel still waits, within its own bound,
 * for every copy it issued before it exits, so the GPU and the workspace
 * stay usable for the next call. */
#define SEKV_FLAG_SHORT_WAITS 2

/*
 * One layer of the span cache.  [DE]/[ZH] Methodik 2 and 3: per span the GPU
 * holds an anchor token at full resolution, a routing summary and (this
 * build's reading of the "size-corrected summary") a summary key/value; the
 * low-rank basis lives in the basis store, on the host or in device memory.
 *
 * Index names: b sequence, c KV head, k span ordinal, g = b*Hkv + c.
 *   n_spans   int32 [B]                   spans of sequence b (<= max_spans)
 *   body_len  int32 [B][max_spans]        |S_k|, tokens strictly between
 *                                         anchor k and the next span's anchor;
 *                                         0 means the span has no body
 *   k_full,   bf16 [B][Hkv][n_full_cap][128], n_full_cap = n_sink + max_spans
 *   v_full                                + n_recent.  Rows of group g: the
 *                                         n_sink sinks, the n_spans[b] anchors
 *                                         in span order, the n_recent recent
 *                                         tokens; rows past those must hold
 *                                         finite values (zero them)
 *   s_route   f32  [B][Hkv][max_spans][64]  unit routing summaries
 *   k_sum,    bf16 [B][Hkv][max_spans][128] summary keys / values (finite)
 *   v_sum
 *   rec_off   int64 [B][Hkv][max_spans]   byte offset of span k's basis
 *                                         record in `store` (multiple of 16)
 *   rec_rank  int32 [B][Hkv][max_spans]   rK | (rV << 16), the record's ranks
 *   store     basis records; device memory, or host memory (store_on_host=1)
 *             that the device can address (pinned and mapped)
 *
 * Basis record of a span with body b >= 1 and ranks rK, rV ([DE]/[ZH]
 * Methodik 2: truncated SVD K_S ~ U_K diag(sigma_K g_K) Vt_K with soft gates
 * g; likewise V).  All offsets relative to the record start, every field
 * 16-byte aligned, r4(r) / r8(r) = r rounded up to a multiple of 4 / 8.
 * Padding entries must be zero (the GPU reads them):
 *   int32 b, rK, rV, 0                          16 bytes
 *   f32  sigma_K[r4(rK)], f32 g_K[r4(rK)]       8*r4(rK)
 *   bf16 Vt_K[rK][128]                          256*rK
 *   bf16 U_K[b][r8(rK)]  (row-major, columns    2*b*r8(rK)
 *                         rK.. zero)
 *   bf16 U_V[b][r8(rV)]                         2*b*r8(rV)
 *   f32  sigma_V[r4(rV)], f32 g_V[r4(rV)]       8*r4(rV)
 *   bf16 Vt_V[rV][128]                          256*rV
 * Vt rows are stored swizzled: row j's 128 values form sixteen 16-byte
 * chunks (chunk c = columns 8c..8c+7), and chunk c is stored at chunk
 * position c ^ (j & 7) of the row (so that eight consecutive rows read the
 * same columns from eight different shared-memory banks).  U rows likewise:
 * token row t of a U block has W = r8(r) / 8 chunks, and chunk c is stored at
 * chunk position c ^ m(t), m(t) = (t >> (3 - log2 g)) & (g - 1) with g the
 * largest power of two dividing W (m = 0 for odd W; t & 7 for W = 8).
 * Record size = the sum of the right-hand column (sekv_record_size).
 */
typedef struct sekv_layer_cache {
  const int32_t* n_spans;
  const int32_t* body_len;
  const void* k_full;
  const void* v_full;
  const float* s_route;
  const void* k_sum;
  const void* v_sum;
  const int64_t* rec_off;
  const int32_t* rec_rank;
  const void* store;
  int32_t store_on_host;
  /* Optional (NULL: n_recent for every sequence).  int32 [B]: the number of
   * full-resolution rows after the anchors of sequence b.  A cache kept up to
   * date during decode (sekv_append_token) holds the open span -- its anchor
   * and body, not yet closed by a next anchor -- at full resolution in front
   * of the recent window, so its tail is n_recent plus the open span's
   * length; all rows still fit the n_full_cap rows of each group. */
  const int32_t* n_tail;
} sekv_layer_cache;

/* Which call a workspace is sized for. */
typedef enum sekv_call {
  SEKV_CALL_ROUTE = 0,
  SEKV_CALL_FETCH = 1,
  SEKV_CALL_DECODE = 2,   /* sekv_decode_attention and sekv_decode_step */
  SEKV_CALL_BUILD = 3
} sekv_call;

/* Bytes of one basis record (0 when body <= 0); see the layout above. */
int64_t sekv_record_size(int32_t body, int32_t rank_k, int32_t rank_v);

/* Workspace bytes the given call needs for this configuration; ctx_len is
 * used by SEKV_CALL_BUILD only.  Returns 0 for an invalid configuration. */
size_t sekv_workspace_size(const sekv_config* cfg, int32_t which, int64_t ctx_len);

/* Zero a workspace (cudaMemsetAsync on `stream`).  Needed once, before the
 * workspace's first use. */
sekv_status sekv_workspace_init(void* workspace, size_t bytes, cudaStream_t stream);

/* Synchronise `stream`, copy the workspace's device status into *code and
 * *detail (either may be NULL) and clear it.  Returns SEKV_OK when the GPU
 * flagged nothing, SEKV_ERR_DEVICE or SEKV_ERR_TIMEOUT when it did.  The
 * first error of a call wins:
 *   code 1  bad input: an expansion list not ascending, out of range or
 *           naming an empty body (detail: the list position, or the
 *           (sequence, KV head) whose count is out of range), or a build
 *           that found more spans than max_spans (detail: the sequence);
 *   code 2  a bounded wait ran out (SEKV_ERR_TIMEOUT; detail: which wait --
 *           3 copies still landing when a warp drains before exit, 4 a warp
 *           waiting for its next page or record, 5 the routing weights or a
 *           routing page landing, 7 partials landing in the merge);
 *   code 3  the records do not fit: a fetch group's records exceed its
 *           staging share (detail: the group), or a build's records exceed
 *           the store (detail: the bytes needed, in MiB);
 *   code 4  a record rank above what the kernel handles (detail: the rank; the
 *           record is skipped). */
sekv_status sekv_workspace_status(void* workspace, cudaStream_t stream,
                                  int32_t* code, int32_t* detail);

/*
 * sekv_route -- zoom-in routing of one layer.
 * [DE]/[ZH] Methodik 3: the query is projected into the routing space of the
 * span summaries; a sigmoid gate scores each span; a learned per-head,
 * per-layer threshold decides whether it is expanded.  Readings: y_h =
 * W_r[c] q_h for query head h of KV head c = h / (Hq/Hkv); z_{h,k} = y_h .
 * s_route[b][c][k]; head h expands span k iff z_{h,k} > theta[h] (theta in
 * logit space, so this is sigmoid(z) > sigmoid(theta)); KV head c expands
 * the union over its query heads; spans with body_len 0 never expand.
 *   q        bf16 [B][Hq][128]
 *   W_r      f32  [Hkv][64][128]
 *   theta    f32  [Hq]
 *   expanded int32 [B][Hkv][max_spans]  out: ascending span ordinals
 *   n_expanded int32 [B][Hkv]           out: list lengths
 *   z_out    f32  [B][Hq][max_spans]    out, optional (NULL): the logits
 * Deterministic: the lists are bit-reproducible.
 */
sekv_status sekv_route(const sekv_config* cfg, const sekv_layer_cache* cache,
                       const void* q, const float* W_r, const float* theta,
                       int32_t* expanded, int32_t* n_expanded, float* z_out,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * sekv_fetch_bases -- copy the basis records of the expanded spans from the
 * host tier into device staging memory.  [DE]/[ZH] Methodik 3: an expanded
 * span's basis is loaded asynchronously from the CPU; the Bedeutung section
 * names the CPU-GPU bandwidth as the method's cost.
 * The cache's store must be host memory the device can address.  A gather
 * kernel reads the records over the host link and writes them to `staging`:
 * group g's records go to [g*staging_per_group, (g+1)*staging_per_group),
 * packed in list order; staged_off[g][e] receives the byte offset of list
 * entry e (relative to `staging`).  Runs on `stream`; use a side stream and
 * an event to overlap it with other work.
 *   expanded, n_expanded  device lists from sekv_route
 *   staging               device, >= B*Hkv*staging_per_group bytes, 16-aligned
 *   staged_off            int64 [B][Hkv][max_spans] (device, out)
 * A group whose records exceed staging_per_group sets SEKV_ERR_CAPACITY in the
 * workspace status and copies none of that group's records.
 */
sekv_status sekv_fetch_bases(const sekv_config* cfg, const sekv_layer_cache* cache,
                             const int32_t* expanded, const int32_t* n_expanded,
                             void* staging, int64_t staging_per_group,
                             int64_t* staged_off, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * sekv_fetch_bases_copy -- the same fetch driven from the host: one
 * cudaMemcpyAsync per run of adjacent records, on `copy_stream`, then the
 * record offsets, then `done` is recorded on `copy_stream` (the caller makes
 * the attention's stream wait on it).  [DE]/[ZH] Methodik 3: the expanded
 * span's basis is loaded asynchronously from the CPU.
 * The expansion lists and the record offsets must be on the host: this is
 * the path's one device-to-host control crossing per layer (the caller copies
 * sekv_route's lists back and synchronises before the call).  Records of list
 * entries whose store offsets follow each other are copied together.
 *   cache                 store on the host (pinned); only store is read
 *   expanded_host, n_expanded_host   host copies of sekv_route's lists
 *   rec_off_host          host copy of cache->rec_off, int64 [B][Hkv][max_spans]
 *   staging, staging_per_group       as in sekv_fetch_bases
 *   staged_off_host       pinned host scratch, int64 [B][Hkv][max_spans]
 *   staged_off            device, int64 [B][Hkv][max_spans] (out, as in
 *                         sekv_fetch_bases, copied from staged_off_host)
 *   n_copies              out (may be NULL): the record copies issued
 * Record sizes come from the records' headers in the host store.  A group
 * whose records exceed staging_per_group, a list entry out of range, or a
 * header that disagrees with the span returns SEKV_ERR_CAPACITY or
 * SEKV_ERR_INVALID before any copy is issued.  The host blocks only to issue
 * the copies; nothing waits for them.
 */
sekv_status sekv_fetch_bases_copy(const sekv_config* cfg, const sekv_layer_cache* cache,
                                  const int32_t* expanded_host, const int32_t* n_expanded_host,
                                  const int64_t* rec_off_host, void* staging,
                                  int64_t staging_per_group, int64_t* staged_off_host,
                                  int64_t* staged_off, int32_t* n_copies,
                                  cudaStream_t copy_stream, cudaEvent_t done);

/*
 * Residency cache of basis records in device memory, kept from call to call
 * (this library's answer to the pages' CPU-GPU bandwidth limit, [DE] Bedeutung
 * / [ZH] 意义: an expanded span whose record is still resident costs no
 * host-link traffic).  Per (sequence, KV head) group: n_slots slots of
 * slot_bytes each, a table span -> slot, and for every slot its span and the
 * last call that used it.  Records larger than a slot are never cached.
 * The slots live right after the staging area in the caller's staging
 * buffer: group g's slot s starts at byte
 *   B*Hkv*staging_per_group + (g*n_slots + s)*slot_bytes
 * of `staging`, so staged offsets of cached and uncached records share one
 * base.  The table lives in a caller buffer of sekv_basis_cache_bytes()
 * bytes, which sekv_basis_cache_init() sets to "empty" (once, before the first
 * fetch).  One cache serves one layer's store.
 */
size_t sekv_basis_cache_bytes(const sekv_config* cfg, int32_t n_slots);
sekv_status sekv_basis_cache_init(const sekv_config* cfg, void* table, int32_t n_slots,
                                  cudaStream_t stream);

/*
 * sekv_fetch_bases_cached -- sekv_fetch_bases through the residency cache.
 * For each list entry: a span whose record is resident (hit) gets its slot's
 * offset; a miss that fits a slot takes a slot that no entry of this call
 * uses (the first such slots from the group's clock hand on, evicting what
 * they held) and its record is copied there from the host store; a miss that
 * does not fit a slot, or finds no free slot, is copied to the staging area
 * as in sekv_fetch_bases.  Two kernels on `stream` (plan, then copy).
 *   staging     device, >= B*Hkv*(staging_per_group + n_slots*slot_bytes)
 *   slot_bytes  multiple of 16
 *   hits        int32 [B][Hkv] (device, out, may be NULL): hits per group
 *   copied      int64 [B][Hkv] (device, out, may be NULL): record bytes this
 *               call copies over the host link, per group
 * Errors as in sekv_fetch_bases (the staging share per group applies to the
 * records that do not go to slots).
 */
sekv_status sekv_fetch_bases_cached(const sekv_config* cfg, const sekv_layer_cache* cache,
                                    const int32_t* expanded, const int32_t* n_expanded,
                                    void* staging, int64_t staging_per_group, void* table,
                                    int32_t n_slots, int32_t slot_bytes, int64_t* staged_off,
                                    int32_t* hits, int64_t* copied, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/*
 * sekv_decode_attention -- mixed-resolution attention of one layer for a
 * given expansion list.  [DE]/[ZH] Methodik 3: sink, anchor and recent rows
 * enter with their full K/V; an unexpanded span with body >= 1 enters once
 * with its summary key/value and the size correction ln|S| added to its
 * logit; an expanded span enters with every token of its body rebuilt from
 * its basis, khat = U_K diag(sigma_K g_K) Vt_K (likewise vhat).  The kernel
 * scores expanded spans in factor space and never forms khat or vhat.
 *   q          bf16 [B][Hq][128]
 *   expanded, n_expanded  ascending lists (device), e.g. from sekv_route
 *   staging, staged_off   NULL: records are read from cache->store (device);
 *                         else the record of list entry e of group g is at
 *                         staging + staged_off[g*max_spans + e]
 *   scale      logit scale (1/sqrt(128) for standard attention)
 *   out        f32 [B][Hq][128]; lse f32 [B][Hq] (natural log; may be NULL)
 */
sekv_status sekv_decode_attention(const sekv_config* cfg, const sekv_layer_cache* cache,
                                  const void* q, const int32_t* expanded,
                                  const int32_t* n_expanded, const void* staging,
                                  const int64_t* staged_off, float scale, float* out,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/*
 * sekv_decode_step -- routing and mixed-resolution attention of one layer in
 * one kernel, bases read from device memory (cache->store_on_host == 0).
 * Same results as sekv_route followed by sekv_decode_attention.  Optional
 * outputs expanded/n_expanded (NULL to skip) receive the ascending lists.
 */
sekv_status sekv_decode_step(const sekv_config* cfg, const sekv_layer_cache* cache,
                             const void* q, const float* W_r, const float* theta,
                             float scale, float* out, float* lse, int32_t* expanded,
                             int32_t* n_expanded, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * sekv_decode_step_multi -- sekv_decode_step for n_q query tokens per
 * sequence over the same cache (for example the draft tokens of speculative
 * decoding, or queries that share one prefix).  Each query token routes and
 * attends on its own, as [DE]/[ZH] Methodik 3 describe for one query: its
 * expansion set is the union over its GQA group's heads, its expanded spans
 * contribute their reconstructed tokens and its other spans their summaries.
 * Each (token, head) pair is one column of the kernel's tensor-core tiles,
 * eight columns per launch: the tokens go in blocks of 8 / (n_q_heads /
 * n_kv_heads) (sekv_query_blocks(cfg, n_q) blocks), one launch per block in
 * stream order.  The tokens of a block share one pass over the cache: the
 * union of their expansion sets is loaded once.
 *   n_q  1 .. SEKV_MAX_QUERY_TOKENS (else SEKV_ERR_UNSUPPORTED)
 *   q    bf16 [B][n_q][Hq][128];  out f32 [B][n_q][Hq][128];  lse f32
 *        [B][n_q][Hq] (nullable); theta, W_r and workspace as
 *        sekv_decode_step.
 *   expanded, n_expanded  optional (NULL to skip): per block k, the
 *        ascending union over the block's tokens, at expanded[k][g][...]
 *        ([blocks][B*Hkv][max_spans]) and n_expanded[k][g] ([blocks][B*Hkv]).
 * n_q = 1 is sekv_decode_step.
 */
/*
 * sekv_query_blocks -- launches (blocks of query tokens) that
 * sekv_decode_step_multi makes for n_q tokens: ceil(n_q / (8 / (n_q_heads /
 * n_kv_heads))); 0 for an invalid configuration.  Host only.
 */
int32_t sekv_query_blocks(const sekv_config* cfg, int32_t n_q);

sekv_status sekv_decode_step_multi(const sekv_config* cfg, const sekv_layer_cache* cache,
                                   const void* q, int32_t n_q, const float* W_r,
                                   const float* theta, float scale, float* out, float* lse,
                                   int32_t* expanded, int32_t* n_expanded, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/*
 * sekv_decode_step_noalloc -- sekv_decode_step without a caller workspace.
 * The SeKV pages have no counterpart for this call; it exists for callers
 * that cannot allocate device memory and have no spare buffer to lend: for
 * example a plugin inside a serving engine that has already handed every byte
 * of the GPU to its own memory pool, or a decode loop that must not call
 * cudaMalloc (which can synchronise the whole device) between tokens.
 * Instead of a workspace the call uses one scratch array of
 * SEKV_NOALLOC_SCRATCH_BYTES (8 MiB) that the library keeps in device memory
 * on every GPU that loads it, for the life of the process; nothing is
 * allocated or freed, by the library or anything it calls.
 *   - Limit: the configuration must need at most SEKV_NOALLOC_SCRATCH_BYTES of
 *     scratch, i.e. sekv_workspace_size(cfg, SEKV_CALL_DECODE, 0) <= 8 MiB
 *     (e.g. batch 1 x 8 KV heads x 4 160 spans needs about 2 MiB); larger
 *     shapes return SEKV_ERR_CAPACITY before anything is launched.
 *   - The first call on a device looks up the array's device address (once
 *     per device and context, with that device current); make that first
 *     call before any stream capture.  After a device reset (cudaDeviceReset)
 *     the next call looks the address up again, so it too must come before
 *     any capture.
 *   - All calls on a device share the one array, which keeps the previous
 *     call's contents; every call clears the counters it needs.  Calls that
 *     overlap on the GPU (other streams, other threads) race on it and give
 *     wrong results: serialise them.
 *   - Errors the GPU detects are not reported by this call; the status word
 *     lives in the shared array, and sekv_noalloc_status reads it (after the
 *     call's work has finished, before the next call clears it).
 * Arguments, layouts and results are those of sekv_decode_step; flags in
 * cfg are ignored (no overlap with the preceding kernel).
 */
#define SEKV_NOALLOC_SCRATCH_BYTES (8u << 20)
sekv_status sekv_decode_step_noalloc(const sekv_config* cfg, const sekv_layer_cache* cache,
                                     const void* q, const float* W_r, const float* theta,
                                     float scale, float* out, float* lse, int32_t* expanded,
                                     int32_t* n_expanded, cudaStream_t stream);

/* The status word of the no-alloc scratch array on the current device (no
 * counterpart on the pages either): synchronises `stream`, then reads and
 * clears it like sekv_workspace_status -- *code 0 and SEKV_OK when the GPU
 * found nothing, else the device error code and its detail, and
 * SEKV_ERR_TIMEOUT or SEKV_ERR_DEVICE.  Read it after a
 * sekv_decode_step_noalloc call on that stream and before the next one. */
sekv_status sekv_noalloc_status(cudaStream_t stream, int32_t* code, int32_t* detail);

/* Outputs of sekv_build_spans: one layer of the cache (layouts as in
 * sekv_layer_cache; every array with its full capacity) plus the device
 * basis store and its capacity in bytes. */
typedef struct sekv_cache_out {
  int32_t* n_spans;
  int32_t* body_len;
  void* k_full;
  void* v_full;
  float* s_route;
  void* k_sum;
  void* v_sum;
  int64_t* rec_off;
  int32_t* rec_rank;
  void* store;
  int64_t store_capacity;
} sekv_cache_out;

/*
 * sekv_build_spans -- prefill build of one layer's span cache.
 * [DE]/[ZH] Methodik 1: surprisal H_t = -log p(x_t | x_<t) from the prefill
 * pass (an input here) marks span boundaries; boundary tokens are anchors kept
 * at full resolution; a span is the run of tokens between two anchors.
 * Readings: the first middle token (index n_sink) opens span 0; token t opens
 * a new span iff (H_t > tau and t - s >= len_min) or t - s == len_max, s the
 * current span's anchor; the last span ends at ctx_len - n_recent.
 * [DE]/[ZH] Methodik 2: per span a routing summary s = u / |u| with
 * u = sum_i H_i W_r k_i over the body, summary key/value = the body means
 * (bf16, round to nearest even), and a truncated SVD basis per K and V with
 * the caller's soft gates: rank = longest prefix of components (descending
 * sigma) whose gate exceeds 0.5, at most min(rank_cap, |S|).
 *   K, V   bf16 [B][Hkv][ctx_len][128]    H f32 [B][ctx_len]
 *   W_r    f32 [Hkv][64][128]
 *   gates  f32 [B][Hkv][2][max_spans][rank_cap] (index 0 keys, 1 values)
 * Records are packed group by group in span order from the start of
 * out->store.  More than max_spans spans in a sequence, or records beyond
 * store_capacity, set a device status (SEKV_ERR_DEVICE from
 * sekv_workspace_status); the cache is then incomplete.
 * Workspace: sekv_workspace_size(cfg, SEKV_CALL_BUILD, ctx_len).
 */
sekv_status sekv_build_spans(const sekv_config* cfg, int64_t ctx_len, const void* K,
                             const void* V, const float* H, const float* W_r,
                             const float* gates, const sekv_cache_out* out, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Measurement helper (no counterpart on the pages): synchronise `stream` and
 * return in *flops the fp32 operations (an fma counts 2) that the span SVDs
 * of the sekv_build_spans calls on this build workspace performed since the
 * last read -- Gram matrices, the Jacobi sweeps actually run, projections --
 * then clear the count.  For reporting the build's arithmetic rate. */
sekv_status sekv_build_flops(void* workspace, cudaStream_t stream, int64_t* flops);

/*
 * Decode-time maintenance of one layer's cache.  The pages describe the cache
 * built at prefill and the zoom-in during decode, not how the cache follows
 * the tokens that decoding appends; these calls take this reading of them:
 * the GPU keeps the very last part of the text at full resolution ([DE]
 * explainer part 2 / [ZH] 两层记忆), so each new token joins the recent
 * window; the token leaving the window continues the segmentation walk of
 * Methodik 1 (it opens a span iff (H_t > tau and the open span's length >=
 * len_min) or that length == len_max); a span is the run of tokens between
 * two neighbouring anchors, so it can be built (routing summary, summary
 * key/value, gated SVD basis: Methodik 2) once the next anchor closes it.
 * Closed spans wait, with the open span -- anchor and body -- at full
 * resolution at the head of the tail (sekv_layer_cache.n_tail) until
 * sekv_maint_flush builds them.  After every append or flush the cache
 * equals the prefill build of the same prefix whose recent window is taken
 * to start at the anchor of the first span not yet built.
 *
 * The maintained cache is a sekv_cache_out of the prefill build plus
 * n_tail (int32 [B], caller-owned) and a state buffer of
 * sekv_maint_state_size bytes (caller-owned, kept between calls; it holds the
 * open anchors, the surprisal of the tail tokens and the end of the records in
 * `store`).  Records of closing spans are appended after the last record in
 * `store`.  The workspace is a build workspace (SEKV_CALL_BUILD); device
 * errors go to its status word (code 3: no room left -- rows, spans or store
 * -- with the sequence or the MiB needed as detail).  All sequences of the
 * batch start from the same length (sekv_maint_init's ctx_len).
 */
size_t sekv_maint_state_size(const sekv_config* cfg);

/* Starts maintenance of a cache that sekv_build_spans built from K, V, H of
 * length ctx_len (same arguments): the build's last span, which the end of
 * the middle region closed, is open again -- its anchor and body return to
 * full resolution from K and V, and n_tail and the state are set. */
sekv_status sekv_maint_init(const sekv_config* cfg, int64_t ctx_len, const void* K,
                            const void* V, const float* H, const sekv_cache_out* out,
                            int32_t* n_tail, void* state, size_t state_bytes, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/* Appends one token to every sequence: k_new, v_new bf16 [B][Hkv][128]
 * (16-byte aligned), h_new f32 [B] its surprisal.  The token joins the tail;
 * the token leaving the recent window continues the segmentation walk, and a
 * span this closes waits in the tail (at full resolution) until
 * sekv_maint_flush builds it.  At most 128 closed spans per sequence may wait
 * (then flush first: an append that would close one more sets device error
 * code 3 and does not close it).  The sequence lengths live in the state
 * (set by sekv_maint_init, advanced by each call), so a decode loop can
 * capture this call in a CUDA graph.  The cache (out, n_tail) is updated in
 * place on `stream`; read it with a sekv_layer_cache that carries n_tail. */
sekv_status sekv_append_token(const sekv_config* cfg, const void* k_new, const void* v_new,
                              const float* h_new, const sekv_cache_out* out, int32_t* n_tail,
                              void* state, size_t state_bytes, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Builds every closed span waiting in the tails (Methodik 2: routing summary,
 * summary key/value, gated SVD basis, with W_r and gates as sekv_build_spans,
 * gates indexed by span ordinal) as the next span ordinals of each sequence;
 * their body rows leave full resolution.  Flushing after every append builds
 * each span as soon as it closes; flushing every few tokens batches the
 * builds (the cache between flushes holds the waiting spans at full
 * resolution, which is the same prefill build with a longer tail). */
sekv_status sekv_maint_flush(const sekv_config* cfg, const float* W_r, const float* gates,
                             const sekv_cache_out* out, int32_t* n_tail, void* state,
                             size_t state_bytes, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/* Human-readable name of a status. */
const char* sekv_status_string(sekv_status status);

/* Number of kernels the last successful call on this thread launched. */
int32_t sekv_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SEKV_H_ */
