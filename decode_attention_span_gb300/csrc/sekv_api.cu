// C-ABI entry points of libsekv (decode side).  Argument checking, workspace
// layout, TMA tensor-map encoding and kernel launches.  No call allocates.
#include <string.h>

#include <mutex>

#include "decode_attn.cuh"
#include "host_common.h"
#include "route_fetch.cuh"
#include "decode_host.h"

using namespace sekv;

namespace sekv {

thread_local int32_t g_launches = 0;

bool config_ok(const sekv_config* cfg, sekv_status* why) {
  if (!cfg) { *why = SEKV_ERR_INVALID; return false; }
  if (cfg->head_dim != 128 || cfg->route_dim != 64) { *why = SEKV_ERR_UNSUPPORTED; return false; }
  if (cfg->batch < 1 || cfg->n_kv_heads < 1 || cfg->n_q_heads < 1 || cfg->n_sink < 0 ||
      cfg->n_recent < 0 || cfg->max_spans < 64 || cfg->max_spans % 64 != 0 ||
      cfg->n_q_heads % cfg->n_kv_heads != 0 || cfg->batch > 65535 || cfg->n_kv_heads > 65535) {
    *why = SEKV_ERR_INVALID;
    return false;
  }
  // the routing kernel concatenates at most kRouteMaxChunks slices
  if (cfg->max_spans > kRouteChunk * kRouteMaxChunks) {
    *why = SEKV_ERR_UNSUPPORTED;
    return false;
  }
  // the kernels split rows and spans among CTAs in 32-bit arithmetic
  if ((2 * int64_t(cfg->n_sink + cfg->n_recent) + 5 * int64_t(cfg->max_spans)) * 256 >=
      (int64_t(1) << 31)) {
    *why = SEKV_ERR_UNSUPPORTED;
    return false;
  }
  if (cfg->n_q_heads / cfg->n_kv_heads > SEKV_MAX_GROUP || cfg->rank_cap > SEKV_MAX_RANK) {
    *why = SEKV_ERR_UNSUPPORTED;
    return false;
  }
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace sekv

namespace sekv {

int device_sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// CTAs per (sequence, KV head) group of the decode kernel.  CTAs never wait
// for one another, so the grid may take several waves; cg is picked so that
// the last wave is as full as possible (1 to 4 waves of one CTA per SM, the
// fewest waves among the best fills), and large enough that every CTA's span
// share fits its shared-memory caches.
int decode_cg(const sekv_config* cfg, int sms) {
  const int ng = cfg->batch * cfg->n_kv_heads;
  int best = 1;
  double best_fill = -1.0;
  for (int waves = 1; waves <= 4; ++waves) {
    int cg = waves * sms / ng;
    if (cg < 1) cg = 1;
    const long long ctas = (long long)ng * cg;
    const long long slots = (ctas + sms - 1) / sms * sms;
    const double fill = double(ctas) / double(slots);
    if (fill > best_fill + 0.02) {
      best_fill = fill;
      best = cg;
    }
  }
  while (best < kMaxCg && cfg->max_spans / best + 8 > kSpanCap) ++best;
  return best > kMaxCg ? kMaxCg : best;
}

int route_chunks(const sekv_config* cfg) { return (cfg->max_spans + kRouteChunk - 1) / kRouteChunk; }

WsLayout ws_layout(const sekv_config* cfg, int sms) {
  WsLayout L{};
  L.ng = cfg->batch * cfg->n_kv_heads;
  L.cg = decode_cg(cfg, sms);
  L.route_chunks = route_chunks(cfg);
  const size_t ng = L.ng, ms = cfg->max_spans;
  size_t off = 0;
  L.status = off;     off += align256(64);
  L.groups = off;     off += align256(ng * sizeof(GroupState));
  L.cta_n = off;      off += align256(ng * L.cg * 4);
  L.cta_list = off;   off += align256(ng * ms * 4);
  L.partials = off;   off += align256(ng * L.cg * sizeof(Partial));
  L.route_list = off; off += align256(ng * ms * 4);
  L.route_cnt = off;  off += align256(ng * L.route_chunks * 4);
  L.plan = off;       off += align256(ng * ms * 3 * 8);
  L.plan_n = off;     off += align256(ng * 4);
  L.total = off;
  return L;
}

void count_launch(int n) { g_launches += n; }
void reset_launches() { g_launches = 0; }

}  // namespace sekv


namespace sekv {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

// Rows of `row_elems` elements as a 4-D tensor (half-row, row, half, group)
// so that one box of `box_rows` rows brings both 128-byte halves of each
// row: in shared memory the first halves of the box's rows come first, then
// the second halves, each 128B-swizzled by the row index.
bool encode_rows4d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                   uint64_t row_elems, uint64_t rows, uint64_t groups, int elem_bytes,
                   uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base) return false;
  const uint64_t half = row_elems / 2;
  const cuuint64_t dims[4] = {half, rows, 2, groups};
  const cuuint64_t strides[3] = {row_elems * elem_bytes, half * elem_bytes,
                                 rows * row_elems * elem_bytes};
  const cuuint32_t box[4] = {uint32_t(half), box_rows, 2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, dtype, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sekv

extern "C" {

int64_t sekv_record_size(int32_t body, int32_t rank_k, int32_t rank_v) {
  if (body <= 0 || rank_k < 0 || rank_v < 0) return 0;
  return record_bytes(body, rank_k, rank_v);
}

const char* sekv_status_string(sekv_status s) {
  switch (s) {
    case SEKV_OK: return "ok";
    case SEKV_ERR_INVALID: return "invalid argument";
    case SEKV_ERR_CAPACITY: return "buffer or workspace too small";
    case SEKV_ERR_CUDA: return "CUDA runtime error";
    case SEKV_ERR_TIMEOUT: return "bounded wait ran out";
    case SEKV_ERR_UNSUPPORTED: return "unsupported size";
    case SEKV_ERR_DEVICE: return "device reported bad data";
  }
  return "unknown status";
}

int32_t sekv_last_launch_count(void) { return g_launches; }

size_t sekv_workspace_size(const sekv_config* cfg, int32_t which, int64_t ctx_len) {
  sekv_status why;
  if (!config_ok(cfg, &why)) return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  if (which == SEKV_CALL_BUILD) return build_workspace_size(cfg, ctx_len);
  return ws_layout(cfg, sms).total;
}

sekv_status sekv_workspace_init(void* workspace, size_t bytes, cudaStream_t stream) {
  if (!workspace || bytes == 0) return SEKV_ERR_INVALID;
  return cudaMemsetAsync(workspace, 0, bytes, stream) == cudaSuccess ? SEKV_OK : SEKV_ERR_CUDA;
}

sekv_status sekv_workspace_status(void* workspace, cudaStream_t stream, int32_t* code,
                                  int32_t* detail) {
  if (!workspace) return SEKV_ERR_INVALID;
  int32_t h[2] = {0, 0};
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SEKV_ERR_CUDA;
  if (cudaMemcpy(h, workspace, 8, cudaMemcpyDeviceToHost) != cudaSuccess) return SEKV_ERR_CUDA;
  if (cudaMemset(workspace, 0, 8) != cudaSuccess) return SEKV_ERR_CUDA;
  if (code) *code = h[0];
  if (detail) *detail = h[1];
  if (h[0] == 0) return SEKV_OK;
  return h[0] == DEV_WAIT_TIMEOUT ? SEKV_ERR_TIMEOUT : SEKV_ERR_DEVICE;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// decode launches
// ----------------------------------------------------------------------------
namespace sekv {

sekv_status check_cache(const sekv_config* cfg, const sekv_layer_cache* c, bool need_store) {
  if (!c || !c->n_spans || !c->body_len || !c->k_full || !c->v_full || !c->k_sum || !c->v_sum ||
      !c->rec_off || !c->rec_rank)
    return SEKV_ERR_INVALID;
  if (need_store && !c->store) return SEKV_ERR_INVALID;
  if (!aligned16(c->k_full) || !aligned16(c->v_full) || !aligned16(c->k_sum) ||
      !aligned16(c->v_sum) || !aligned16(c->body_len) || !aligned16(c->rec_off) ||
      !aligned16(c->rec_rank) || (c->s_route && !aligned16(c->s_route)) ||
      (c->store && !aligned16(c->store)))
    return SEKV_ERR_INVALID;
  (void)cfg;
  return SEKV_OK;
}

sekv_status fill_decode_params(const sekv_config* cfg, const sekv_layer_cache* cache,
                               const WsLayout& L, void* ws, DecodeParams& P, bool fused) {
  const int ng = L.ng;
  const uint64_t cap_full = uint64_t(cfg->n_sink) + cfg->max_spans + cfg->n_recent;
  bool ok = true;
  ok &= encode_rows4d(&P.tm_kfull, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache->k_full, 128, cap_full, ng, 2, kFullRows);
  ok &= encode_rows4d(&P.tm_vfull, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache->v_full, 128, cap_full, ng, 2, kFullRows);
  ok &= encode_rows4d(&P.tm_ksum, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache->k_sum, 128, cfg->max_spans, ng, 2, kRows);
  ok &= encode_rows4d(&P.tm_vsum, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache->v_sum, 128, cfg->max_spans, ng, 2, kRows);
  if (fused) {
    ok &= encode_rows4d(&P.tm_sroute, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cache->s_route, 64, cfg->max_spans, ng, 4, kRouteSpans);
  } else {
    P.tm_sroute = P.tm_ksum;
  }
  if (!ok) return SEKV_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.n_spans = cache->n_spans;
  P.n_tail = cache->n_tail;
  P.body_len = cache->body_len;
  P.rec_off = cache->rec_off;
  P.rec_rank = cache->rec_rank;
  P.status = reinterpret_cast<int32_t*>(w + L.status);
  P.groups = reinterpret_cast<GroupState*>(w + L.groups);
  P.cta_n = reinterpret_cast<int32_t*>(w + L.cta_n);
  P.cta_list = reinterpret_cast<int32_t*>(w + L.cta_list);
  P.partials = reinterpret_cast<float*>(w + L.partials);
  P.B = cfg->batch;
  P.Hq = cfg->n_q_heads;
  P.Hkv = cfg->n_kv_heads;
  P.G = cfg->n_q_heads / cfg->n_kv_heads;
  P.nq = 1;
  P.nq_all = 1;
  P.hpg = P.G;
  P.n_sink = cfg->n_sink;
  P.n_recent = cfg->n_recent;
  P.max_spans = cfg->max_spans;
  P.cg = L.cg;
  P.fused = fused ? 1 : 0;
  P.wait_ns = (cfg->flags & SEKV_FLAG_SHORT_WAITS) ? 0ull : 2000000000ull;
  return SEKV_OK;
}

// Rank k-steps of 16 the kernel instance needs for this configuration.
int decode_ks(const sekv_config* cfg) {
  const int ks = (cfg->rank_cap + 15) / 16;
  return ks < 1 ? 1 : (ks > 4 ? 4 : ks);
}

sekv_status launch_decode(const DecodeParams& P0, const WsLayout& L, const sekv_config* cfg,
                          cudaStream_t stream, bool overlap) {
  static const void* const fns[8] = {
      decode_kernel_fn_ks1(false), decode_kernel_fn_ks2(false), decode_kernel_fn_ks3(false),
      decode_kernel_fn_ks4(false), decode_kernel_fn_ks1(true),  decode_kernel_fn_ks2(true),
      decode_kernel_fn_ks3(true),  decode_kernel_fn_ks4(true)};
  static std::once_flag once[8];
  static cudaError_t attr_err[8] = {};
  const int ks = decode_ks(cfg);
  const int fi = ks - 1 + (P0.nq_all > 1 ? 4 : 0);
  const void* fn = fns[fi];
  std::call_once(once[fi], [&] {
    attr_err[fi] = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  });
  if (attr_err[fi] != cudaSuccess) return SEKV_ERR_CUDA;
  DecodeParams P = P0;
  P.rank_lim = 16 * ks;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(L.cg, cfg->n_kv_heads, cfg->batch);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = kSmemAlloc;
  lc.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = overlap ? 1 : 0;
  void* args[] = {&P};
  if (cudaLaunchKernelExC(&lc, fn, args) != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(1);
  return SEKV_OK;
}

}  // namespace sekv

namespace {
// Query tokens per launch of the multi-query step: the columns of one
// launch are (token, head) pairs, at most 8.
int query_tokens_per_block(const sekv_config* cfg) {
  const int hpg = cfg->n_q_heads / cfg->n_kv_heads;
  return hpg >= 1 && hpg <= 8 ? 8 / hpg : 1;
}

sekv_status decode_step_impl(const sekv_config* cfg, const sekv_layer_cache* cache,
                             const void* q, int n_q, const float* W_r, const float* theta,
                             float scale, float* out, float* lse, int32_t* expanded,
                             int32_t* n_expanded, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  const int hpg = cfg->n_q_heads / cfg->n_kv_heads;
  if (n_q < 1 || n_q > SEKV_MAX_QUERY_TOKENS || hpg > 8) return SEKV_ERR_UNSUPPORTED;
  sekv_status st = check_cache(cfg, cache, true);
  if (st != SEKV_OK) return st;
  if (!q || !W_r || !theta || !out || !workspace || !cache->s_route) return SEKV_ERR_INVALID;
  if (cache->store_on_host) return SEKV_ERR_UNSUPPORTED;
  if (!aligned16(W_r) || !aligned16(q)) return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  const WsLayout L = ws_layout(cfg, sms);
  if (workspace_bytes < L.total) return SEKV_ERR_CAPACITY;
  DecodeParams P;
  memset(&P, 0, sizeof(P));
  st = fill_decode_params(cfg, cache, L, workspace, P, true);
  if (st != SEKV_OK) return st;
  P.store = static_cast<const uint8_t*>(cache->store);
  P.W_r = W_r;
  P.theta = theta;
  P.scale_log2 = scale * kLog2e;
  P.nq_all = n_q;
  // blocks of up to 8 / hpg tokens, one launch each (8 columns per launch);
  // in stream order, and each may overlap the previous one's tail
  const int tpb = query_tokens_per_block(cfg);
  const size_t row = size_t(cfg->n_q_heads) * kHeadDim;  // elements of one token's heads
  const size_t ng = size_t(cfg->batch) * cfg->n_kv_heads;
  for (int k = 0, q0 = 0; q0 < n_q; ++k, q0 += tpb) {
    P.nq = n_q - q0 < tpb ? n_q - q0 : tpb;
    P.G = P.nq * hpg;
    P.q = static_cast<const __nv_bfloat16*>(q) + q0 * row;
    P.out = out + q0 * row;
    P.lse = lse ? lse + size_t(q0) * cfg->n_q_heads : nullptr;
    P.expanded_out = expanded ? expanded + k * ng * cfg->max_spans : nullptr;
    P.n_expanded_out = n_expanded ? n_expanded + k * ng : nullptr;
    const bool overlap = k > 0 || (cfg->flags & SEKV_FLAG_OVERLAP_PREVIOUS) != 0;
    st = launch_decode(P, L, cfg, stream, overlap);
    if (st != SEKV_OK) return st;
  }
  return SEKV_OK;
}
}  // namespace

extern "C" sekv_status sekv_decode_step(const sekv_config* cfg, const sekv_layer_cache* cache,
                                        const void* q, const float* W_r, const float* theta,
                                        float scale, float* out, float* lse, int32_t* expanded,
                                        int32_t* n_expanded, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  return decode_step_impl(cfg, cache, q, 1, W_r, theta, scale, out, lse, expanded, n_expanded,
                          workspace, workspace_bytes, stream);
}

extern "C" int32_t sekv_query_blocks(const sekv_config* cfg, int32_t n_q) {
  if (!cfg || n_q < 1 || cfg->n_kv_heads < 1 || cfg->n_q_heads % cfg->n_kv_heads != 0) return 0;
  const int tpb = query_tokens_per_block(cfg);
  return (n_q + tpb - 1) / tpb;
}

extern "C" sekv_status sekv_decode_step_multi(const sekv_config* cfg,
                                              const sekv_layer_cache* cache, const void* q,
                                              int32_t n_q, const float* W_r, const float* theta,
                                              float scale, float* out, float* lse,
                                              int32_t* expanded, int32_t* n_expanded,
                                              void* workspace, size_t workspace_bytes,
                                              cudaStream_t stream) {
  return decode_step_impl(cfg, cache, q, n_q, W_r, theta, scale, out, lse, expanded, n_expanded,
                          workspace, workspace_bytes, stream);
}

extern "C" sekv_status sekv_decode_attention(const sekv_config* cfg,
                                             const sekv_layer_cache* cache, const void* q,
                                             const int32_t* expanded, const int32_t* n_expanded,
                                             const void* staging, const int64_t* staged_off,
                                             float scale, float* out, float* lse,
                                             void* workspace, size_t workspace_bytes,
                                             cudaStream_t stream) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  const bool staged = staging != nullptr;
  if (staged != (staged_off != nullptr)) return SEKV_ERR_INVALID;
  sekv_status st = check_cache(cfg, cache, !staged);
  if (st != SEKV_OK) return st;
  if (!staged && cache->store_on_host) return SEKV_ERR_UNSUPPORTED;
  if (!q || !expanded || !n_expanded || !out || !workspace) return SEKV_ERR_INVALID;
  if (!aligned16(q) || (staged && !aligned16(staging))) return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  const WsLayout L = ws_layout(cfg, sms);
  if (workspace_bytes < L.total) return SEKV_ERR_CAPACITY;
  DecodeParams P;
  memset(&P, 0, sizeof(P));
  st = fill_decode_params(cfg, cache, L, workspace, P, false);
  if (st != SEKV_OK) return st;
  P.store = static_cast<const uint8_t*>(staged ? staging : cache->store);
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.out = out;
  P.lse = lse;
  P.list = expanded;
  P.list_n = n_expanded;
  P.staged_off = staged_off;
  P.scale_log2 = scale * kLog2e;
  return launch_decode(P, L, cfg, stream, false);
}

extern "C" sekv_status sekv_route(const sekv_config* cfg, const sekv_layer_cache* cache,
                                  const void* q, const float* W_r, const float* theta,
                                  int32_t* expanded, int32_t* n_expanded, float* z_out,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  if (!cache || !cache->n_spans || !cache->body_len || !cache->s_route) return SEKV_ERR_INVALID;
  if (!q || !W_r || !theta || !expanded || !n_expanded || !workspace) return SEKV_ERR_INVALID;
  if (!aligned16(cache->s_route) || !aligned16(W_r)) return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  const WsLayout L = ws_layout(cfg, sms);
  if (workspace_bytes < L.total) return SEKV_ERR_CAPACITY;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  RouteParams P;
  P.n_spans = cache->n_spans;
  P.body_len = cache->body_len;
  P.s_route = cache->s_route;
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.W_r = W_r;
  P.theta = theta;
  P.expanded = expanded;
  P.n_expanded = n_expanded;
  P.z_out = z_out;
  P.status = reinterpret_cast<int32_t*>(w + L.status);
  P.groups = reinterpret_cast<GroupState*>(w + L.groups);
  P.list_scratch = reinterpret_cast<int32_t*>(w + L.route_list);
  P.cnt_scratch = reinterpret_cast<int32_t*>(w + L.route_cnt);
  P.B = cfg->batch;
  P.Hq = cfg->n_q_heads;
  P.Hkv = cfg->n_kv_heads;
  P.G = cfg->n_q_heads / cfg->n_kv_heads;
  P.max_spans = cfg->max_spans;
  P.chunks = L.route_chunks;
  route_kernel<<<dim3(L.route_chunks, cfg->n_kv_heads, cfg->batch), kRouteThreads, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(1);
  return SEKV_OK;
}

extern "C" sekv_status sekv_fetch_bases(const sekv_config* cfg, const sekv_layer_cache* cache,
                                        const int32_t* expanded, const int32_t* n_expanded,
                                        void* staging, int64_t staging_per_group,
                                        int64_t* staged_off, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  if (!cache || !cache->n_spans || !cache->body_len || !cache->rec_off || !cache->rec_rank ||
      !cache->store)
    return SEKV_ERR_INVALID;
  if (!expanded || !n_expanded || !staging || !staged_off || !workspace) return SEKV_ERR_INVALID;
  if (staging_per_group <= 0 || staging_per_group % 16 != 0 || !aligned16(staging) ||
      !aligned16(cache->store))
    return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  const WsLayout L = ws_layout(cfg, sms);
  if (workspace_bytes < L.total) return SEKV_ERR_CAPACITY;
  const void* dev_store = cache->store;
  if (cache->store_on_host) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, cache->store) != cudaSuccess ||
        pa.type != cudaMemoryTypeHost || pa.devicePointer == nullptr) {
      cudaGetLastError();
      return SEKV_ERR_INVALID;  // not page-locked host memory the device can address
    }
    dev_store = pa.devicePointer;
  }
  FetchParams P;
  P.n_spans = cache->n_spans;
  P.body_len = cache->body_len;
  P.rec_off = cache->rec_off;
  P.rec_rank = cache->rec_rank;
  P.store = static_cast<const uint8_t*>(dev_store);
  P.expanded = expanded;
  P.n_expanded = n_expanded;
  P.staging = static_cast<uint8_t*>(staging);
  P.per_group = staging_per_group;
  P.staged_off = staged_off;
  P.status = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + L.status);
  P.Hkv = cfg->n_kv_heads;
  P.max_spans = cfg->max_spans;
  fetch_kernel<<<dim3(L.ng, kFetchParts), 256, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(1);
  return SEKV_OK;
}



extern "C" sekv_status sekv_fetch_bases_copy(const sekv_config* cfg, const sekv_layer_cache* cache,
                                             const int32_t* expanded_host,
                                             const int32_t* n_expanded_host,
                                             const int64_t* rec_off_host, void* staging,
                                             int64_t staging_per_group, int64_t* staged_off_host,
                                             int64_t* staged_off, int32_t* n_copies,
                                             cudaStream_t copy_stream, cudaEvent_t done) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  if (!cache || !cache->store || !cache->store_on_host) return SEKV_ERR_INVALID;
  if (!expanded_host || !n_expanded_host || !rec_off_host || !staging || !staged_off_host ||
      !staged_off || !done)
    return SEKV_ERR_INVALID;
  if (staging_per_group <= 0 || staging_per_group % 16 != 0 || !aligned16(staging) ||
      !aligned16(cache->store))
    return SEKV_ERR_INVALID;
  const int ng = cfg->batch * cfg->n_kv_heads;
  const size_t ms = size_t(cfg->max_spans);
  const uint8_t* store = static_cast<const uint8_t*>(cache->store);
  // plan every copy before issuing any: offsets, sizes from the headers, checks
  int64_t copies = 0;
  for (int g = 0; g < ng; ++g) {
    const int ne = n_expanded_host[g];
    if (ne < 0 || ne > cfg->max_spans) return SEKV_ERR_INVALID;
    int64_t pos = 0;
    for (int e = 0; e < ne; ++e) {
      const int k = expanded_host[g * ms + e];
      if (k < 0 || k >= cfg->max_spans || (e > 0 && k <= expanded_host[g * ms + e - 1]))
        return SEKV_ERR_INVALID;
      const int64_t off = rec_off_host[g * ms + k];
      if (off < 0 || off % 16 != 0) return SEKV_ERR_INVALID;
      const int32_t* hdr = reinterpret_cast<const int32_t*>(store + off);
      const int64_t sz = sekv_record_size(hdr[0], hdr[1], hdr[2]);
      if (sz <= 0 || hdr[1] > SEKV_MAX_RANK || hdr[2] > SEKV_MAX_RANK) return SEKV_ERR_INVALID;
      staged_off_host[g * ms + e] = int64_t(g) * staging_per_group + pos;
      pos += sz;
    }
    if (pos > staging_per_group) return SEKV_ERR_CAPACITY;
  }
  // one copy per run of records that follow each other in the store and land
  // next to each other in staging
  uint8_t* stg = static_cast<uint8_t*>(staging);
  for (int g = 0; g < ng; ++g) {
    const int ne = n_expanded_host[g];
    int e = 0;
    while (e < ne) {
      const int64_t src0 = rec_off_host[g * ms + expanded_host[g * ms + e]];
      const int64_t dst0 = staged_off_host[g * ms + e];
      int64_t len = 0;
      int e1 = e;
      while (e1 < ne) {
        const int64_t off = rec_off_host[g * ms + expanded_host[g * ms + e1]];
        if (off != src0 + len) break;
        const int32_t* hdr = reinterpret_cast<const int32_t*>(store + off);
        len += sekv_record_size(hdr[0], hdr[1], hdr[2]);
        ++e1;
      }
      if (cudaMemcpyAsync(stg + dst0, store + src0, size_t(len), cudaMemcpyHostToDevice,
                          copy_stream) != cudaSuccess)
        return SEKV_ERR_CUDA;
      ++copies;
      e = e1;
    }
  }
  if (cudaMemcpyAsync(staged_off, staged_off_host, size_t(ng) * ms * sizeof(int64_t),
                      cudaMemcpyHostToDevice, copy_stream) != cudaSuccess)
    return SEKV_ERR_CUDA;
  if (cudaEventRecord(done, copy_stream) != cudaSuccess) return SEKV_ERR_CUDA;
  if (n_copies) *n_copies = int32_t(copies);
  return SEKV_OK;
}

// ----------------------------------------------------------------------------
// residency cache of basis records
// ----------------------------------------------------------------------------
namespace {

struct CacheTable {
  size_t slot_of, span_of, stamp, epoch, hand, total;
};

CacheTable cache_table(const sekv_config* cfg, int32_t n_slots) {
  CacheTable T{};
  const size_t ng = size_t(cfg->batch) * cfg->n_kv_heads, ms = cfg->max_spans;
  size_t off = 0;
  T.slot_of = off; off += align256(ng * ms * 4);
  T.span_of = off; off += align256(ng * size_t(n_slots) * 4);
  T.stamp = off;   off += align256(ng * size_t(n_slots) * 4);
  T.epoch = off;   off += align256(ng * 4);
  T.hand = off;    off += align256(ng * 4);
  T.total = off;
  return T;
}

}  // namespace

extern "C" size_t sekv_basis_cache_bytes(const sekv_config* cfg, int32_t n_slots) {
  sekv_status why;
  if (!config_ok(cfg, &why) || n_slots < 1 || n_slots > kCacheMaxSlots) return 0;
  return cache_table(cfg, n_slots).total;
}

extern "C" sekv_status sekv_basis_cache_init(const sekv_config* cfg, void* table,
                                             int32_t n_slots, cudaStream_t stream) {
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  if (!table || n_slots < 1 || n_slots > kCacheMaxSlots) return SEKV_ERR_INVALID;
  const CacheTable T = cache_table(cfg, n_slots);
  uint8_t* t = static_cast<uint8_t*>(table);
  // slot_of and span_of: -1 (empty); stamps, epochs and hands: 0
  if (cudaMemsetAsync(t, 0xff, T.stamp, stream) != cudaSuccess) return SEKV_ERR_CUDA;
  if (cudaMemsetAsync(t + T.stamp, 0, T.total - T.stamp, stream) != cudaSuccess)
    return SEKV_ERR_CUDA;
  return SEKV_OK;
}

extern "C" sekv_status sekv_fetch_bases_cached(const sekv_config* cfg,
                                               const sekv_layer_cache* cache,
                                               const int32_t* expanded, const int32_t* n_expanded,
                                               void* staging, int64_t staging_per_group,
                                               void* table, int32_t n_slots, int32_t slot_bytes,
                                               int64_t* staged_off, int32_t* hits,
                                               int64_t* copied, void* workspace,
                                               size_t workspace_bytes, cudaStream_t stream) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  if (!cache || !cache->n_spans || !cache->body_len || !cache->rec_off || !cache->rec_rank ||
      !cache->store || !cache->store_on_host)
    return SEKV_ERR_INVALID;
  if (!expanded || !n_expanded || !staging || !staged_off || !workspace || !table)
    return SEKV_ERR_INVALID;
  if (staging_per_group <= 0 || staging_per_group % 16 != 0 || !aligned16(staging) ||
      !aligned16(cache->store) || n_slots < 1 || n_slots > kCacheMaxSlots || slot_bytes < 16 ||
      slot_bytes % 16 != 0)
    return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  const WsLayout L = ws_layout(cfg, sms);
  if (workspace_bytes < L.total) return SEKV_ERR_CAPACITY;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, cache->store) != cudaSuccess ||
      pa.type != cudaMemoryTypeHost || pa.devicePointer == nullptr) {
    cudaGetLastError();
    return SEKV_ERR_INVALID;  // not page-locked host memory the device can address
  }
  const CacheTable T = cache_table(cfg, n_slots);
  uint8_t* t = static_cast<uint8_t*>(table);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  CacheParams P;
  P.n_spans = cache->n_spans;
  P.body_len = cache->body_len;
  P.rec_off = cache->rec_off;
  P.rec_rank = cache->rec_rank;
  P.store = static_cast<const uint8_t*>(pa.devicePointer);
  P.expanded = expanded;
  P.n_expanded = n_expanded;
  P.staging = static_cast<uint8_t*>(staging);
  P.per_group = staging_per_group;
  P.pool_base = int64_t(L.ng) * staging_per_group;
  P.slot_of = reinterpret_cast<int32_t*>(t + T.slot_of);
  P.span_of = reinterpret_cast<int32_t*>(t + T.span_of);
  P.stamp = reinterpret_cast<int32_t*>(t + T.stamp);
  P.epoch = reinterpret_cast<int32_t*>(t + T.epoch);
  P.hand = reinterpret_cast<int32_t*>(t + T.hand);
  P.plan = reinterpret_cast<int64_t*>(w + L.plan);
  P.plan_n = reinterpret_cast<int32_t*>(w + L.plan_n);
  P.staged_off = staged_off;
  P.hits = hits;
  P.copied = copied;
  P.status = reinterpret_cast<int32_t*>(w + L.status);
  P.Hkv = cfg->n_kv_heads;
  P.max_spans = cfg->max_spans;
  P.n_slots = n_slots;
  P.slot_bytes = slot_bytes;
  cache_plan_kernel<<<L.ng, 256, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  cache_copy_kernel<<<dim3(L.ng, kFetchParts), 256, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(2);
  return SEKV_OK;
}
