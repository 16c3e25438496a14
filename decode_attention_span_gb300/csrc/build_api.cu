// C-ABI entry point of the prefill cache build (sekv_build_spans).
#include <mutex>

#include "build.cuh"
#include "host_common.h"

using namespace sekv;

namespace {

struct BuildWs {
  size_t status, starts, rel_off, gtotal, gbase, counters, cls_list, total;
  int64_t cls_cap;
};

BuildWs build_ws(const sekv_config* cfg) {
  BuildWs L{};
  const size_t B = cfg->batch, ng = size_t(cfg->batch) * cfg->n_kv_heads, ms = cfg->max_spans;
  L.cls_cap = int64_t(ng * ms * 2);
  size_t off = 0;
  L.status = off;   off += align256(64);
  L.starts = off;   off += align256(B * ms * 4);
  L.rel_off = off;  off += align256(ng * ms * 8);
  L.gtotal = off;   off += align256(ng * 8);
  L.gbase = off;    off += align256(ng * 8);
  L.counters = off; off += align256(16 * 4);
  L.cls_list = off; off += align256(size_t(kSvdClasses) * L.cls_cap * 4);
  L.total = off;
  return L;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

namespace sekv {
size_t build_workspace_size(const sekv_config* cfg, int64_t ctx_len) {
  (void)ctx_len;
  return build_ws(cfg).total;
}
}  // namespace sekv

extern "C" sekv_status sekv_build_spans(const sekv_config* cfg, int64_t ctx_len, const void* K,
                                        const void* V, const float* H, const float* W_r,
                                        const float* gates, const sekv_cache_out* out,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
  reset_launches();
  if (!cfg) return SEKV_ERR_INVALID;
  if (cfg->head_dim != 128 || cfg->route_dim != 64) return SEKV_ERR_UNSUPPORTED;
  if (cfg->rank_cap < 0 || cfg->rank_cap > SEKV_MAX_RANK) return SEKV_ERR_UNSUPPORTED;
  if (cfg->batch < 1 || cfg->n_kv_heads < 1 || cfg->max_spans < 64 || cfg->max_spans % 64 ||
      cfg->n_sink < 0 || cfg->n_recent < 0 || cfg->len_min < 1 || cfg->len_max < cfg->len_min ||
      cfg->len_max > 32767 || ctx_len < int64_t(cfg->n_sink) + cfg->n_recent ||
      ctx_len > (int64_t(1) << 26))
    return SEKV_ERR_INVALID;
  if (!K || !V || !H || !W_r || !gates || !out || !workspace) return SEKV_ERR_INVALID;
  if (!out->n_spans || !out->body_len || !out->k_full || !out->v_full || !out->s_route ||
      !out->k_sum || !out->v_sum || !out->rec_off || !out->rec_rank || !out->store ||
      out->store_capacity <= 0)
    return SEKV_ERR_INVALID;
  if (!al16(K) || !al16(V) || !al16(W_r) || !al16(out->k_full) || !al16(out->v_full) ||
      !al16(out->k_sum) || !al16(out->v_sum) || !al16(out->store) || !al16(out->s_route) ||
      (reinterpret_cast<uintptr_t>(H) & 3) || (reinterpret_cast<uintptr_t>(gates) & 3))
    return SEKV_ERR_INVALID;
  const BuildWs L = build_ws(cfg);
  if (workspace_bytes < L.total) return SEKV_ERR_CAPACITY;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  BuildParams P;
  P.K = static_cast<const __nv_bfloat16*>(K);
  P.V = static_cast<const __nv_bfloat16*>(V);
  P.H = H;
  P.W_r = W_r;
  P.gates = gates;
  P.n_spans = out->n_spans;
  P.body_len = out->body_len;
  P.k_full = static_cast<__nv_bfloat16*>(out->k_full);
  P.v_full = static_cast<__nv_bfloat16*>(out->v_full);
  P.s_route = out->s_route;
  P.k_sum = static_cast<__nv_bfloat16*>(out->k_sum);
  P.v_sum = static_cast<__nv_bfloat16*>(out->v_sum);
  P.rec_off = out->rec_off;
  P.rec_rank = out->rec_rank;
  P.store = static_cast<uint8_t*>(out->store);
  P.store_capacity = out->store_capacity;
  P.status = reinterpret_cast<int32_t*>(w + L.status);
  P.flops = reinterpret_cast<unsigned long long*>(w + L.status + 16);
  P.starts = reinterpret_cast<int32_t*>(w + L.starts);
  P.rel_off = reinterpret_cast<int64_t*>(w + L.rel_off);
  P.gtotal = reinterpret_cast<int64_t*>(w + L.gtotal);
  P.gbase = reinterpret_cast<int64_t*>(w + L.gbase);
  P.counters = reinterpret_cast<int32_t*>(w + L.counters);
  P.cls_list = reinterpret_cast<int32_t*>(w + L.cls_list);
  P.cls_cap = L.cls_cap;
  P.only_k = nullptr;
  P.only_n = nullptr;
  P.B = cfg->batch;
  P.Hkv = cfg->n_kv_heads;
  P.T = int(ctx_len);
  P.n_sink = cfg->n_sink;
  P.n_recent = cfg->n_recent;
  P.max_spans = cfg->max_spans;
  P.rank_cap = cfg->rank_cap;
  P.len_min = cfg->len_min;
  P.len_max = cfg->len_max;
  P.tau = cfg->tau;
  const int ng = cfg->batch * cfg->n_kv_heads;
  const int64_t n_mid = ctx_len - cfg->n_sink - cfg->n_recent;
  const int seg_smem = int(((n_mid + 31) / 32) * 4);
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                220 * 1024);
  });
  if (attr != cudaSuccess) return SEKV_ERR_CUDA;
  if (seg_smem > 220 * 1024) return SEKV_ERR_UNSUPPORTED;
  seg_kernel<<<cfg->batch, 1024, seg_smem, stream>>>(P);
  plan_kernel<<<ng, 256, 0, stream>>>(P);
  gather_kernel<<<dim3(ng, 32), 256, 0, stream>>>(P);
  summary_kernel<<<dim3(cfg->max_spans / 8, ng), 256, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  if (launch_svd_all(P, sms, stream) != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(8);
  return SEKV_OK;
}

extern "C" sekv_status sekv_build_flops(void* workspace, cudaStream_t stream, int64_t* flops) {
  if (!workspace || !flops) return SEKV_ERR_INVALID;
  unsigned long long v = 0;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SEKV_ERR_CUDA;
  if (cudaMemcpy(&v, w + 16, 8, cudaMemcpyDeviceToHost) != cudaSuccess) return SEKV_ERR_CUDA;
  if (cudaMemset(w + 16, 0, 8) != cudaSuccess) return SEKV_ERR_CUDA;
  *flops = int64_t(v);
  return SEKV_OK;
}

// ----------------------------------------------------------------------------
// decode-time maintenance (sekv_maint_init, sekv_append_token)
// ----------------------------------------------------------------------------
namespace {

struct MaintState {
  size_t seq_len, s_open, n_pend, pend_rows, pend_len, store_used, pend, only_k, only_n, tail_h,
      total;
};

int64_t full_cap(const sekv_config* cfg) {
  return int64_t(cfg->n_sink) + cfg->max_spans + cfg->n_recent;
}

MaintState maint_state(const sekv_config* cfg) {
  MaintState S{};
  const size_t B = cfg->batch;
  size_t off = 0;
  S.seq_len = off;    off += align256(B * 4);
  S.s_open = off;     off += align256(B * 4);
  S.n_pend = off;     off += align256(B * 4);
  S.pend_rows = off;  off += align256(B * 4);
  S.pend_len = off;   off += align256(B * kMaxPending * 4);
  S.store_used = off; off += align256(8);
  S.pend = off;       off += align256(B * 32);
  S.only_k = off;     off += align256(B * 4);
  S.only_n = off;     off += align256(B * 4);
  S.tail_h = off;     off += align256(B * size_t(full_cap(cfg)) * 4);
  S.total = off;
  return S;
}

bool maint_args_ok(const sekv_config* cfg, int64_t ctx_len, const sekv_cache_out* out,
                   const int32_t* n_tail, const void* state, size_t state_bytes,
                   const void* workspace, size_t workspace_bytes) {
  if (!cfg || cfg->head_dim != 128 || cfg->route_dim != 64) return false;
  if (cfg->batch < 1 || cfg->n_kv_heads < 1 || cfg->max_spans < 64 || cfg->max_spans % 64 ||
      cfg->n_sink < 0 || cfg->n_recent < 1 || cfg->len_min < 1 || cfg->len_max < cfg->len_min ||
      cfg->rank_cap < 0 || cfg->rank_cap > SEKV_MAX_RANK ||
      ctx_len < int64_t(cfg->n_sink) + cfg->n_recent || ctx_len > (int64_t(1) << 30))
    return false;
  if (!out || !out->n_spans || !out->body_len || !out->k_full || !out->v_full ||
      !out->s_route || !out->k_sum || !out->v_sum || !out->rec_off || !out->rec_rank ||
      !out->store || out->store_capacity <= 0 || !n_tail || !state || !workspace)
    return false;
  if (!al16(out->k_full) || !al16(out->v_full) || !al16(out->store)) return false;
  if (state_bytes < maint_state(cfg).total) return false;
  if (workspace_bytes < build_ws(cfg).total) return false;
  return true;
}

MaintParams maint_params(const sekv_config* cfg, int64_t ctx_len, const sekv_cache_out* out,
                         int32_t* n_tail, void* state, void* workspace) {
  const MaintState S = maint_state(cfg);
  const BuildWs L = build_ws(cfg);
  uint8_t* st = static_cast<uint8_t*>(state);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  MaintParams M{};
  M.n_spans = out->n_spans;
  M.n_tail = n_tail;
  M.body_len = out->body_len;
  M.k_full = static_cast<__nv_bfloat16*>(out->k_full);
  M.v_full = static_cast<__nv_bfloat16*>(out->v_full);
  M.s_route = out->s_route;
  M.k_sum = static_cast<__nv_bfloat16*>(out->k_sum);
  M.v_sum = static_cast<__nv_bfloat16*>(out->v_sum);
  M.rec_off = out->rec_off;
  M.rec_rank = out->rec_rank;
  M.store_capacity = out->store_capacity;
  M.seq_len = reinterpret_cast<int32_t*>(st + S.seq_len);
  M.s_open = reinterpret_cast<int32_t*>(st + S.s_open);
  M.n_pend = reinterpret_cast<int32_t*>(st + S.n_pend);
  M.pend_rows = reinterpret_cast<int32_t*>(st + S.pend_rows);
  M.pend_len = reinterpret_cast<int32_t*>(st + S.pend_len);
  M.only_n = reinterpret_cast<int32_t*>(st + S.only_n);
  M.store_used = reinterpret_cast<unsigned long long*>(st + S.store_used);
  M.pend = reinterpret_cast<int32_t*>(st + S.pend);
  M.only_k = reinterpret_cast<int32_t*>(st + S.only_k);
  M.tail_h = reinterpret_cast<float*>(st + S.tail_h);
  M.status = reinterpret_cast<int32_t*>(w + L.status);
  M.starts = reinterpret_cast<int32_t*>(w + L.starts);
  M.rel_off = reinterpret_cast<int64_t*>(w + L.rel_off);
  M.gbase = reinterpret_cast<int64_t*>(w + L.gbase);
  M.counters = reinterpret_cast<int32_t*>(w + L.counters);
  M.cls_list = reinterpret_cast<int32_t*>(w + L.cls_list);
  M.cls_cap = L.cls_cap;
  M.B = cfg->batch;
  M.Hkv = cfg->n_kv_heads;
  M.T = int(ctx_len);
  M.cap = int(full_cap(cfg));
  M.n_sink = cfg->n_sink;
  M.n_recent = cfg->n_recent;
  M.max_spans = cfg->max_spans;
  M.rank_cap = cfg->rank_cap;
  M.len_min = cfg->len_min;
  M.len_max = cfg->len_max;
  M.tau = cfg->tau;
  return M;
}

}  // namespace

extern "C" size_t sekv_maint_state_size(const sekv_config* cfg) {
  if (!cfg || cfg->batch < 1 || cfg->max_spans < 1) return 0;
  return maint_state(cfg).total;
}

extern "C" sekv_status sekv_maint_init(const sekv_config* cfg, int64_t ctx_len, const void* K,
                                       const void* V, const float* H,
                                       const sekv_cache_out* out, int32_t* n_tail, void* state,
                                       size_t state_bytes, void* workspace,
                                       size_t workspace_bytes, cudaStream_t stream) {
  reset_launches();
  if (!maint_args_ok(cfg, ctx_len, out, n_tail, state, state_bytes, workspace, workspace_bytes))
    return SEKV_ERR_INVALID;
  if (!K || !V || !H || !al16(K) || !al16(V)) return SEKV_ERR_INVALID;
  MaintParams M = maint_params(cfg, ctx_len, out, n_tail, state, workspace);
  if (cudaMemsetAsync(state, 0, maint_state(cfg).total, stream) != cudaSuccess) return SEKV_ERR_CUDA;
  const int ng = cfg->batch * cfg->n_kv_heads;
  maint_used_kernel<<<ng, 256, 0, stream>>>(M);
  maint_init_rows_kernel<<<dim3(cfg->n_kv_heads, cfg->batch), 256, 0, stream>>>(
      M, static_cast<const __nv_bfloat16*>(K), static_cast<const __nv_bfloat16*>(V), H);
  maint_init_commit_kernel<<<cfg->batch, 32, 0, stream>>>(M);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(3);
  return SEKV_OK;
}

extern "C" sekv_status sekv_append_token(const sekv_config* cfg, const void* k_new,
                                         const void* v_new, const float* h_new,
                                         const sekv_cache_out* out, int32_t* n_tail, void* state,
                                         size_t state_bytes, void* workspace,
                                         size_t workspace_bytes, cudaStream_t stream) {
  reset_launches();
  const int64_t ctx_len = int64_t(cfg ? cfg->n_sink : 0) + (cfg ? cfg->n_recent : 0);  // checks only
  if (!maint_args_ok(cfg, ctx_len, out, n_tail, state, state_bytes, workspace, workspace_bytes))
    return SEKV_ERR_INVALID;
  if (!k_new || !v_new || !h_new || !al16(k_new) || !al16(v_new)) return SEKV_ERR_INVALID;
  MaintParams M = maint_params(cfg, ctx_len, out, n_tail, state, workspace);
  M.k_new = static_cast<const __nv_bfloat16*>(k_new);
  M.v_new = static_cast<const __nv_bfloat16*>(v_new);
  M.h_new = h_new;
  maint_append_kernel<<<cfg->batch, 256, 0, stream>>>(M);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(1);
  return SEKV_OK;
}

extern "C" sekv_status sekv_maint_flush(const sekv_config* cfg, const float* W_r,
                                        const float* gates, const sekv_cache_out* out,
                                        int32_t* n_tail, void* state, size_t state_bytes,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
  reset_launches();
  const int64_t ctx_len = int64_t(cfg ? cfg->n_sink : 0) + (cfg ? cfg->n_recent : 0);  // checks only
  if (!maint_args_ok(cfg, ctx_len, out, n_tail, state, state_bytes, workspace, workspace_bytes))
    return SEKV_ERR_INVALID;
  if (!W_r || !gates || !al16(W_r) || (reinterpret_cast<uintptr_t>(gates) & 3))
    return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  MaintParams M = maint_params(cfg, ctx_len, out, n_tail, state, workspace);
  M.gates = gates;
  const BuildWs L = build_ws(cfg);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if (cudaMemsetAsync(w + L.counters, 0, 16 * 4, stream) != cudaSuccess) return SEKV_ERR_CUDA;
  const dim3 grid(cfg->n_kv_heads, cfg->batch);
  maint_flush_plan_kernel<<<grid, kMaxPending, 0, stream>>>(M);
  // the waiting spans' summaries and bases: the build's kernels, in place on
  // the full rows (K = the rows of each group, T = their capacity, H = the
  // surprisal by row)
  BuildParams P{};
  P.K = M.k_full;
  P.V = M.v_full;
  P.H = M.tail_h;
  P.W_r = W_r;
  P.gates = gates;
  P.n_spans = M.n_spans;
  P.body_len = M.body_len;
  P.k_full = M.k_full;
  P.v_full = M.v_full;
  P.s_route = M.s_route;
  P.k_sum = M.k_sum;
  P.v_sum = M.v_sum;
  P.rec_off = M.rec_off;
  P.rec_rank = M.rec_rank;
  P.store = static_cast<uint8_t*>(out->store);
  P.store_capacity = out->store_capacity;
  P.status = M.status;
  P.flops = reinterpret_cast<unsigned long long*>(w + L.status + 16);
  P.starts = M.starts;
  P.rel_off = M.rel_off;
  P.gtotal = reinterpret_cast<int64_t*>(w + L.gtotal);
  P.gbase = M.gbase;
  P.counters = M.counters;
  P.cls_list = M.cls_list;
  P.cls_cap = M.cls_cap;
  P.only_k = M.only_k;
  P.only_n = M.only_n;
  P.B = M.B;
  P.Hkv = M.Hkv;
  P.T = M.cap;
  P.n_sink = M.n_sink;
  P.n_recent = M.n_recent;
  P.max_spans = M.max_spans;
  P.rank_cap = M.rank_cap;
  P.len_min = M.len_min;
  P.len_max = M.len_max;
  P.tau = M.tau;
  summary_kernel<<<dim3(kMaxPending / 8, cfg->batch * cfg->n_kv_heads), 256, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  if (launch_svd_all(P, sms, stream) != cudaSuccess) return SEKV_ERR_CUDA;
  maint_flush_move_kernel<<<grid, 256, 0, stream>>>(M);
  maint_flush_commit_kernel<<<cfg->batch, 32, 0, stream>>>(M);
  if (cudaGetLastError() != cudaSuccess) return SEKV_ERR_CUDA;
  count_launch(9);
  return SEKV_OK;
}
