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
