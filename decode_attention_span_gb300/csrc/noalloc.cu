// sekv_decode_step_noalloc: the fused decode step without a caller
// workspace.  Its scratch (counters, expansion entries, per-CTA partial
// softmax states) lives in one statically sized device array owned by this
// library, so the call allocates nothing at any point.
#include <string.h>

#include <mutex>

#include "decode_host.h"
#include "host_common.h"

namespace {

constexpr size_t kNoAllocScratchBytes = SEKV_NOALLOC_SCRATCH_BYTES;

// Every GPU that loads libsekv holds this array until the process exits.
// Host code must not pass the symbol itself to a kernel: on the host it is
// only a stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

std::mutex g_mu;
void* g_scratch_ptr[64] = {};
CUcontext g_scratch_ctx[64] = {};

// Device address of the scratch array on the current device.  It is looked
// up with the device current and cached per device together with the
// context it was found in: after a device reset (a new primary context, the
// module loaded again) the next call looks it up afresh instead of handing a
// stale address to the kernel.
sekv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SEKV_ERR_CUDA;
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (get_ctx == nullptr) return SEKV_ERR_CUDA;
  CUcontext ctx = nullptr;  // null until the runtime has made the primary context current
  if (get_ctx(&ctx) != CUDA_SUCCESS) return SEKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SEKV_ERR_CUDA;
    }
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SEKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return SEKV_OK;
}

}  // namespace

using namespace sekv;

extern "C" sekv_status sekv_decode_step_noalloc(const sekv_config* cfg,
                                                const sekv_layer_cache* cache, const void* q,
                                                const float* W_r, const float* theta,
                                                float scale, float* out, float* lse,
                                                int32_t* expanded, int32_t* n_expanded,
                                                cudaStream_t stream) {
  reset_launches();
  sekv_status why;
  if (!config_ok(cfg, &why)) return why;
  sekv_status st = check_cache(cfg, cache, true);
  if (st != SEKV_OK) return st;
  if (!q || !W_r || !theta || !out || !cache->s_route) return SEKV_ERR_INVALID;
  if (cache->store_on_host) return SEKV_ERR_UNSUPPORTED;
  if (!aligned16(W_r) || !aligned16(q)) return SEKV_ERR_INVALID;
  const int sms = device_sm_count();
  if (sms <= 0) return SEKV_ERR_CUDA;
  const WsLayout L = ws_layout(cfg, sms);
  if (L.total > kNoAllocScratchBytes) return SEKV_ERR_CAPACITY;  // shape too large for the array
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != SEKV_OK) return st;
  // The array keeps whatever the previous call left: the status word and the
  // per-(sequence, KV head) counters must start at zero.
  if (cudaMemsetAsync(scratch, 0, L.cta_n, stream) != cudaSuccess) return SEKV_ERR_CUDA;
  DecodeParams P;
  memset(&P, 0, sizeof(P));
  st = fill_decode_params(cfg, cache, L, scratch, P, true);
  if (st != SEKV_OK) return st;
  P.store = static_cast<const uint8_t*>(cache->store);
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.W_r = W_r;
  P.theta = theta;
  P.out = out;
  P.lse = lse;
  P.expanded_out = expanded;
  P.n_expanded_out = n_expanded;
  P.scale_log2 = scale * kLog2e;
  return launch_decode(P, L, cfg, stream, false);
}

extern "C" sekv_status sekv_noalloc_status(cudaStream_t stream, int32_t* code, int32_t* detail) {
  void* scratch = nullptr;
  sekv_status st = scratch_address(&scratch);
  if (st != SEKV_OK) return st;
  // the status word is the first 8 bytes of the array (as of a workspace)
  return sekv_workspace_status(scratch, stream, code, detail);
}
