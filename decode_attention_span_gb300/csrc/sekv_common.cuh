// Shared device helpers for libsekv (sm_103a): inline PTX for mbarriers,
// bulk and tensor TMA copies, ldmatrix, mma.sync and programmatic dependent
// launch, plus the workspace layout that host and device code agree on.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sekv.h"

namespace sekv {

constexpr int kHeadDim = 128;
constexpr int kRouteDim = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// device status codes (first error wins); detail carries an index or a count
enum DeviceError : int32_t {
  DEV_OK = 0,
  DEV_BAD_LIST = 1,        // expansion list not ascending / out of range / empty body
  DEV_WAIT_TIMEOUT = 2,    // a bounded spin ran out
  DEV_STAGING_FULL = 3,    // fetch: a group's records exceed its staging share
  DEV_BAD_RANK = 4,        // a record rank above the supported maximum
};

// ----------------------------------------------------------------------------
// workspace layout (bytes, all offsets 256-aligned)
// ----------------------------------------------------------------------------
struct GroupState {        // one per (sequence, KV head); zero between calls
  int32_t done;            // decode: CTAs that have written their partial
  int32_t route_done;      // route kernel: chunks finished
  int32_t full_next;       // decode: full-resolution pages taken from the group's pool
  int32_t pad;
};

struct Partial {           // one CTA's softmax state for up to 8 heads
  float m[8];              // running max (log2 domain)
  float l[8];              // sum of 2^(x - m)
  float o[8][kHeadDim];    // sum of 2^(x - m) * value
};

struct WsLayout {
  size_t status, groups, cta_n, cta_list, partials, route_list, route_cnt, plan, plan_n, total;
  int ng, cg, route_chunks;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking probe of a phase (test_wait never suspends the thread, so a
// bounded loop of probes has a known duration).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Four independent phase tests in one go (their latencies overlap); bit i of
// the result is set iff barrier i has completed the phase of parity q_i.
__device__ __forceinline__ uint32_t mbar_test4(uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t q0, uint32_t q1, uint32_t q2,
                                               uint32_t q3) {
  uint32_t m;
  asm volatile(
      "{\n .reg .pred p0, p1, p2, p3;\n .reg .b32 t0, t1, t2, t3;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p0, [%1], %5;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p1, [%2], %6;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p2, [%3], %7;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p3, [%4], %8;\n"
      " selp.b32 t0, 1, 0, p0;\n selp.b32 t1, 2, 0, p1;\n"
      " selp.b32 t2, 4, 0, p2;\n selp.b32 t3, 8, 0, p3;\n"
      " or.b32 t0, t0, t1;\n or.b32 t2, t2, t3;\n or.b32 %0, t0, t2;\n}\n"
      : "=r"(m)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(q0), "r"(q1), "r"(q2), "r"(q3)
      : "memory");
  return m;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One phase test that may suspend the warp until the phase completes or
// about hint_ns nanoseconds pass, whichever is first.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait in which the hardware parks the warp instead of a polling loop
// (no shared-memory traffic while it waits); returns false once `limit_ns`
// nanoseconds have passed without the phase completing (the caller flags an
// error).  limit_ns == 0 gives up at once if the phase is not complete at the
// first test.
__device__ __forceinline__ bool mbar_wait_parked(uint64_t* bar, uint32_t parity,
                                                 uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  if (limit_ns == 0) return false;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity, 20000u)) return true;
    if ((i & 15u) == 15u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait: returns false after `limit` polls (the caller flags an error).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's view of global memory (including other CTAs' writes
// it has acquired) before its later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// L2 policy for data read exactly once: evicted first, so that it does not
// push out what is reused (code, routing weights, counters).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for data many CTAs read (the routing weights of a KV head).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 4-D tiled tensor copy global -> shared with an L2 cache hint.
__device__ __forceinline__ void tma_g2s_4d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                int z, int w, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
      "l"(pol)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Read-only 16-byte load issued where it stands: a volatile asm keeps the
// compiler from sinking it to the value's first use, so its round trip
// overlaps the work in between.
__device__ __forceinline__ float4 ldg_nc_early(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void set_device_error(int32_t* status, int32_t code, int32_t detail) {
  if (atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// byte address inside a 128B-swizzled box of 128-byte rows
__device__ __forceinline__ uint32_t swz128(uint32_t base, int row, int chunk16) {
  return base + row * 128 + ((chunk16 ^ (row & 7)) << 4);
}

__host__ __device__ inline int r4(int r) { return (r + 3) & ~3; }
__host__ __device__ inline int r8(int r) { return (r + 7) & ~7; }

// U rows of a basis record hold W = r8(r) / 8 sixteen-byte chunks; chunk c of
// token row t is stored at chunk position c ^ u_swz(t, W).  With g the largest
// power of two dividing W, rows t and t + 8/g start in the same bank group;
// the XOR with bits of t above log2(8/g) (below g) moves them apart, so the 8
// rows an ldmatrix reads hit 8 different bank groups.  It stays below W and
// depends on t mod 8 only.
__host__ __device__ inline int u_swz(int t, int W) {
  const int g = W & -W;
  const int s = 3 - ((g > 1) + (g > 2) + (g > 4));
  return (t >> s) & (g - 1);
}
// element offset of column j of row t in a U block with row stride rs = r8(r)
__host__ __device__ inline int u_col(int t, int j, int rs) {
  return (((j >> 3) ^ u_swz(t, rs >> 3)) << 3) | (j & 7);
}
__host__ __device__ inline int64_t pad16(int64_t n) { return (n + 15) & ~int64_t(15); }

// Basis record layout (see sekv.h): byte offsets of its parts.
struct RecordLayout {
  int64_t uk, uv, vpart, total;
};
__host__ __device__ inline RecordLayout record_layout(int b, int rK, int rV) {
  RecordLayout L;
  L.uk = 16 + 8 * r4(rK) + 256 * int64_t(rK);
  L.uv = L.uk + 2 * int64_t(b) * r8(rK);
  L.vpart = L.uv + 2 * int64_t(b) * r8(rV);
  L.total = L.vpart + 8 * r4(rV) + 256 * int64_t(rV);
  return L;
}

__host__ __device__ inline int64_t record_bytes(int b, int rK, int rV) {
  if (b <= 0) return 0;
  return record_layout(b, rK, rV).total;
}

}  // namespace sekv
