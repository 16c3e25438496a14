// Standalone zoom-in routing (sekv_route) and the host-tier basis fetch
// (sekv_fetch_bases).
//
// Routing: SeKV technical summary, Methodik 3 (gist.science, German page) /
// 方法论 3 (Chinese page): project the query into the summaries' routing
// space, gate every span with a sigmoid, expand where a per-head, per-layer
// threshold is exceeded.  Fetch: same section; expanded bases are loaded
// from the CPU tier on demand.
#include "route_fetch.cuh"

namespace sekv {



// grid (chunks, Hkv, B).  Each CTA scores spans [chunk*256, +256) of one
// (sequence, KV head); the last CTA of the pair concatenates the slices.
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteParams P) {
  __shared__ float qs[8][kHeadDim];
  __shared__ float ys[8][kRouteDim];
  __shared__ float th[8];
  __shared__ int wsum[kRouteThreads / 32];
  __shared__ int s_base, s_last;
  const int chunk = blockIdx.x, c = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int g = b * P.Hkv + c, G = P.G;
  const size_t gs = size_t(g) * P.max_spans;
  const int n_sp = P.n_spans[b];
  const int k0 = chunk * kRouteChunk;
  const __nv_bfloat16* qg = P.q + (size_t(b) * P.Hq + size_t(c) * G) * kHeadDim;
  for (int i = tid; i < 8 * kHeadDim; i += kRouteThreads)
    (&qs[0][0])[i] = (i / kHeadDim) < G ? __bfloat162float(qg[i]) : 0.f;
  if (tid < 8) th[tid] = tid < G ? P.theta[c * G + tid] : 0.f;
  if (tid == 0) s_base = 0;
  __syncthreads();
  {
    const int jr = tid & 63, hh = tid >> 6;  // heads hh, hh + 4
    const float4* wrow = reinterpret_cast<const float4*>(P.W_r + (size_t(c) * kRouteDim + jr) * kHeadDim);
    float a0 = 0.f, a1 = 0.f;
    for (int d4 = 0; d4 < 32; ++d4) {
      const float4 wv = __ldg(wrow + d4);
      const float4 q0 = reinterpret_cast<const float4*>(qs[hh])[d4];
      const float4 q1 = reinterpret_cast<const float4*>(qs[hh + 4])[d4];
      a0 = fmaf(wv.x, q0.x, fmaf(wv.y, q0.y, fmaf(wv.z, q0.z, fmaf(wv.w, q0.w, a0))));
      a1 = fmaf(wv.x, q1.x, fmaf(wv.y, q1.y, fmaf(wv.z, q1.z, fmaf(wv.w, q1.w, a1))));
    }
    ys[hh][jr] = a0;
    ys[hh + 4][jr] = a1;
  }
  __syncthreads();
  const int lane = tid & 31, wid = tid >> 5;
  for (int i = 0; i < kRouteChunk / kRouteThreads; ++i) {
    const int k = k0 + i * kRouteThreads + tid;
    bool ex = false;
    if (k < n_sp) {
      const float4* s4 = reinterpret_cast<const float4*>(P.s_route + (gs + k) * kRouteDim);
      float z[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) z[h] = 0.f;
#pragma unroll 4
      for (int dc = 0; dc < 16; ++dc) {
        const float4 s = __ldg(s4 + dc);
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float4 y = reinterpret_cast<const float4*>(ys[h])[dc];
          z[h] = fmaf(s.x, y.x, fmaf(s.y, y.y, fmaf(s.z, y.z, fmaf(s.w, y.w, z[h]))));
        }
      }
      const int body = P.body_len[size_t(b) * P.max_spans + k];
      bool hit = false;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < G) {
          hit |= z[h] > th[h];
          if (P.z_out) P.z_out[(size_t(b) * P.Hq + size_t(c) * G + h) * P.max_spans + k] = z[h];
        }
      }
      ex = hit && body > 0;
    }
    // ascending block compaction of this pass
    const uint32_t bal = __ballot_sync(0xffffffffu, ex);
    if (lane == 0) wsum[wid] = __popc(bal);
    __syncthreads();
    int base = s_base;
    for (int ww = 0; ww < wid; ++ww) base += wsum[ww];
    if (ex) P.list_scratch[gs + k0 + base + __popc(bal & ((1u << lane) - 1u))] = k;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
      for (int ww = 0; ww < kRouteThreads / 32; ++ww) t += wsum[ww];
      s_base += t;
    }
    __syncthreads();
  }
  if (tid == 0) P.cnt_scratch[size_t(g) * P.chunks + chunk] = s_base;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&P.groups[g].route_done, 1) == P.chunks - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // concatenate the chunks' slices: all counts in one round trip, prefix in
  // shared memory, then every entry copied in one flattened pass
  __shared__ int s_pre[kRouteMaxChunks + 1];
  for (int ch = tid; ch < P.chunks; ch += kRouteThreads)
    s_pre[ch + 1] = __ldcg(P.cnt_scratch + size_t(g) * P.chunks + ch);
  __syncthreads();
  if (tid == 0) {
    s_pre[0] = 0;
    for (int ch = 0; ch < P.chunks; ++ch) s_pre[ch + 1] += s_pre[ch];
  }
  __syncthreads();
  const int pre = s_pre[P.chunks];
  for (int e = tid; e < pre; e += kRouteThreads) {
    int lo = 0, hi = P.chunks;  // last chunk whose prefix is <= e
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] <= e) lo = mid; else hi = mid;
    }
    P.expanded[gs + e] = __ldcg(P.list_scratch + gs + size_t(lo) * kRouteChunk + (e - s_pre[lo]));
  }
  if (tid == 0) {
    P.n_expanded[g] = pre;
    P.groups[g].route_done = 0;
  }
}

// ----------------------------------------------------------------------------
// fetch: gather the expanded spans' records from host memory into staging
// ----------------------------------------------------------------------------


// grid (B*Hkv, kFetchParts): every part computes the group's offsets; part p
// copies list entries e with e % kFetchParts == p, one record per block pass.
__global__ void __launch_bounds__(256) fetch_kernel(const FetchParams P) {
  __shared__ long long incl[256];
  __shared__ int ks[256];
  __shared__ long long carry;
  const int g = blockIdx.x, part = blockIdx.y, tid = threadIdx.x, b = g / P.Hkv;
  const size_t gs = size_t(g) * P.max_spans;
  const int n_sp = P.n_spans[b];
  int ne = P.n_expanded[g];
  if (ne < 0 || ne > n_sp) ne = 0;
  for (int pass = 0; pass < 2; ++pass) {
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int e0 = 0; e0 < ne; e0 += 256) {
      const int e = e0 + tid;
      long long size = 0;
      int k = -1;
      if (e < ne) {
        k = P.expanded[gs + e];
        if (k >= 0 && k < n_sp) {
          const int rank = P.rec_rank[gs + k];
          size = record_bytes(P.body_len[size_t(b) * P.max_spans + k], rank & 0xffff,
                              (rank >> 16) & 0xffff);
        } else {
          k = -1;
        }
      }
      ks[tid] = k;
      incl[tid] = size;
      __syncthreads();
      for (int o = 1; o < 256; o <<= 1) {
        const long long v = tid >= o ? incl[tid - o] : 0;
        __syncthreads();
        incl[tid] += v;
        __syncthreads();
      }
      if (pass == 1) {
        if (e < ne && part == 0) P.staged_off[gs + e] = int64_t(g) * P.per_group + carry + incl[tid] - size;
        for (int t = 0; t < 256 && e0 + t < ne; ++t) {
          if (((e0 + t) % kFetchParts) != part || ks[t] < 0) continue;
          const long long sz = incl[t] - (t ? incl[t - 1] : 0);
          const long long st = carry + incl[t] - sz;
          const int4* src = reinterpret_cast<const int4*>(P.store + P.rec_off[gs + ks[t]]);
          int4* dst = reinterpret_cast<int4*>(P.staging + int64_t(g) * P.per_group + st);
          // eight 16-byte loads in flight per thread: the host link's latency
          // is hidden by concurrency, not by one load at a time
          const long long n16 = sz / 16;
          for (long long i0 = 0; i0 < n16; i0 += 256 * kFetchUnroll) {
            int4 v[kFetchUnroll];
#pragma unroll
            for (int u = 0; u < kFetchUnroll; ++u) {
              const long long i = i0 + tid + 256 * u;
              if (i < n16) v[u] = __ldcs(src + i);
            }
#pragma unroll
            for (int u = 0; u < kFetchUnroll; ++u) {
              const long long i = i0 + tid + 256 * u;
              if (i < n16) dst[i] = v[u];
            }
          }
        }
      }
      __syncthreads();
      if (tid == 0) carry += incl[255];
      __syncthreads();
    }
    if (pass == 0 && carry > P.per_group) {
      if (part == 0 && tid == 0) set_device_error(P.status, DEV_STAGING_FULL, g);
      return;
    }
  }
}

}  // namespace sekv
