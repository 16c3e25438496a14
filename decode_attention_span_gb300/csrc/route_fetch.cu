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
  const int lane = tid & 31, wid = tid >> 5;
  {
    // y = W_r q: warp w takes rows 8w .. 8w + 7; lane (r, dq) = (lane / 4,
    // lane % 4) loads 16-byte chunks dq + 4 i (i < 8) of row 8w + r, all
    // eight at once, multiplies them with the same chunks of every head's
    // query and sums over dq by shuffles
    const int r = lane >> 2, dq = lane & 3;
    const float4* wrow =
        reinterpret_cast<const float4*>(P.W_r + (size_t(c) * kRouteDim + 8 * wid + r) * kHeadDim);
    float4 wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[i] = __ldg(wrow + dq + 4 * i);
    float acc[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float4 qv = reinterpret_cast<const float4*>(qs[h])[dq + 4 * i];
        acc[h] = fmaf(wv[i].w, qv.w, fmaf(wv[i].z, qv.z, fmaf(wv[i].y, qv.y, fmaf(wv[i].x, qv.x, acc[h]))));
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
    }
    if (dq == 0) {
#pragma unroll
      for (int h = 0; h < 8; ++h) ys[h][8 * wid + r] = acc[h];
    }
  }
  __syncthreads();
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
          // kFetchUnroll 16-byte loads in flight per thread: the host link's
          // latency is hidden by concurrency, not by one load at a time
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

namespace sekv {

// ----------------------------------------------------------------------------
// residency cache: plan (one CTA per group), then copy (kFetchParts per group)
// ----------------------------------------------------------------------------

// Block-wide exclusive prefix of v (256 threads); *total receives the sum.
// Shuffle scans within the warps and over the eight warp sums: three
// barriers.  sh holds at least 16 entries.
__device__ __forceinline__ long long block_excl_scan(long long v, long long* sh, long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    long long t = lane < 8 ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < 8) sh[8 + lane] = t;  // inclusive over the warps
  }
  __syncthreads();
  const long long incl = (wid > 0 ? sh[8 + wid - 1] : 0) + x;
  *total = sh[15];
  __syncthreads();  // sh is free for the next scan
  return incl - v;
}

__global__ void __launch_bounds__(256) cache_plan_kernel(const CacheParams P) {
  __shared__ long long scan[256];
  __shared__ int victims[kCacheMaxSlots];
  __shared__ int s_nvict, s_last;
  const int g = blockIdx.x, b = g / P.Hkv, tid = threadIdx.x;
  const size_t gs = size_t(g) * P.max_spans, gsl = size_t(g) * P.n_slots;
  const int n_sp = P.n_spans[b];
  int ne = P.n_expanded[g];
  if (ne < 0 || ne > n_sp) {
    if (tid == 0) set_device_error(P.status, DEV_BAD_LIST, g);
    ne = 0;
  }
  const int epoch = P.epoch[g] + 1;
  // Entry classes: 0 = a hit (or a bad entry), 1 = a miss that goes to a
  // slot, 2 = a miss that goes to staging.  Reads only tables that no
  // concurrent write of this call can change for the entry's own span.
  auto classify = [&](int e, int& k, int64_t& sz) -> int {
    k = P.expanded[gs + e];
    const int prev = e > 0 ? P.expanded[gs + e - 1] : -1;
    if (k < 0 || k >= n_sp || k <= prev) {
      k = -1;
      return 0;
    }
    if (P.slot_of[gs + k] >= 0) return 0;
    const int rank = P.rec_rank[gs + k];
    sz = record_bytes(P.body_len[size_t(b) * P.max_spans + k], rank & 0xffff,
                      (rank >> 16) & 0xffff);
    return sz <= P.slot_bytes ? 1 : 2;
  };
  // pass 1: hits keep their slots (marked as used by this call); count the
  // misses that fit a slot
  long long hit_n = 0, miss_n = 0;
  for (int e = tid; e < ne; e += 256) {
    int k;
    int64_t sz = 0;
    const int cls = classify(e, k, sz);
    if (k < 0) {
      set_device_error(P.status, DEV_BAD_LIST, e);
    } else if (cls == 0) {
      const int s = P.slot_of[gs + k];
      P.stamp[gsl + s] = epoch;
      P.staged_off[gs + e] = P.pool_base + (int64_t(gsl) + s) * P.slot_bytes;
      ++hit_n;
    } else if (cls == 1) {
      ++miss_n;
    }
  }
  long long n_hits, n_miss;
  block_excl_scan(hit_n, scan, &n_hits);
  block_excl_scan(miss_n, scan, &n_miss);
  // victims: the first slots from the clock hand on that no entry of this
  // call uses (free, or last used by an earlier call)
  if (tid == 0) {
    s_nvict = 0;
    s_last = -1;
  }
  __syncthreads();
  const int want = int(n_miss < P.n_slots ? n_miss : P.n_slots);
  const int hand = P.hand[g];
  for (int c0 = 0; c0 < P.n_slots && s_nvict < want; c0 += 256) {
    const int i = c0 + tid;
    int s = -1;
    bool ok = false;
    if (i < P.n_slots) {
      s = (hand + i) % P.n_slots;
      ok = P.span_of[gsl + s] < 0 || P.stamp[gsl + s] < epoch;
    }
    long long tot;
    const long long before = block_excl_scan(ok ? 1 : 0, scan, &tot);
    const int base = s_nvict;
    if (ok && base + before < want) {
      victims[base + before] = s;
      if (base + before == want - 1) s_last = i;
    }
    __syncthreads();
    if (tid == 0) s_nvict = int(base + tot < want ? base + tot : want);
    __syncthreads();
  }
  const int nv = s_nvict;
  // pass 2 (twice: measure, then commit): misses in list order; the first nv
  // that fit a slot take the victims, the rest go to staging, which must
  // hold them all before anything is evicted
  for (int commit = 0; commit < 2; ++commit) {
    long long carry_m = 0, carry_s = 0, carry_p = 0, carry_b = 0;
    for (int e0 = 0; e0 < ne; e0 += 256) {
      const int e = e0 + tid;
      int k = -1, cls = 0;
      int64_t sz = 0;
      if (e < ne) cls = classify(e, k, sz);
      __syncthreads();  // every lane has read the tables before this chunk writes them
      long long tm, ts, tp;
      const long long jm = carry_m + block_excl_scan(cls == 1 ? 1 : 0, scan, &tm);
      if (cls == 1 && jm >= nv) cls = 2;
      const long long js = carry_s + block_excl_scan(cls == 2 ? sz : 0, scan, &ts);
      long long tb;
      const long long jp = carry_p + block_excl_scan(cls != 0 ? 1 : 0, scan, &tp);
      block_excl_scan(cls != 0 ? sz : 0, scan, &tb);
      if (commit && cls != 0) {
        int64_t dst;
        if (cls == 1) {
          const int v = victims[jm];
          const int old = P.span_of[gsl + v];
          if (old >= 0) P.slot_of[gs + old] = -1;
          P.span_of[gsl + v] = k;
          P.slot_of[gs + k] = v;
          P.stamp[gsl + v] = epoch;
          dst = P.pool_base + (int64_t(gsl) + v) * P.slot_bytes;
        } else {
          dst = int64_t(g) * P.per_group + js;
        }
        P.staged_off[gs + e] = dst;
        int64_t* pl = P.plan + (gs + jp) * 3;
        pl[0] = P.rec_off[gs + k];
        pl[1] = dst;
        pl[2] = sz;
      }
      carry_m += tm;
      carry_s += ts;
      carry_p += tp;
      carry_b += tb;
    }
    if (!commit && carry_s > P.per_group) {
      // nothing is evicted or copied for this group
      if (tid == 0) {
        set_device_error(P.status, DEV_STAGING_FULL, g);
        P.plan_n[g] = 0;
        if (P.hits) P.hits[g] = int(n_hits);
        if (P.copied) P.copied[g] = 0;
      }
      return;
    }
    if (commit && tid == 0) {
      P.plan_n[g] = int(carry_p);
      if (P.copied) P.copied[g] = carry_b;
    }
    __syncthreads();
  }
  if (tid == 0) {
    P.epoch[g] = epoch;
    if (s_last >= 0) P.hand[g] = (hand + s_last + 1) % P.n_slots;
    if (P.hits) P.hits[g] = int(n_hits);
  }
}

// grid (B*Hkv, kFetchParts): part p copies the plan's entries c with
// c % kFetchParts == p from the host store over the host link.
__global__ void __launch_bounds__(256) cache_copy_kernel(const CacheParams P) {
  const int g = blockIdx.x, part = blockIdx.y, tid = threadIdx.x;
  const size_t gs = size_t(g) * P.max_spans;
  const int n = P.plan_n[g];
  for (int c = part; c < n; c += kFetchParts) {
    const int64_t* pl = P.plan + (gs + c) * 3;
    const int4* src = reinterpret_cast<const int4*>(P.store + pl[0]);
    int4* dst = reinterpret_cast<int4*>(P.staging + pl[1]);
    const long long n16 = pl[2] / 16;
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

}  // namespace sekv
